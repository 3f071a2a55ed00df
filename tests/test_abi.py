"""The C ABI on the host (no GPU): the library loads, exports every entry point
that include/aircache.h declares, and rejects bad arguments before touching
CUDA.  Only host-side paths run here; no kernel is launched."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "aircache.h")


@pytest.fixture(scope="module")
def A():
    from lvlm_kv_cache_gb300 import build

    build.build()
    from lvlm_kv_cache_gb300 import aircache

    aircache.lib()
    return aircache


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"AIRCACHE_API\s+[\w\s\*]+?\b(aircache_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ["aircache_score", "aircache_budget", "aircache_select", "aircache_compact",
              "aircache_compress", "aircache_workspace_size", "aircache_compress_bound",
              "aircache_get_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(A):
    lib = A.lib()
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing


def fake_problem(A, **over):
    """A problem whose device pointers are fake, aligned addresses: valid for
    host-side checks only (never launched)."""
    L = over.pop("L", 4)
    arr = (ctypes.c_void_p * L)(*[0x100000 + 0x10000 * i for i in range(L)])
    p = A.ProblemStruct(
        num_layers=L, num_requests=2, h_q=8, h_kv=2, head_dim=128, dtype=A.BF16,
        max_visual=1000, max_text=64, max_elite=0, variant=0,
        total_tokens=1000 + 900 + 64 + 50, total_visual=1900,
        cu_seqlens=0x200000, cu_visual=0x300000,
        q_text=ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)),
        k=ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)),
        v=ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)),
        q_stride_tok=8 * 128, q_stride_head=128, kv_stride_tok=2 * 128, kv_stride_head=128,
        alpha=0.9, r=0.1)
    for k, v in over.items():
        setattr(p, k, v)
    p._keep = arr
    return p


def test_sizes_of_a_valid_problem(A):
    p = fake_problem(A)
    ws = A.lib().aircache_workspace_size(ctypes.byref(p))
    assert ws > 0 and ws % 256 == 0
    bound = A.lib().aircache_compress_bound(ctypes.byref(p))
    assert bound == A.math_bound(4, 2, 114, 1900, 0.1) == 4 * 114 + math.ceil(0.1 * 4 * 1900) + 2 * 9
    assert A.lib().aircache_compress_launches(ctypes.byref(p)) > 0


def test_launch_count_and_kernel_names(A):
    """The kernels one aircache_compress call launches, by scoring path: the
    first clears the call's counters and error word (so aircache_compress_profile
    times it too), then the elite step, the scoring, the selection and the
    compaction."""
    lib = A.lib()
    stream = ["zero_block", "elite_window", "score_pass1", "score_pass2", "score_pass2k", "budget_select",
              "gather_compact"]
    wide = ["zero_block", "elite_window", "score_wide", "select_topk", "gather_compact"]
    q = fake_problem(A, dtype=A.F32)  # fp32: the wide path
    assert lib.aircache_compress_launches(ctypes.byref(q)) == len(wide)
    assert [lib.aircache_kernel_name(ctypes.byref(q), i).decode() for i in range(len(wide))] == wide
    assert lib.aircache_kernel_name(ctypes.byref(q), len(wide)) is None
    # bf16 with evenly strided layers takes the streaming path where the driver
    # can encode its key tensor map (a GPU host); here the wide path is allowed
    p = fake_problem(A)
    n = lib.aircache_compress_launches(ctypes.byref(p))
    names = stream if n == len(stream) else wide
    assert n == len(names)
    assert [lib.aircache_kernel_name(ctypes.byref(p), i).decode() for i in range(n)] == names


@pytest.mark.parametrize("field,value,code", [
    ("num_layers", 0, -1), ("num_layers", 257, -1), ("num_requests", 0, -1),
    ("h_q", 7, -1), ("h_kv", 0, -1), ("head_dim", 96, -2), ("head_dim", 0, -1),
    ("dtype", 7, -2), ("max_visual", 2, -1), ("max_text", 0, -1), ("max_text", 9000, -2),
    ("max_elite", 65, -1), ("max_elite", -1, -1), ("variant", 2 << 16, -1), ("variant", 1 << 25, -1), ("variant", 4, -1), ("variant", 5 << 8, -1),
    ("total_visual", 5, -1), ("total_tokens", 1901, -1), ("total_visual", 2001, -1),
    ("cu_seqlens", None, -1), ("cu_visual", None, -1),
    ("kv_stride_tok", 0, -1), ("kv_stride_tok", 3, -1), ("q_stride_head", 4, -1),
    ("alpha", -0.1, -1), ("alpha", 1.5, -1), ("alpha", float("nan"), -1),
    ("r", 0.0, -1), ("r", 1.01, -1), ("r", float("nan"), -1),
])
def test_invalid_problem_rejected_on_host(A, field, value, code):
    p = fake_problem(A, **{field: value})
    lib = A.lib()
    assert lib.aircache_workspace_size(ctypes.byref(p)) == 0
    assert lib.aircache_compress_bound(ctypes.byref(p)) == -1
    rc = lib.aircache_compress(ctypes.byref(p), ctypes.c_void_p(0x400000), 1 << 40,
                               ctypes.c_void_p(0x500000), ctypes.c_void_p(0x600000),
                               ctypes.c_void_p(0x700000), 10 ** 6, ctypes.c_void_p(0x800000),
                               None, None, None)
    assert rc == code


def test_wait_test_hook_is_accepted(A):
    # bit 24 of the variant word is the bounded-wait test hook (the workspace is unchanged)
    p = fake_problem(A)
    q = fake_problem(A, variant=A.VARIANT_WAIT_TEST)
    assert A.VARIANT_WAIT_TEST == 1 << 24
    assert A.lib().aircache_workspace_size(ctypes.byref(q)) == A.lib().aircache_workspace_size(ctypes.byref(p)) > 0


def test_unaligned_layer_pointer_rejected(A):
    p = fake_problem(A)
    arr = (ctypes.c_void_p * 4)(0x100000, 0x100008, 0x120000, 0x130000)
    p.k = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    p._keep2 = arr
    assert A.lib().aircache_workspace_size(ctypes.byref(p)) == 0


def test_workspace_checks_before_any_launch(A):
    p = fake_problem(A)
    lib = A.lib()
    need = lib.aircache_workspace_size(ctypes.byref(p))
    args = (ctypes.c_void_p(0x500000), ctypes.c_void_p(0x600000), ctypes.c_void_p(0x700000))
    # too small
    assert lib.aircache_score(ctypes.byref(p), ctypes.c_void_p(0x400000), need - 1, *args, None) == -3
    # misaligned workspace
    assert lib.aircache_score(ctypes.byref(p), ctypes.c_void_p(0x400010), need, *args, None) == -1
    # missing outputs
    assert lib.aircache_score(ctypes.byref(p), ctypes.c_void_p(0x400000), need, None, None, None,
                              None) == -1
    assert lib.aircache_compact(ctypes.byref(p), ctypes.c_void_p(0x500000), ctypes.c_void_p(0x600000),
                                ctypes.c_void_p(0x400000), need, ctypes.c_void_p(0x700008),
                                ctypes.c_void_p(0x800000), ctypes.c_void_p(0x900000), 100, None) == -1


def test_status_strings(A):
    for code in range(-8, 1):
        assert A.status_string(code) not in ("", "unknown status")
    assert A.status_string(-99) == "unknown status"


def test_workspace_grows_with_max_elite(A):
    a = A.lib().aircache_workspace_size(ctypes.byref(fake_problem(A, max_elite=8)))
    b = A.lib().aircache_workspace_size(ctypes.byref(fake_problem(A, max_elite=64)))
    c = A.lib().aircache_workspace_size(ctypes.byref(fake_problem(A)))
    assert 0 < a < b == c


def test_per_head_sets_only_through_the_fused_call(A):
    # one index set per KV head (variant bits 16-23 = 1): the staged calls refuse it on the host
    p = fake_problem(A, variant=1 << 16)
    lib = A.lib()
    need = lib.aircache_workspace_size(ctypes.byref(p))
    assert need > lib.aircache_workspace_size(ctypes.byref(fake_problem(A)))  # per-head I_v and index sets
    ws = ctypes.c_void_p(0x400000)
    bufs = (ctypes.c_void_p(0x500000), ctypes.c_void_p(0x600000), ctypes.c_void_p(0x700000))
    assert lib.aircache_score(ctypes.byref(p), ws, need, *bufs, None) == -2
    assert lib.aircache_select(ctypes.byref(p), bufs[0], bufs[1], ws, need, bufs[2], None) == -2
    assert lib.aircache_compact(ctypes.byref(p), bufs[0], bufs[1], ws, need, ctypes.c_void_p(0x800000),
                                ctypes.c_void_p(0x900000), ctypes.c_void_p(0xa00000), 100, None) == -2
