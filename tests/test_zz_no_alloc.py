"""aircache_budget_noalloc: the budget step with the library's fixed device
scratch instead of a caller workspace.

The GPU test runs the workspace entry point aircache_budget and then the
no-allocation entry point twice in a row on the same I_v (the second call
relies on the first having left its scratch reusable) and requires the same
statistics, the same keep counts and a clean device status each time.  The
keep counts are also checked directly against the oracle's budget of the same
I_v, so the test does not rest on the workspace path alone.  The
file is named to be collected last, so the scratch is also exercised after
every other GPU test of a session; it passes on its own in a fresh process
too.  The host-side limit check needs no GPU."""
import ctypes

import numpy as np
import pytest
import torch

from lvlm_kv_cache_gb300 import workloads as W

MAX_UNITS = 2048  # AIRCACHE_NOALLOC_MAX_UNITS in include/aircache.h


@pytest.fixture(scope="module")
def A():
    from lvlm_kv_cache_gb300 import build

    build.build()
    from lvlm_kv_cache_gb300 import aircache

    aircache.lib()
    return aircache


def make_problem(A, wl):
    s = wl.spec
    return A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text), s.alpha,
                     s.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual)


@pytest.mark.gpu
@pytest.mark.parametrize("name,layers,requests", [("ragged", 6, 5), ("7b", 28, 1)])
def test_noalloc_budget_matches_workspace_budget(A, name, layers, requests):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = W.make(name, seed=11, device="cuda", layers=layers, requests=requests)
    prob = make_problem(A, wl)
    L, B = prob.L, prob.B
    ws = prob.new_workspace()
    iv = torch.empty((L, prob.total_visual), dtype=torch.float32, device="cuda")
    elite = torch.empty((L * B, prob.max_text), dtype=torch.int32, device="cuda")
    n_tk = torch.empty(L * B, dtype=torch.int32, device="cuda")
    A.aircache_score(prob, ws, iv, elite, n_tk)
    stats_ref = torch.zeros((L * B, 2), dtype=torch.float64, device="cuda")
    keep_ref = torch.zeros(L * B, dtype=torch.int32, device="cuda")
    A.aircache_budget(prob, iv, ws, stats_ref, keep_ref)
    assert A.aircache_get_error(ws) == 0
    ref_s, ref_k = stats_ref.cpu().numpy(), keep_ref.cpu().numpy()
    assert np.all(np.isfinite(ref_s)) and np.all(ref_k >= 1)

    for call in range(2):
        stats = torch.full((L * B, 2), float("nan"), dtype=torch.float64, device="cuda")
        keep = torch.full((L * B,), -1, dtype=torch.int32, device="cuda")
        status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
        A.aircache_budget_noalloc(prob, iv, stats, keep, device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        # both entry points launch the same kernel with the same block size, so
        # the reduction order is the same and the results agree bit for bit
        np.testing.assert_array_equal(stats.cpu().numpy(), ref_s)
        assert np.array_equal(keep.cpu().numpy(), ref_k), f"call {call}: keep counts differ"

    # against the oracle: (s_t, s_k) of the same I_v in fp64 to the float-float
    # precision of the device reduction, and the oracle's keep counts exactly
    from oracle import oracle as O

    iv_h = iv.cpu().numpy().astype(np.float64)
    cu_v = wl.cu_visual.cpu().numpy()
    for b in range(B):
        n_v = int(cu_v[b + 1] - cu_v[b])
        st, sk = [], []
        for l in range(L):
            s_t, s_k, _, _ = O.stats(iv_h[l, cu_v[b]:cu_v[b + 1]])
            st.append(s_t)
            sk.append(s_k)
            np.testing.assert_allclose(ref_s[l * B + b], [s_t, s_k], rtol=1e-9, atol=1e-12)
        _, keep_o = O.budget(st, sk, n_v, wl.spec.r)
        keep_g = ref_k[[l * B + b for l in range(L)]]
        assert np.array_equal(keep_g, keep_o), f"request {b}: keep differs from the oracle"

    # stats may be omitted
    keep = torch.full((L * B,), -1, dtype=torch.int32, device="cuda")
    A.aircache_budget_noalloc(prob, iv, None, keep)
    torch.cuda.synchronize()
    assert np.array_equal(keep.cpu().numpy(), ref_k)


def host_only_problem(A, L, B):
    """Valid for host-side checks only: its device pointers are fake aligned
    addresses and nothing is ever launched on it."""
    arr = (ctypes.c_void_p * L)(*[0x100000 + 0x10000 * i for i in range(L)])
    n_v, n_t = 100, 8
    return A.ProblemStruct(
        num_layers=L, num_requests=B, h_q=8, h_kv=2, head_dim=128, dtype=A.BF16,
        max_visual=n_v, max_text=n_t, max_elite=0, variant=0,
        total_tokens=B * (n_v + n_t), total_visual=B * n_v,
        cu_seqlens=0x200000, cu_visual=0x300000,
        q_text=ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)),
        k=ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)),
        v=ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)),
        q_stride_tok=8 * 128, q_stride_head=128, kv_stride_tok=2 * 128, kv_stride_head=128,
        alpha=0.9, r=0.1)


def test_noalloc_rejects_problems_beyond_its_scratch(A):
    lib = A.lib()
    fake = ctypes.c_void_p(0x400000)
    big = host_only_problem(A, 256, 9)  # 2304 layer-request pairs
    assert 256 * 9 > MAX_UNITS
    rc = lib.aircache_budget_noalloc(ctypes.byref(big), fake, None, fake, None, None)
    assert rc == A.ERR_UNSUPPORTED
    # the workspace entry point's own validation accepts the same problem
    assert lib.aircache_workspace_size(ctypes.byref(big)) > 0
    bad = host_only_problem(A, 4, 2)
    assert lib.aircache_budget_noalloc(ctypes.byref(bad), None, None, fake, None, None) == A.ERR_INVALID_ARG
    assert lib.aircache_budget_noalloc(ctypes.byref(bad), fake, None, None, None, None) == A.ERR_INVALID_ARG
