"""Host-side checks of the decode entry points (no GPU, nothing launched):
sizes, the split count, and argument errors returned before any CUDA call."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def A():
    from lvlm_kv_cache_gb300 import build

    build.build()
    from lvlm_kv_cache_gb300 import aircache

    aircache.lib()
    return aircache


def fake(A, **over):
    p = A.DecodeProblemStruct(
        num_seqs=8, h_q=28, h_kv=4, head_dim=128, dtype=A.BF16, kv_dtype=A.BF16,
        kv_rows=100000, max_rows=2048,
        q=0x100000, k=0x200000, v=0x300000, row_begin=0x400000, row_end=0x400008,
        k_new=None, v_new=None,
        q_stride_seq=28 * 128, q_stride_head=128, kv_stride_row=4 * 128, kv_stride_head=128,
        new_stride_seq=0, new_stride_head=0, out=0x500000)
    for k, v in over.items():
        setattr(p, k, v)
    return p


def test_sizes_and_splits(A):
    lib = A.lib()
    p = fake(A)
    ws = lib.aircache_decode_workspace_size(ctypes.byref(p))
    n = lib.aircache_decode_splits(ctypes.byref(p))
    assert ws > 0 and ws % 256 == 0
    assert 1 <= n <= 64
    # the partials hold (max, sum) and D floats per (sequence, query head, split)
    assert ws >= 8 * 28 * n * (128 + 2) * 4
    # a short hint needs fewer splits; a long one never more than 64
    assert lib.aircache_decode_splits(ctypes.byref(fake(A, max_rows=64))) == 1
    assert lib.aircache_decode_splits(ctypes.byref(fake(A, max_rows=10 ** 7, num_seqs=1, h_kv=1, h_q=1))) == 64
    assert lib.aircache_decode_splits(ctypes.byref(fake(A, max_rows=0))) == 1


@pytest.mark.parametrize("field,value,code", [
    ("num_seqs", -1, -1), ("num_seqs", 65536, -1), ("h_q", 27, -1), ("h_kv", 0, -1),
    ("head_dim", 96, -1), ("dtype", 0, -2), ("h_q", 68, -2), ("kv_dtype", 0, -1), ("kv_dtype", 3, -1),
    ("kv_dtype", 2, -1), ("flags", 2, -1), ("reserved1", 1, -1), ("row_index", 0x800000, -1),
    ("kv_rows", 0, -1), ("kv_rows", 1 << 31, -1), ("max_rows", -1, -1),
    ("q", None, -1), ("k", None, -1), ("out", None, -1), ("row_begin", None, -1),
    ("k", 0x200008, -1), ("q", 0x100004, -1), ("kv_stride_row", 4 * 128 + 4, -1),
    ("kv_stride_head", 0, -1), ("q_stride_head", 4, -1), ("k_new", 0x600000, -1),
])
def test_invalid_decode_rejected_on_host(A, field, value, code):
    lib = A.lib()
    p = fake(A, **{field: value})
    assert lib.aircache_decode_workspace_size(ctypes.byref(p)) == 0
    assert lib.aircache_decode_splits(ctypes.byref(p)) == -1
    assert lib.aircache_decode(ctypes.byref(p), ctypes.c_void_p(0x700000), 1 << 40, None) == code


def test_decode_workspace_checks(A):
    lib = A.lib()
    p = fake(A)
    need = lib.aircache_decode_workspace_size(ctypes.byref(p))
    assert lib.aircache_decode(ctypes.byref(p), ctypes.c_void_p(0x700000), need - 1, None) == -3
    assert lib.aircache_decode(ctypes.byref(p), ctypes.c_void_p(0x700010), need, None) == -1
    assert lib.aircache_decode(ctypes.byref(p), None, need, None) == -1


def fake_quant(A, **over):
    p = A.QuantProblemStruct(num_units=28, h_kv=4, head_dim=128, dtype=A.BF16, reserved0=0, reserved1=0,
                             rows=30000, k=0x100000, v=0x200000, kv_stride_row=512, kv_stride_head=128,
                             offsets=0x300000, k8=0x400000, v8=0x500000, k_scale=0x600000, v_scale=0x700000)
    for k, v in over.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("field,value", [
    ("num_units", -1), ("h_kv", 0), ("head_dim", 96), ("dtype", 0), ("reserved0", 1), ("rows", 0),
    ("k", None), ("v8", None), ("k_scale", None), ("offsets", None), ("k", 0x100008), ("k8", 0x400004),
    ("kv_stride_row", 510), ("kv_stride_head", 0),
])
def test_invalid_quantize_rejected_on_host(A, field, value):
    p = fake_quant(A, **{field: value})
    assert A.lib().aircache_quantize_int8(ctypes.byref(p), None, None) == -1


def test_gather_rows_need_bf16(A):
    p = fake(A, row_index=0x800000, index_len=100, kv_dtype=A.INT8, k_scale=0x900000, v_scale=0x910000,
             kv_stride_row=512, kv_stride_head=128)
    assert A.lib().aircache_decode_workspace_size(ctypes.byref(p)) == 0
    assert A.lib().aircache_decode(ctypes.byref(p), ctypes.c_void_p(0x700000), 1 << 40, None) == -2
