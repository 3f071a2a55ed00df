"""GPU parity of the int8 storage of the kept cache (aircache_quantize_int8,
reading R17) and of decoding from it (aircache_decode with int8 rows).

Quantisation: codes and scales are exact functions of the inputs in fp32 on
both sides (max |x|, s = max / 127, x / s correctly rounded, round half away
from zero), so they must match the oracle bit for bit.  Decoding from int8:
the kernel computes with the exact integer codes and applies the scales to the
logits and to the weighted sum, so it is compared with the oracle's decode over
the dequantised rows s * c (held in fp32, which moves each value by at most
2^-24 relative) under the same bf16-weight bound as the bf16 decode."""
import numpy as np
import pytest
import torch

from lvlm_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu

U = 1.02 * 2.0 ** -8


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lvlm_kv_cache_gb300 import build

    build.build()
    from lvlm_kv_cache_gb300 import aircache

    aircache.lib()
    return aircache


def check_units(oracle, k, k8, ks, offsets):
    """Every unit's codes and scales against the oracle, bit for bit."""
    kb = W.host_bits(k)
    c8 = k8.cpu().numpy()
    sc = ks.cpu().numpy()
    offs = offsets.cpu().numpy()
    for u in range(len(offs) - 1):
        b, e = int(offs[u]), int(offs[u + 1])
        codes, scales = oracle.quantize_int8(kb[b:e])
        assert np.array_equal(sc[u], scales), f"unit {u}: scales"
        assert np.array_equal(c8[b:e], codes), f"unit {u}: codes"


def test_quantize_the_compressed_arena(A, oracle):
    wl = W.make("ragged", seed=21, device="cuda", layers=3, requests=4)
    s = wl.spec
    prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text),
                     alpha=s.alpha, r=s.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual)
    res = A.compress(prob)
    rows = int(res["out_offsets"][-1])
    k, v = res["out_k"][:rows], res["out_v"][:rows]
    k8, v8, ks, vs = A.quantize_int8(k, v, res["out_offsets"])
    check_units(oracle, k, k8, ks, res["out_offsets"])
    check_units(oracle, v, v8, vs, res["out_offsets"])


@pytest.mark.parametrize("d", [64, 128])
def test_quantize_edge_cases(A, oracle, d):
    g = torch.Generator(device="cuda").manual_seed(22)
    h_kv = 3
    wide = torch.randn((600, h_kv + 1, d), generator=g, device="cuda").to(torch.bfloat16)
    k = wide[:, :h_kv]             # strided rows (an unused head)
    k[100:180, 1] = 0.0            # a unit whose head 1 is all zero
    k[200, 2, 5] = 1000.0          # a large outlier in one unit
    v = torch.randn((600, h_kv + 1, d), generator=g, device="cuda").to(torch.bfloat16)[:, :h_kv]
    offs = torch.tensor([0, 100, 100, 180, 201, 599], dtype=torch.int64, device="cuda")  # an empty unit
    k8, v8, ks, vs = A.quantize_int8(k, v, offs)
    check_units(oracle, k.contiguous(), k8, ks, offs)
    check_units(oracle, v.contiguous(), v8, vs, offs)
    assert float(ks[2, 1]) == 0.0 and not k8[100:180, 1].any()


def test_quantize_bounds_error(A):
    k = torch.zeros((10, 2, 64), dtype=torch.bfloat16, device="cuda")
    offs = torch.tensor([0, 4, 12], dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    k8 = torch.zeros((10, 2, 64), dtype=torch.int8, device="cuda")
    sc = torch.zeros((2, 2), dtype=torch.float32, device="cuda")
    A.aircache_quantize_int8(k, k, offs, k8, k8.clone(), sc, sc.clone(), st)
    assert int(st.item()) == A.ERR_DEVICE_BOUNDS


def dequant(codes, scales):
    return (codes.astype(np.float32) * scales.astype(np.float32)[None, :, None]).astype(np.float32)


def tolerance(q, k, v, ref):
    """The bf16-weight bound for fp32 k, v [n, H_kv, D] and bf16-bit q [H_q, D]."""
    h_q, d = q.shape
    g = h_q // k.shape[1]
    qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    kf, vf = k.astype(np.float64), v.astype(np.float64)
    tol = np.zeros((h_q, d))
    for h in range(h_q):
        x = kf[:, h // g] @ qf[h] / np.sqrt(d)
        w = np.exp(x - x.max())
        w /= w.sum()
        tol[h] = U / (1 - U) * (w @ np.abs(vf[:, h // g] - ref[h])) + 1e-5 * np.abs(vf[:, h // g]).max()
    return tol


def decode_int8_check(A, oracle, di, max_rows):
    k8, v8, ks, vs = A.quantize_int8(di.k, di.v, di.offsets)
    prob = A.DecodeProblem(di.q, k8, v8, offsets=di.offsets, max_rows=max_rows, k_new=di.k_new,
                           v_new=di.v_new, k_scale=ks, v_scale=vs)
    out = A.decode(prob).cpu().numpy().astype(np.float64)
    qb = W.host_bits(di.q)
    c_k, c_v = k8.cpu().numpy(), v8.cpu().numpy()
    s_k, s_v = ks.cpu().numpy(), vs.cpu().numpy()
    offs = di.offsets.cpu().numpy()
    for s in range(len(offs) - 1):
        b, e = int(offs[s]), int(offs[s + 1])
        kd, vd = dequant(c_k[b:e], s_k[s]), dequant(c_v[b:e], s_v[s])
        if di.k_new is not None:
            kn = di.k_new[s:s + 1].float().cpu().numpy()
            vn = di.v_new[s:s + 1].float().cpu().numpy()
            kd, vd = np.concatenate([kd, kn]), np.concatenate([vd, vn])
        if len(kd) == 0:
            assert np.all(out[s] == 0.0)
            continue
        ref = oracle.decode(qb[s], kd, vd)
        tol = tolerance(qb[s], kd, vd, ref)
        err = np.abs(out[s] - ref)
        assert np.all(err <= tol), f"sequence {s}: worst err/tol {(err / tol).max():.2f}"
    return out


@pytest.mark.parametrize("max_rows", [0, 1000, 10 ** 6])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_from_int8_matches_oracle(A, oracle, max_rows, d):
    di = W.decode_inputs([1, 17, 64, 65, 300, 2500], 28, 4, d, seed=23, device="cuda", q_scale=2.0)
    decode_int8_check(A, oracle, di, max_rows)


def test_decode_from_int8_with_new_row_and_empty(A, oracle):
    di = W.decode_inputs([0, 5, 130, 0, 900], 28, 4, 128, seed=24, device="cuda", q_scale=2.0, new_row=True)
    decode_int8_check(A, oracle, di, 900)


@pytest.mark.parametrize("q_scale", [1e20, 1e-20, 1e-37])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_from_int8_extreme_query_magnitudes(A, oracle, q_scale, d):
    # the int8 path feeds Q to its f16 MMAs times a power of two chosen from
    # the group's largest |q|: no overflow for huge queries (one-hot weights),
    # no loss for tiny ones (near-uniform weights), and the exponent clamp for
    # a maximum near the bottom of the bf16 range
    di = W.decode_inputs([3, 64, 1000], 28, 4, d, seed=27, device="cuda", q_scale=q_scale)
    decode_int8_check(A, oracle, di, 1000)


def test_decode_from_int8_early_cache_matches_plain_launches(A, oracle):
    # int8 rows with programmatic dependent launch (the codes are not written by
    # the kernel before each call; the queries are): the same bits as plain
    # launches
    di = W.decode_inputs([700, 33, 4100, 5], 28, 4, 128, seed=28, device="cuda", q_scale=2.0, new_row=True)
    k8, v8, ks, vs = A.quantize_int8(di.k, di.v, di.offsets)
    outs = {}
    for early in (False, True):
        ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
        res = []
        for m in (0, 1000, 10 ** 6):
            q = torch.empty_like(di.q)
            q.copy_(di.q)  # written by the kernel right before the decode kernel
            p = A.DecodeProblem(q, k8, v8, offsets=di.offsets, max_rows=m, k_new=di.k_new, v_new=di.v_new,
                                k_scale=ks, v_scale=vs, early_cache=early)
            A.aircache_decode(p, ws)
            res.append(p.out)
        assert A.aircache_get_error(ws) == A.OK
        outs[early] = [r.clone() for r in res]
    for a, b in zip(outs[False], outs[True]):
        assert torch.equal(a, b)


def test_decode_from_int8_rows_past_a_range(A, oracle):
    # the codes after the last range are garbage for this call: never mixed in
    di = W.decode_inputs([40, 77], 8, 2, 128, seed=25, device="cuda")
    k8, v8, ks, vs = A.quantize_int8(di.k, di.v, di.offsets)
    k8big = torch.full((k8.shape[0] + 100,) + tuple(k8.shape[1:]), 127, dtype=torch.int8, device="cuda")
    v8big = k8big.clone()
    k8big[:k8.shape[0]] = k8
    v8big[:v8.shape[0]] = v8
    prob = A.DecodeProblem(di.q, k8big, v8big, offsets=di.offsets, max_rows=77, k_scale=ks, v_scale=vs)
    out = A.decode(prob)
    prob2 = A.DecodeProblem(di.q, k8, v8, offsets=di.offsets, max_rows=77, k_scale=ks, v_scale=vs)
    assert torch.equal(out, A.decode(prob2))


def test_decode_from_the_quantised_compressed_arena(A, oracle):
    wl = W.make("ragged", seed=26, device="cuda", layers=2, requests=3)
    s = wl.spec
    prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text),
                     alpha=s.alpha, r=s.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual)
    res = A.compress(prob)
    offs = res["out_offsets"]
    k8, v8, ks, vs = A.quantize_int8(res["out_k"], res["out_v"], offs)
    B, L = prob.B, prob.L
    g = torch.Generator(device="cuda").manual_seed(27)
    qs = torch.randn((L, B, s.H_q, s.D), generator=g, device="cuda").to(torch.bfloat16)
    rows = offs.cpu().numpy()
    c_k, c_v, s_k, s_v = k8.cpu().numpy(), v8.cpu().numpy(), ks.cpu().numpy(), vs.cpu().numpy()
    for l in range(L):
        dp = A.DecodeProblem(qs[l], k8, v8, row_begin=offs[l * B:(l + 1) * B], row_end=offs[l * B + 1:(l + 1) * B + 1],
                             max_rows=int(np.diff(rows).max()), k_scale=ks[l * B:(l + 1) * B],
                             v_scale=vs[l * B:(l + 1) * B])
        out = A.decode(dp).cpu().numpy().astype(np.float64)
        qb = W.host_bits(qs[l])
        for b in range(B):
            u = l * B + b
            r0, r1 = int(rows[u]), int(rows[u + 1])
            kd, vd = dequant(c_k[r0:r1], s_k[u]), dequant(c_v[r0:r1], s_v[u])
            ref = oracle.decode(qb[b], kd, vd)
            assert np.all(np.abs(out[b] - ref) <= tolerance(qb[b], kd, vd, ref)), f"layer {l} request {b}"


def test_quantize_many_values_and_exact_halves(A, oracle):
    # a million values over units of varied scale, plus exact half-integer
    # quotients (max 254 -> s = 2, x = 5 -> 2.5 -> 3): bit-exact everywhere
    g = torch.Generator(device="cuda").manual_seed(28)
    rows, h_kv, d = 4000, 2, 128
    k = (torch.randn((rows, h_kv, d), generator=g, device="cuda") *
         torch.exp(torch.randn((rows, 1, 1), generator=g, device="cuda") * 2)).to(torch.bfloat16)
    k[:10] = 0.0
    k[0, 0, 0], k[1, 0, 1], k[2, 0, 2], k[3, 1, 3] = 254.0, 5.0, -5.0, 3.0
    offs = torch.tensor([0, 10, 333, 1000, 2500, 4000], dtype=torch.int64, device="cuda")
    k8, v8, ks, vs = A.quantize_int8(k, k, offs)
    check_units(oracle, k, k8, ks, offs)
    assert int(k8[1, 0, 1]) == 3 and int(k8[2, 0, 2]) == -3
