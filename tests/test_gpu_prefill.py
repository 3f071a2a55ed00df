"""Scoring fused into prefill: the causal prefill attention of every layer
(aircache_prefill) against a plain fp32 PyTorch attention, and the compression
taken from the prefill's own logits (aircache_prefill_compress) against the
oracle and against aircache_compress on the same inputs."""
import math

import numpy as np
import pytest
import torch

import parity_utils as PU
from lvlm_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from lvlm_kv_cache_gb300 import build

    build.build()
    from lvlm_kv_cache_gb300 import aircache

    aircache.lib()
    return aircache


def q_all_of(wl, seed=5):
    """Every prompt row's query, [L, T, H_q, D]: seeded visual-token queries,
    then the workload's text queries, request by request (visual-first)."""
    s = wl.spec
    qv = W.visual_queries(wl, seed)
    cu_s, cu_v, cu_t = W.offsets(s)
    q = torch.empty((s.L, wl.total_tokens, s.H_q, s.D), dtype=s.dtype, device=wl.q.device)
    for b in range(s.B):
        nv = cu_v[b + 1] - cu_v[b]
        q[:, cu_s[b]:cu_s[b] + nv] = qv[:, cu_v[b]:cu_v[b + 1]]
        q[:, cu_s[b] + nv:cu_s[b + 1]] = wl.q[:, cu_t[b]:cu_t[b + 1]]
    return q


def problem(A, wl, **kw):
    s = wl.spec
    return A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text), s.alpha, s.r,
                     **kw)


def reference_attention(q, k, v, lo, hi, h, g):
    """fp32 causal attention of rows lo..hi-1 (one request), query head h:
    (output [n, D], the weights' |v| sums for the error bound)."""
    qq = q[lo:hi, h].float()
    kk = k[lo:hi, h // g].float()
    vv = v[lo:hi, h // g].float()
    s = qq @ kk.T / math.sqrt(q.shape[-1])
    n = hi - lo
    mask = torch.ones((n, n), dtype=torch.bool, device=q.device).triu(1)
    s = s.masked_fill(mask, float("-inf"))
    p = torch.softmax(s, dim=1)
    return p @ vv, p @ vv.abs()


def check_attention(attn, q, k, v, wl, layers, heads):
    """The kernel rounds each softmax weight to bf16 (relative error <= 2^-9) and
    its output to bf16: |o - o*| <= 2^-9 sum_j w_j |v_j| + 2^-9 |o*| (both
    doubled here), plus fp32 accumulation."""
    s = wl.spec
    g = s.H_q // s.H_kv
    cu_s, _, _ = W.offsets(s)
    worst = 0.0
    for l in layers:
        for b in range(s.B):
            for h in heads:
                ref, absw = reference_attention(q[l], k[l], v[l], cu_s[b], cu_s[b + 1], h, g)
                got = attn[l, cu_s[b]:cu_s[b + 1], h].float()
                bound = 2.0 ** -8 * absw + 2.0 ** -8 * ref.abs() + 1e-5
                err = (got - ref).abs()
                assert bool((err <= bound).all()), f"l={l} b={b} h={h}: {float((err / bound).max())}"
                worst = max(worst, float((err / bound).max()))
    return worst


def small_workload():
    spec = W.Spec("prefill", 3, 2, 8, 2, 128, [200, 300, 129], [40, 70, 1], torch.bfloat16, 0.9, 0.1,
                  heavy_frac=0.1, heavy_bias=1.5, layer_scale=(0.5, 2.0))
    return W.generate(spec, seed=3, device="cuda")


def test_prefill_attention_small(A):
    wl = small_workload()
    q = q_all_of(wl)
    prob = problem(A, wl)
    attn = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = prob.new_workspace()
    A.aircache_prefill(prob, q, attn, ws)
    assert A.aircache_get_error(ws) == 0
    worst = check_attention(attn, q, wl.k, wl.v, wl, range(wl.spec.L), range(wl.spec.H_q))
    print("prefill attention: worst error / bound", worst)


def test_prefill_attention_7b_two_layers_sampled_heads(A):
    wl = W.make("7b", device="cuda", layers=2)
    q = q_all_of(wl)
    prob = problem(A, wl)
    attn = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    ws = prob.new_workspace()
    A.aircache_prefill(prob, q, attn, ws)
    assert A.aircache_get_error(ws) == 0
    worst = check_attention(attn, q, wl.k, wl.v, wl, [1], [0, 13, 27])
    print("7b prefill attention: worst error / bound", worst)


def _check_against_oracle(oracle, wl, host):
    s = wl.spec
    cu_s, cu_v, _ = W.offsets(s)
    report = {}
    for b in range(s.B):
        ivs = {}
        for l in range(s.L):
            q, k, _ = PU.unit_views(wl, l, b, cu_s, cu_v)
            n_v = cu_v[b + 1] - cu_v[b]
            el, _ = oracle.elite(q, k, n_v, s.alpha)
            iv_o, _ = oracle.score(q, k, n_v, el)
            PU.check_iv(iv_o, host["iv"][l, cu_v[b]:cu_v[b + 1]], f"(l={l}, b={b})")
            ivs[l] = iv_o
        PU.check_request(oracle, wl, b, cu_s, cu_v, host, report, ivs)
        for l in range(s.L):
            PU.check_compaction(oracle, wl, l, b, cu_s, cu_v, host)
    assert report.get("near_half_exempt", 0) == 0 and report.get("keep_boundary", 0) == 0, report
    return report


@pytest.mark.parametrize("which", ["small", "7b"])
def test_prefill_compress_matches_oracle_and_compress(A, oracle, which):
    wl = small_workload() if which == "small" else W.make("7b", device="cuda", layers=3)
    q = q_all_of(wl)
    prob = problem(A, wl)
    attn, out = A.prefill_compress(prob, q)
    torch.cuda.synchronize()
    # the attention is the plain prefill's, bit for bit
    attn2 = torch.empty_like(attn)
    ws = prob.new_workspace()
    A.aircache_prefill(prob, q, attn2, ws)
    torch.cuda.synchronize()
    assert torch.equal(attn, attn2)
    host = PU.gpu_to_host(out, prob)
    rep = _check_against_oracle(oracle, wl, host)
    # against the compression that streams the keys itself
    ref = PU.gpu_to_host(A.compress(prob), prob)
    np.testing.assert_allclose(host["iv"], ref["iv"], rtol=1e-4, atol=1e-9)
    assert np.array_equal(host["keep"], ref["keep"])
    print(which, "prefill-fused compression report", rep)


def test_prefill_rejects_unsupported(A):
    wl = W.make("tiny", device="cuda")  # fp32, D = 64
    prob = problem(A, wl)
    s = wl.spec
    q = torch.zeros((s.L, wl.total_tokens, s.H_q, s.D), dtype=torch.float32, device="cuda")
    attn = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    ws = prob.new_workspace()
    with pytest.raises(A.AirCacheError) as e:
        A.aircache_prefill(prob, q, attn, ws)
    assert e.value.status == A.ERR_UNSUPPORTED
