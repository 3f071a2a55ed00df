"""GPU parity of the visual observation window (reading R14: the last 32
visual tokens' queries over the visual keys; variant window 4, q_visual)."""
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


@pytest.mark.parametrize("name,layers,requests,prefix", [("7b", 4, None, False), ("ragged", 2, 4, False),
                                                         ("ragged", 2, 3, True)])
def test_visual_window_matches_the_oracle(A, oracle, name, layers, requests, prefix):
    wl = W.make(name, seed=51, device="cuda", layers=layers, requests=requests)
    s = wl.spec
    qv = W.visual_queries(wl, seed=52)
    npf = [min(7 * b, t) for b, t in enumerate(s.n_text)] if prefix else [0] * s.B
    k, v, npt = W.with_prefix(wl, npf) if prefix else (wl.k, wl.v, None)
    prob = A.Problem(wl.q, k, v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text), s.alpha, s.r,
                     total_tokens=wl.total_tokens, total_visual=wl.total_visual, window_mode=4, q_visual=qv,
                     n_prefix=npt)
    out = A.compress(prob)
    cu_s, cu_v, cu_t = W.offsets(s)
    iv = out["iv"].cpu().numpy().astype(np.float64)
    keep = out["keep"].cpu().numpy()
    offs = out["out_offsets"].cpu().numpy()
    ok = W.host_bits(out["out_k"])
    for b in range(s.B):
        q = [W.host_bits(wl.q[l, cu_t[b]:cu_t[b + 1]]) for l in range(s.L)]
        kb = [W.host_bits(k[l, cu_s[b]:cu_s[b + 1]]) for l in range(s.L)]
        qvb = [W.host_bits(qv[l, cu_v[b]:cu_v[b + 1]]) for l in range(s.L)]
        ref = oracle.request(q, kb, s.n_visual[b], s.alpha, s.r, window_mode=4, qv_layers=qvb, n_p=npf[b])
        for l in range(s.L):
            u = l * s.B + b
            gi = iv[l, cu_v[b]:cu_v[b + 1]]
            PU.check_iv(ref["iv"][l], gi, f"request {b} layer {l}")
            kk = int(keep[u])
            sel = oracle.select(gi, kk)
            assert np.array_equal(out["idx"][l, cu_v[b]:cu_v[b] + kk].cpu().numpy(), sel)
            rows = oracle.compact(kb[l], s.n_visual[b], s.n_text[b], sel, n_p=npf[b])
            assert np.array_equal(ok[offs[u]:offs[u + 1]], rows)


def test_visual_window_needs_the_visual_queries(A):
    wl = W.make("ragged", seed=53, device="cuda", layers=1, requests=2)
    s = wl.spec
    with pytest.raises(A.AirCacheError):
        prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text), s.alpha,
                         s.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual, window_mode=4)
        A.compress(prob)
