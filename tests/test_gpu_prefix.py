"""GPU parity of the visual span at an offset (reading R18: [prefix text]
[visual][other text], through the problem's n_prefix array).

The layout moves rows, not arithmetic: every output of aircache_compress on
the prefix layout must equal, bit for bit, its output on the same tokens laid
out visual-first (the oracle is pinned to the same equivalence), and the
prefix layout is also checked against the oracle directly."""
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


def run(A, wl, k, v, n_prefix=None):
    s = wl.spec
    prob = A.Problem(wl.q, k, v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text), s.alpha, s.r,
                     total_tokens=wl.total_tokens, total_visual=wl.total_visual, n_prefix=n_prefix)
    out = A.compress(prob)
    torch.cuda.synchronize()
    return out


def prefixes(spec, seed):
    rng = np.random.default_rng(seed)
    n = [int(rng.integers(0, t + 1)) for t in spec.n_text]
    n[0] = 0                      # one request without a prefix
    n[-1] = spec.n_text[-1]       # one whose visual span ends the prompt
    return n


@pytest.mark.parametrize("name,layers,requests", [("ragged", 3, 5), ("tiny", None, None), ("7b", 4, None)])
def test_prefix_layout_equals_visual_first(A, name, layers, requests):
    wl = W.make(name, seed=31, device="cuda", layers=layers, requests=requests)
    npf = prefixes(wl.spec, 32) if wl.spec.B > 1 else [min(5, wl.spec.n_text[0])]
    kp, vp, npt = W.with_prefix(wl, npf)
    a = run(A, wl, wl.k, wl.v)
    b = run(A, wl, kp, vp, npt)
    for key in ("iv", "keep", "out_offsets"):
        assert torch.equal(a[key], b[key]), key
    # idx holds keep[l, b] defined entries per unit (the rest of its slots are scratch)
    cu_v = W.offsets(wl.spec)[1]
    keep = a["keep"].cpu().numpy()
    for l in range(wl.spec.L):
        for r in range(wl.spec.B):
            kk = int(keep[l * wl.spec.B + r])
            assert torch.equal(a["idx"][l, cu_v[r]:cu_v[r] + kk], b["idx"][l, cu_v[r]:cu_v[r] + kk])
    rows = int(a["out_offsets"][-1])
    assert torch.equal(a["out_k"][:rows], b["out_k"][:rows])
    assert torch.equal(a["out_v"][:rows], b["out_v"][:rows])


def test_prefix_layout_against_the_oracle(A, oracle):
    wl = W.make("ragged", seed=33, device="cuda", layers=2, requests=3)
    s = wl.spec
    npf = [4, 17, s.n_text[2]]
    kp, vp, npt = W.with_prefix(wl, npf)
    out = run(A, wl, kp, vp, npt)
    cu_s, cu_v, cu_t = W.offsets(s)
    iv = out["iv"].cpu().numpy().astype(np.float64)
    keep = out["keep"].cpu().numpy()
    offs = out["out_offsets"].cpu().numpy()
    ok = W.host_bits(out["out_k"])
    for b in range(s.B):
        q = [W.host_bits(wl.q[l, cu_t[b]:cu_t[b + 1]]) for l in range(s.L)]
        k = [W.host_bits(kp[l, cu_s[b]:cu_s[b + 1]]) for l in range(s.L)]
        ref = oracle.request(q, k, s.n_visual[b], s.alpha, s.r, n_p=npf[b])
        for l in range(s.L):
            u = l * s.B + b
            gi = iv[l, cu_v[b]:cu_v[b + 1]]
            PU.check_iv(ref["iv"][l], gi, f"request {b} layer {l}")
            # selection and compaction on the GPU's own I_v and keep counts
            kk = int(keep[u])
            sel = oracle.select(gi, kk)
            assert np.array_equal(out["idx"][l, cu_v[b]:cu_v[b] + kk].cpu().numpy(), sel)
            rows = oracle.compact(k[l], s.n_visual[b], s.n_text[b], sel, n_p=npf[b])
            assert np.array_equal(ok[offs[u]:offs[u + 1]], rows)


def test_prefix_longer_than_the_text_is_a_device_error(A):
    wl = W.make("ragged", seed=34, device="cuda", layers=1, requests=2)
    npt = torch.tensor([0, wl.spec.n_text[1] + 1], dtype=torch.int32, device="cuda")
    s = wl.spec
    prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text), s.alpha, s.r,
                     total_tokens=wl.total_tokens, total_visual=wl.total_visual, n_prefix=npt)
    with pytest.raises(A.AirCacheError):
        A.compress(prob)
