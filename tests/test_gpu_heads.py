"""GPU parity of one index set per KV head (reading R19: group-wise top-k;
variant bits 16-23 = 1, aircache_compress on the streaming path).

Per (layer, request, KV head) the GPU's set must equal the oracle's selection
on the oracle's per-KV-group I_v up to swaps whose I_v gap lies within the I_v
tolerance, and each head's compacted rows must be, bit for bit, the rows that
set names.  The layer's I_v and keep counts are those of the shared-set mode."""
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


def run(A, wl, head_sets):
    s = wl.spec
    prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text), s.alpha, s.r,
                     total_tokens=wl.total_tokens, total_visual=wl.total_visual, head_sets=head_sets)
    out = A.compress(prob)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name,layers,requests", [("7b", 4, None), ("ragged", 3, 4), ("llama_mha", 2, 2)])
def test_per_head_sets_match_the_oracle(A, oracle, name, layers, requests):
    wl = W.make(name, seed=41, device="cuda", layers=layers, requests=requests)
    s = wl.spec
    shared = run(A, wl, False)
    out = run(A, wl, True)
    assert torch.equal(shared["iv"], out["iv"]) and torch.equal(shared["keep"], out["keep"])
    assert torch.equal(shared["out_offsets"], out["out_offsets"])
    cu_s, cu_v, cu_t = W.offsets(s)
    keep = out["keep"].cpu().numpy()
    offs = out["out_offsets"].cpu().numpy()
    idx = out["idx"].cpu().numpy()          # [L, H_kv, total_visual]
    ok, ov = W.host_bits(out["out_k"]), W.host_bits(out["out_v"])
    # the oracle on a sample of requests (all of them for the small cases)
    for b in (range(s.B) if s.B <= 4 else [0, s.B - 1]):
        q = [W.host_bits(wl.q[l, cu_t[b]:cu_t[b + 1]]) for l in range(s.L)]
        k = [W.host_bits(wl.k[l, cu_s[b]:cu_s[b + 1]]) for l in range(s.L)]
        v = [W.host_bits(wl.v[l, cu_s[b]:cu_s[b + 1]]) for l in range(s.L)]
        ref = oracle.request(q, k, s.n_visual[b], s.alpha, s.r, per_head=True)
        for l in range(s.L):
            u = l * s.B + b
            kk = int(keep[u])
            sets = idx[l, :, cu_v[b]:cu_v[b] + kk]
            for h in range(s.H_kv):
                PU.check_selection_vs_oracle_iv(ref["iv_heads"][l][h], sets[h], kk)
            rows_k = oracle.compact_heads(k[l], s.n_visual[b], s.n_text[b], sets)
            rows_v = oracle.compact_heads(v[l], s.n_visual[b], s.n_text[b], sets)
            assert np.array_equal(ok[offs[u]:offs[u + 1]], rows_k), f"layer {l} request {b}: K rows"
            assert np.array_equal(ov[offs[u]:offs[u + 1]], rows_v), f"layer {l} request {b}: V rows"


def test_per_head_sets_refuse_the_wide_path(A):
    wl = W.make("tiny", seed=42, device="cuda")  # fp32: the wide scoring path
    with pytest.raises(A.AirCacheError):
        run(A, wl, True)
