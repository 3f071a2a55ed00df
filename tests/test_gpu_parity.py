"""GPU parity: the CUDA library through its C ABI against the fp64 oracle.

Every case draws seeded synthetic inputs on the GPU, runs the staged entry
points (score -> budget -> select -> compact) and the fused aircache_compress,
checks that both agree bit for bit, and compares them with the oracle under the
acceptance rules in parity_utils."""
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


def make_problem(A, wl, **kw):
    s = wl.spec
    args = dict(alpha=s.alpha, r=s.r)
    args.update(kw)
    return A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text),
                     total_tokens=wl.total_tokens, total_visual=wl.total_visual, **args)


def run_staged(A, prob):
    dev = prob.layers[1][0].device
    L, B, TV = prob.L, prob.B, prob.total_visual
    ws = prob.new_workspace()
    iv = torch.full((L, TV), float("nan"), dtype=torch.float32, device=dev)
    elite = torch.full((L * B, prob.max_text), -1, dtype=torch.int32, device=dev)
    n_tk = torch.zeros(L * B, dtype=torch.int32, device=dev)
    A.aircache_score(prob, ws, iv, elite, n_tk)
    assert A.aircache_get_error(ws) == 0
    stats = torch.zeros((L * B, 2), dtype=torch.float64, device=dev)
    keep = torch.zeros(L * B, dtype=torch.int32, device=dev)
    A.aircache_budget(prob, iv, ws, stats, keep)
    assert A.aircache_get_error(ws) == 0
    idx = torch.full((L, TV), -1, dtype=torch.int32, device=dev)
    A.aircache_select(prob, iv, keep, ws, idx)
    assert A.aircache_get_error(ws) == 0
    rows = prob.compress_bound()
    out_k = torch.empty((rows, prob.h_kv, prob.d), dtype=prob.dtype, device=dev)
    out_v = torch.empty_like(out_k)
    offs = torch.empty(L * B + 1, dtype=torch.int64, device=dev)
    A.aircache_compact(prob, idx, keep, ws, out_k, out_v, offs)
    assert A.aircache_get_error(ws) == 0
    out = {"iv": iv, "keep": keep, "idx": idx, "out_k": out_k, "out_v": out_v, "out_offsets": offs}
    return PU.gpu_to_host(out, prob, n_tk=n_tk, elite=elite, stats=stats)


def run_fused(A, prob):
    out = A.compress(prob)
    return PU.gpu_to_host(out, prob)


def assert_same(staged, fused, prob):
    assert np.array_equal(staged["iv"], fused["iv"], equal_nan=True)
    assert np.array_equal(staged["keep"], fused["keep"])
    assert np.array_equal(staged["out_offsets"], fused["out_offsets"])
    for l in range(prob.L):
        for b in range(prob.B):
            u = l * prob.B + b
            kp = int(staged["keep"][u])
            v0 = int(prob.cu_visual[b])
            assert np.array_equal(staged["idx"][l, v0:v0 + kp], fused["idx"][l, v0:v0 + kp])
    assert np.array_equal(staged["out_k"], fused["out_k"])
    assert np.array_equal(staged["out_v"], fused["out_v"])


def full_check(A, oracle, wl, units="all", compact_units="all", score_requests=None, strict=True, **kw):
    window_mode, budget_mode = kw.get("window_mode", 0), kw.get("budget_mode", 0)
    prob = make_problem(A, wl, **kw)
    staged = run_staged(A, prob)
    fused = run_fused(A, prob)
    assert_same(staged, fused, prob)
    spec = wl.spec
    cu_s, cu_v, _ = W.offsets(spec)
    assert np.array_equal(staged["out_offsets"], PU.expected_offsets(spec, staged["keep"]))
    all_units = [(l, b) for l in range(spec.L) for b in range(spec.B)]
    chk = all_units if units == "all" else units
    report = {}
    oracle_iv = {}
    for (l, b) in chk:
        oracle_iv[(l, b)] = PU.check_unit(oracle, wl, l, b, cu_s, cu_v, staged, report, window_mode)
    reqs = range(spec.B) if score_requests is None else score_requests
    for b in reqs:
        by_layer = {l: oracle_iv[(l, b)] for l in range(spec.L) if (l, b) in oracle_iv}
        PU.check_request(oracle, wl, b, cu_s, cu_v, staged, report, by_layer, budget_mode)
    cu = all_units if compact_units == "all" else compact_units
    for (l, b) in cu:
        PU.check_compaction(oracle, wl, l, b, cu_s, cu_v, staged)
    if strict:
        # no keep count may rest on a rounding exemption: every one equals the
        # oracle's budget on the GPU's I_v and on the oracle's own I_v
        assert report.get("near_half_exempt", 0) == 0, report
        assert report.get("keep_boundary", 0) == 0, report
    return staged, report


def test_tiny_fp32(A, oracle):
    wl = W.make("tiny", device="cuda")
    _, rep = full_check(A, oracle, wl)
    print("tiny report", rep)


@pytest.mark.parametrize("name,layers,requests", [
    ("7b", 3, None), ("llama_mha", 2, 2), ("video_r01", 2, 1), ("video_r10", 2, 2), ("ragged", 2, 7),
])
def test_reduced_configs(A, oracle, name, layers, requests):
    wl = W.make(name, device="cuda", layers=layers, requests=requests)
    _, rep = full_check(A, oracle, wl)
    print(name, "report", rep)


def test_7b_full_size(A, oracle):
    """The benchmarked workload at full size: I_v of every layer against the
    oracle, every budget and selection, and compaction of a sample of layers."""
    wl = W.make("7b", device="cuda")
    comp = [(l, 0) for l in (0, 9, 27)]
    _, rep = full_check(A, oracle, wl, compact_units=comp)
    print("7b full report", rep)


@pytest.mark.parametrize("name", ["llama_mha", "video_r01", "video_r10", "ragged"])
def test_full_size_sampled(A, oracle, name):
    """Full-size configurations: I_v on sampled (layer, request) units, budgets
    and selections of every request on the GPU's I_v, sampled compaction."""
    wl = W.make(name, device="cuda")
    s = wl.spec
    rng = np.random.default_rng(1)
    units = sorted({(int(rng.integers(s.L)), int(rng.integers(s.B))) for _ in range(4)})
    _, rep = full_check(A, oracle, wl, units=units, compact_units=units)
    print(name, "report", rep)


def test_streaming_path_kernels(A):
    """The 7b-shaped problem (bf16, evenly strided layers) takes the streaming
    path: the zeroing kernel, the elite step, the three scoring passes, the
    selection and the compaction."""
    wl = W.make("7b", device="cuda", layers=2)
    prob = make_problem(A, wl)
    assert A.kernel_names(prob) == ["zero_block", "elite_window", "score_pass1", "score_pass2", "score_pass2k",
                                    "budget_select", "gather_compact"]


def test_deterministic(A):
    wl = W.make("7b", device="cuda", layers=4)
    prob = make_problem(A, wl)
    a = run_fused(A, prob)
    b = run_fused(A, prob)
    for key in ("iv", "keep", "idx", "out_offsets", "out_k", "out_v"):
        assert np.array_equal(a[key], b[key], equal_nan=True), key


def test_values_in_pinned_host_memory(A):
    """Values left in page-locked host memory (read in place by the compaction,
    the kept rows only): the same compressed cache, bit for bit, as with every
    value in device memory; also through the host-tensor API."""
    wl = W.make("7b", device="cuda", layers=3)
    dev_out = run_fused(A, make_problem(A, wl))
    hv = wl.v.cpu().pin_memory()
    s = wl.spec
    prob_h = A.Problem(wl.q, wl.k, hv, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text),
                       s.alpha, s.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual)
    host_out = run_fused(A, prob_h)
    for key in ("iv", "keep", "idx", "out_offsets", "out_k", "out_v"):
        assert np.array_equal(dev_out[key], host_out[key], equal_nan=True), key
    ok_, ov_, of_ = A.compress_host(wl.q.cpu(), wl.k.cpu(), hv, wl.cu_seqlens.cpu(), wl.cu_visual.cpu(),
                                    max(s.n_visual), max(s.n_text), s.alpha, s.r)
    rows = int(of_[-1])
    assert np.array_equal(W.host_bits(ok_[:rows]), dev_out["out_k"][:rows])
    assert np.array_equal(W.host_bits(ov_[:rows]), dev_out["out_v"][:rows])


def test_prefill_rejects_values_in_host_memory(A):
    """The prefill attention reads every value: host-resident values are refused."""
    wl = W.make("7b", device="cuda", layers=1)
    s = wl.spec
    hv = wl.v.cpu().pin_memory()
    prob_h = A.Problem(wl.q, wl.k, hv, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text),
                       s.alpha, s.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual)
    q_all = torch.zeros((s.L, wl.total_tokens, s.H_q, s.D), dtype=s.dtype, device="cuda")
    attn = torch.empty_like(q_all)
    with pytest.raises(A.AirCacheError) as e:
        A.aircache_prefill(prob_h, q_all, attn, prob_h.new_workspace())
    assert e.value.status == A.ERR_UNSUPPORTED


# ------------------------------------------------------------------ edge cases

def custom_workload(n_visual, n_text, L=2, H_q=8, H_kv=2, D=128, dtype=torch.bfloat16, seed=0,
                    alpha=0.9, r=0.1, scale=1.0):
    spec = W.Spec("custom", len(n_visual), L, H_q, H_kv, D, list(n_visual), list(n_text), dtype,
                  alpha, r, entry_std=scale, heavy_frac=0.1, heavy_bias=1.5, layer_scale=(0.5, 2.0))
    return W.generate(spec, seed=seed, device="cuda")


def test_alpha_zero_many_row_chunks(A, oracle):
    """alpha = 0: every text token is elite, so the query rows of one KV head
    span several row chunks."""
    wl = custom_workload([300, 131], [40, 17], H_q=28, H_kv=4, alpha=0.0)
    staged, _ = full_check(A, oracle, wl)
    assert staged["n_tk"].tolist() == [40, 17] * 2


def test_mixed_narrow_and_wide_units(A, oracle):
    """alpha = 0 with one short and one long text: request 0's units have
    g * N_tk = 21 query rows per KV head (narrow scoring path), request 1's
    have 7 * 17 = 119 (wide path), in every layer; budgets and offsets span
    both paths."""
    wl = custom_workload([700, 390], [3, 17], L=3, H_q=28, H_kv=4, alpha=0.0)
    staged, _ = full_check(A, oracle, wl)
    assert staged["n_tk"].tolist() == [3, 17] * 3


def test_narrow_two_row_tiles(A, oracle):
    """MHA-style g = 1 with 20 elite rows per KV head: the narrow path's
    second 16-row m-tile and a ragged last key tile."""
    wl = custom_workload([1000, 333], [20, 25], L=2, H_q=4, H_kv=4, alpha=0.0)
    staged, _ = full_check(A, oracle, wl)
    assert staged["n_tk"].tolist() == [20, 25] * 2


def test_many_elite_text_tiles(A, oracle):
    """alpha = 0 with 200 text tokens: the elite text keys span two 128-key
    tiles and the rows of one KV head span 25 row chunks."""
    wl = custom_workload([300], [200], L=2, H_q=8, H_kv=2, alpha=0.0)
    staged, _ = full_check(A, oracle, wl)
    assert staged["n_tk"].tolist() == [200, 200]


def test_alpha_one(A, oracle):
    wl = custom_workload([257, 64], [33, 5], alpha=1.0)
    full_check(A, oracle, wl)


def test_minimum_lengths(A, oracle):
    wl = custom_workload([3, 3, 5], [1, 2, 1], L=3)
    full_check(A, oracle, wl)


def test_keep_everything_and_keep_one(A, oracle):
    wl = custom_workload([200, 70], [12, 9], r=1.0)
    staged, _ = full_check(A, oracle, wl)
    wl2 = custom_workload([200, 70], [12, 9], r=1e-4)
    staged2, _ = full_check(A, oracle, wl2)
    assert staged2["keep"].max() <= 2


def test_long_visual_span_unstaged_select(A, oracle):
    """30,000 visual positions: more keys than the selection stages in shared
    memory, so its radix passes and emission read I_v from global memory."""
    wl = custom_workload([30000, 500], [16, 8], L=2, H_q=4, H_kv=2)
    full_check(A, oracle, wl)


def test_long_visual_span_ties(A, oracle):
    """Zero queries over 30,000 visual positions: every I_v of a unit is equal,
    so the unstaged selection keeps the lowest positions."""
    wl = custom_workload([30000], [6], L=2, H_q=4, H_kv=2)
    wl.q.zero_()
    staged, _ = full_check(A, oracle, wl)
    for l in range(2):
        kp = int(staged["keep"][l])
        assert staged["idx"][l, :kp].tolist() == list(range(kp))


def test_zero_queries_give_ties(A, oracle):
    wl = custom_workload([150], [10], L=2)
    wl.q.zero_()
    staged, _ = full_check(A, oracle, wl)
    for l in range(2):
        kp = int(staged["keep"][l])
        assert staged["idx"][l, :kp].tolist() == list(range(kp))


def test_head_dim_64_bf16(A, oracle):
    wl = custom_workload([500, 97], [24, 30], D=64, H_q=12, H_kv=3)
    full_check(A, oracle, wl)


def test_fp32_head_dim_128(A, oracle):
    wl = custom_workload([190, 65], [20, 7], D=128, dtype=torch.float32, scale=0.1)
    full_check(A, oracle, wl)


def test_mha_single_head_group(A, oracle):
    wl = custom_workload([333], [29], H_q=4, H_kv=4, D=128)
    full_check(A, oracle, wl)


def test_strided_fused_kv_layout(A, oracle):
    """K and V as views of one fused [L, T, 2, H_kv, D] buffer (token stride 2*H_kv*D)."""
    wl = custom_workload([260, 90], [19, 23])
    kv = torch.stack([wl.k, wl.v], dim=2).contiguous()
    wl.k = kv[:, :, 0]
    wl.v = kv[:, :, 1]
    assert wl.k.stride(1) == 2 * 2 * 128
    full_check(A, oracle, wl)


def _uneven_layers(t):
    """Copies of the layers of a stacked [L, ...] tensor placed at unevenly spaced
    offsets of one buffer (so no single layer stride describes them)."""
    L, n = t.shape[0], t[0].numel()
    offs = [l * n + 64 * l * l for l in range(L)]  # 64 elements: keeps 16-byte alignment
    buf = torch.empty(offs[-1] + n, dtype=t.dtype, device=t.device)
    return [buf[o:o + n].view(t.shape[1:]).copy_(t[l]) for l, o in enumerate(offs)]


def test_unevenly_placed_layers(A, oracle):
    """Per-layer K/V/Q at uneven addresses: the scoring kernel cannot use one
    tensor map over the layers and copies its stages with cp.async instead."""
    wl = custom_workload([700, 129], [25, 40], L=3, H_q=28, H_kv=4)
    wl.q, wl.k, wl.v = _uneven_layers(wl.q), _uneven_layers(wl.k), _uneven_layers(wl.v)
    full_check_lists(A, oracle, wl)


def full_check_lists(A, oracle, wl):
    """full_check for per-layer lists (the generator's stacked tensors replaced)."""
    s = wl.spec
    prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text),
                     alpha=s.alpha, r=s.r, total_tokens=wl.k[0].shape[0], total_visual=sum(s.n_visual))
    staged = run_staged(A, prob)
    fused = run_fused(A, prob)
    assert_same(staged, fused, prob)
    stacked = W.Workload(s, torch.stack(wl.q), torch.stack(wl.k), torch.stack(wl.v), wl.cu_seqlens, wl.cu_visual)
    cu_s, cu_v, _ = W.offsets(s)
    report = {}
    oiv = {}
    for l in range(s.L):
        for b in range(s.B):
            oiv[(l, b)] = PU.check_unit(oracle, stacked, l, b, cu_s, cu_v, staged, report)
    for b in range(s.B):
        PU.check_request(oracle, stacked, b, cu_s, cu_v, staged, report, {l: oiv[(l, b)] for l in range(s.L)})
        for l in range(s.L):
            PU.check_compaction(oracle, stacked, l, b, cu_s, cu_v, staged)
    return staged, report


def test_device_errors_reported(A):
    wl = custom_workload([100, 50], [10, 8])
    s = wl.spec
    # elite larger than the workspace cap
    prob = make_problem(A, wl, alpha=0.0, max_elite=4)
    ws = prob.new_workspace()
    out = A.alloc_outputs(prob)
    A.aircache_compress(prob, ws, out["out_k"], out["out_v"], out["out_offsets"], out["keep"])
    assert A.aircache_get_error(ws) == A.ERR_ELITE_OVERFLOW
    # inconsistent offsets on the device
    prob = make_problem(A, wl)
    bad = wl.cu_visual.clone()
    bad[1] = 2  # request 0 with two visual tokens
    prob.c.cu_visual = bad.data_ptr()
    ws = prob.new_workspace()
    A.aircache_compress(prob, ws, out["out_k"], out["out_v"], out["out_offsets"], out["keep"])
    assert A.aircache_get_error(ws) == A.ERR_DEVICE_BOUNDS
    # output arena too small
    prob = make_problem(A, wl)
    ws = prob.new_workspace()
    small_k = out["out_k"][:10]
    small_v = out["out_v"][:10]
    A.aircache_compress(prob, ws, small_k, small_v, out["out_offsets"], out["keep"])
    assert A.aircache_get_error(ws) == A.ERR_CAPACITY
    # the same workspace is usable again after an error
    A.aircache_compress(prob, ws, out["out_k"], out["out_v"], out["out_offsets"], out["keep"])
    assert A.aircache_get_error(ws) == 0
    del s


# ------------------------------------------------------- ablation variants

@pytest.mark.parametrize("window_mode", [1, 2, 3])
def test_ablation_windows(A, oracle, window_mode):
    """AirCache notes, "Ablation studies", observation windows: the last 16 /
    32 text tokens or every text token take the elite set's place (texts of
    40 and 9 tokens: a window longer and shorter than the text)."""
    wl = custom_workload([500, 257], [40, 9], L=3, H_q=8, H_kv=2)
    staged, rep = full_check(A, oracle, wl, window_mode=window_mode)
    assert staged["n_tk"].tolist() == [min(w, n) for w in [{1: 16, 2: 32, 3: 10**9}[window_mode]]
                                       for n in (40, 9)] * 3


@pytest.mark.parametrize("budget_mode", [1, 2, 3, 4])
def test_ablation_budgets(A, oracle, budget_mode):
    """AirCache notes, "Ablation studies", layer budgets: uniform, PyramidKV-
    style, strength only, skewness only (bf16 and fp32 paths)."""
    wl = custom_workload([600, 333], [12, 20], L=5, H_q=8, H_kv=2)
    full_check(A, oracle, wl, budget_mode=budget_mode)
    wl32 = custom_workload([200], [7], L=4, H_q=4, H_kv=4, D=64, dtype=torch.float32)
    full_check(A, oracle, wl32, budget_mode=budget_mode)


def test_ablation_window_and_budget_on_7b_layers(A, oracle):
    """A window and a budget variant together on the 7B-shaped workload
    (4 layers), both scoring paths' unit kinds included."""
    wl = W.make("7b", device="cuda", layers=4)
    full_check(A, oracle, wl, window_mode=2, budget_mode=2)
