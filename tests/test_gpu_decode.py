"""GPU parity of the decode step (aircache_decode) against the fp64 oracle.

Acceptance rule, derived from the kernel's arithmetic: the kernel rounds each
softmax weight to bf16 (8 significant bits, so unit roundoff u = 2^-8) and
normalises by the sum of
the rounded weights, so its output is an exact convex combination whose
weights are the oracle's, each perturbed by a relative error of at most u
(plus 2^-21 for the base-2 exponential and the fp32 logit).  Hence, per
element,
    |o - o*| <= u' / (1 - u') * sum_j w_j |v_j - o*|,   u' = 1.02 u,
and the fp32 accumulation adds a few ulps of max |v|.  Where every weight is
exactly representable (a zero query: all weights 1), the output is the exact
mean and the test asks for fp32 rounding only."""
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


def bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def tolerance(q, k, v, o_ref):
    """The per-element bound of the module docstring for one sequence: q [H_q, D]
    bits, k / v [n, H_kv, D] bits, o_ref [H_q, D]."""
    h_q, d = q.shape
    g = h_q // k.shape[1]
    qf, kf, vf = bf16_to_f64(q), bf16_to_f64(k), bf16_to_f64(v)
    tol = np.zeros((h_q, d))
    for h in range(h_q):
        x = kf[:, h // g] @ qf[h] / np.sqrt(d)
        w = np.exp(x - x.max())
        w /= w.sum()
        spread = w @ np.abs(vf[:, h // g] - o_ref[h])
        tol[h] = U / (1 - U) * spread + 1e-6 * np.abs(vf[:, h // g]).max()
    return tol


def run(A, di, max_rows, **kw):
    prob = A.DecodeProblem(di.q, di.k, di.v, offsets=di.offsets, max_rows=max_rows,
                           k_new=di.k_new, v_new=di.v_new, **kw)
    out = A.decode(prob)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), prob


def check_against_oracle(oracle, di, out, seqs=None):
    offs = di.offsets.cpu().numpy()
    qb, kb, vb = W.host_bits(di.q), W.host_bits(di.k), W.host_bits(di.v)
    knb = W.host_bits(di.k_new) if di.k_new is not None else None
    vnb = W.host_bits(di.v_new) if di.v_new is not None else None
    for s in (range(len(offs) - 1) if seqs is None else seqs):
        b, e = int(offs[s]), int(offs[s + 1])
        k, v = kb[b:e], vb[b:e]
        if knb is not None:
            k = np.concatenate([k, knb[s:s + 1]])
            v = np.concatenate([v, vnb[s:s + 1]])
        if len(k) == 0:
            assert np.all(out[s] == 0.0), f"sequence {s}: empty cache must give zeros"
            continue
        ref = oracle.decode(qb[s], k, v)
        tol = tolerance(qb[s], k, v, ref)
        err = np.abs(out[s] - ref)
        assert np.all(err <= tol), (f"sequence {s} ({e - b} rows): max err {err.max():.3e}, "
                                    f"worst err/tol {(err / tol).max():.2f}")


LENGTHS = [1, 2, 15, 16, 17, 63, 64, 65, 127, 129, 300, 1000, 2500]


@pytest.mark.parametrize("h_q,h_kv,d", [(28, 4, 128), (8, 8, 128), (32, 2, 128), (10, 2, 64), (16, 16, 64)])
def test_decode_matches_oracle_ragged(A, oracle, h_q, h_kv, d):
    di = W.decode_inputs(LENGTHS, h_q, h_kv, d, seed=1, device="cuda", q_scale=2.0)
    out, _ = run(A, di, max_rows=max(LENGTHS))
    check_against_oracle(oracle, di, out)


@pytest.mark.parametrize("max_rows", [0, 64, 300, 1000, 5000, 10 ** 6])
def test_split_count_does_not_change_results_beyond_rounding(A, oracle, max_rows):
    # the hint only moves the split points
    di = W.decode_inputs([700, 33, 4100], 28, 4, 128, seed=2, device="cuda", q_scale=2.0)
    out, prob = run(A, di, max_rows=max_rows)
    assert prob.splits() >= 1
    check_against_oracle(oracle, di, out)


def test_rows_past_a_range_are_never_mixed_in(A, oracle):
    # NaN rows after the last sequence (and every other sequence's rows) share
    # tiles with the ranges' tails
    di = W.decode_inputs([5, 70, 131], 28, 4, 128, seed=3, device="cuda", nan_tail=200)
    out, _ = run(A, di, max_rows=131)
    assert np.isfinite(out).all()
    check_against_oracle(oracle, di, out)


@pytest.mark.parametrize("n", [1, 17, 4096, 40000])
def test_zero_query_gives_the_exact_mean(A, n):
    # all weights are exactly 1: out = mean of the value rows; integer values
    # keep every fp32 sum exact
    di = W.decode_inputs([n, 3], 14, 2, 128, seed=4, device="cuda")
    di.q.zero_()
    vals = torch.randint(-8, 9, di.v.shape, generator=torch.Generator(device="cuda").manual_seed(5),
                         device="cuda")
    di.v.copy_(vals.to(torch.bfloat16))
    out, _ = run(A, di, max_rows=n)
    offs = di.offsets.cpu().numpy()
    v = di.v.float().cpu().numpy().astype(np.float64)
    for s in range(2):
        mean = v[offs[s]:offs[s + 1]].mean(0)          # [H_kv, D]
        expect = np.repeat(mean, 7, axis=0)
        np.testing.assert_allclose(out[s], expect, rtol=3e-7, atol=1e-7)


@pytest.mark.parametrize("pos", [0, 63, 64, 1000, 2047])
def test_needle_row_dominates(A, pos):
    # one row aligned with the query at a large logit takes (almost) all weight
    n, d = 2048, 128
    di = W.decode_inputs([n], 7, 1, d, seed=6, device="cuda")
    di.q.copy_((torch.ones_like(di.q, dtype=torch.float32) * 0.5).to(torch.bfloat16))
    di.k[pos] = 8.0  # logit 0.5*8*128/sqrt(128) ~ 45 above the others (~N(0, 0.5^2))
    out, _ = run(A, di, max_rows=n)
    np.testing.assert_allclose(out[0], np.broadcast_to(di.v[pos, 0].float().cpu().numpy(), (7, d)),
                               rtol=0, atol=1e-5)


def test_new_row_and_empty_ranges(A, oracle):
    di = W.decode_inputs([0, 1, 90, 0, 300], 28, 4, 128, seed=7, device="cuda", new_row=True, q_scale=2.0)
    out, _ = run(A, di, max_rows=300)
    check_against_oracle(oracle, di, out)
    # an empty range with the new row: its value row, exactly
    vn = di.v_new.float().cpu().numpy()
    assert np.array_equal(out[0], np.repeat(vn[0], 7, axis=0).astype(np.float64))


def test_empty_sequences_without_new_row_are_zero(A, oracle):
    di = W.decode_inputs([0, 40, 0], 8, 2, 64, seed=8, device="cuda")
    out, _ = run(A, di, max_rows=40)
    check_against_oracle(oracle, di, out)


def test_strided_query_and_padded_arena(A, oracle):
    # q as a head-slice of a wider tensor, K/V arenas with an unused head
    g = torch.Generator(device="cuda").manual_seed(9)
    S, h_q, h_kv, d = 3, 28, 4, 128
    qw = torch.randn((S, h_q + 4, d), generator=g, device="cuda").to(torch.bfloat16)
    kw = torch.randn((500, h_kv + 1, d), generator=g, device="cuda").to(torch.bfloat16)
    vw = torch.randn((500, h_kv + 1, d), generator=g, device="cuda").to(torch.bfloat16)
    q, k, v = qw[:, 2:2 + h_q], kw[:, :h_kv], vw[:, :h_kv]
    offs = torch.tensor([0, 120, 121, 500], dtype=torch.int64, device="cuda")
    prob = A.DecodeProblem(q, k, v, offsets=offs, max_rows=400)
    out = A.decode(prob).cpu().numpy().astype(np.float64)
    di = W.DecodeInputs(q.contiguous(), k.contiguous(), v.contiguous(), offs)
    check_against_oracle(oracle, di, out)


def test_out_of_bounds_range_sets_the_error_word(A, oracle):
    di = W.decode_inputs([10, 20], 8, 2, 64, seed=10, device="cuda")
    begin = di.offsets[:-1].clone()
    end = di.offsets[1:].clone()
    end[1] = di.k.shape[0] + 5  # past the arena
    prob = A.DecodeProblem(di.q, di.k, di.v, row_begin=begin, row_end=end, max_rows=20)
    ws = prob.new_workspace()
    A.aircache_decode(prob, ws)
    assert A.aircache_get_error(ws) == A.ERR_DEVICE_BOUNDS
    out = prob.out.cpu().numpy().astype(np.float64)
    assert np.all(out[1] == 0.0)
    check_against_oracle(oracle, di, out, seqs=[0])
    # the error stays recorded until the caller zeroes the workspace
    prob2 = A.DecodeProblem(di.q, di.k, di.v, offsets=di.offsets, max_rows=20)
    A.aircache_decode(prob2, ws)
    assert A.aircache_get_error(ws) == A.ERR_DEVICE_BOUNDS
    ws.zero_()
    A.aircache_decode(prob2, ws)
    assert A.aircache_get_error(ws) == A.OK
    check_against_oracle(oracle, di, prob2.out.cpu().numpy().astype(np.float64))


def test_workspace_reused_across_calls_and_split_modes(A, oracle):
    # one zeroed workspace serves calls in every merge mode back to back (the
    # global-merge counters reset themselves)
    di = W.decode_inputs([3000, 50, 7000], 28, 4, 128, seed=14, device="cuda", q_scale=2.0)
    probs = [A.DecodeProblem(di.q, di.k, di.v, offsets=di.offsets, max_rows=m) for m in (0, 1000, 10 ** 6)]
    assert [p.splits() for p in probs][0] == 1 and probs[2].splits() > 8
    ws = torch.zeros(max(p.workspace_size() for p in probs), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        for p in probs:
            A.aircache_decode(p, ws)
    assert A.aircache_get_error(ws) == A.OK
    assert int(ws[256:512].view(torch.int32).abs().sum()) == 0
    for p in probs:
        check_against_oracle(oracle, di, p.out.cpu().numpy().astype(np.float64))


def test_decode_over_the_compressed_arena(A, oracle):
    # the consumer reads aircache_compress's output directly: per layer,
    # row ranges out_offsets[l*B + b] .. out_offsets[l*B + b + 1]
    wl = W.make("ragged", seed=11, device="cuda", layers=3, requests=4)
    s = wl.spec
    prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text),
                     alpha=s.alpha, r=s.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual)
    res = A.compress(prob)
    offs = res["out_offsets"]
    B, L = prob.B, prob.L
    g = torch.Generator(device="cuda").manual_seed(12)
    qs = torch.randn((L, B, s.H_q, s.D), generator=g, device="cuda").to(torch.bfloat16)
    rows = offs.cpu().numpy()
    kb, vb = W.host_bits(res["out_k"]), W.host_bits(res["out_v"])
    for l in range(L):
        dp = A.DecodeProblem(qs[l], res["out_k"], res["out_v"], row_begin=offs[l * B:(l + 1) * B],
                             row_end=offs[l * B + 1:(l + 1) * B + 1], max_rows=int(np.diff(rows).max()))
        out = A.decode(dp).cpu().numpy().astype(np.float64)
        qb = W.host_bits(qs[l])
        for b in range(B):
            r0, r1 = int(rows[l * B + b]), int(rows[l * B + b + 1])
            ref = oracle.decode(qb[b], kb[r0:r1], vb[r0:r1])
            tol = tolerance(qb[b], kb[r0:r1], vb[r0:r1], ref)
            assert np.all(np.abs(out[b] - ref) <= tol), f"layer {l} request {b}"
    # all layers in one call (num_seqs = L * B) gives the same outputs
    dp = A.DecodeProblem(qs.reshape(L * B, s.H_q, s.D), res["out_k"], res["out_v"], offsets=offs,
                         max_rows=int(np.diff(rows).max()))
    allo = A.decode(dp).cpu().numpy().reshape(L, B, s.H_q, s.D)
    assert np.isfinite(allo).all()


@pytest.mark.parametrize("batch,prompt", [(16, 16384)])
def test_full_size_cache_sampled(A, oracle, batch, prompt):
    # the full-cache shape the decode measurement uses (one layer of it),
    # checked on sampled sequences
    di = W.decode_inputs([prompt] * batch, 28, 4, 128, seed=13, device="cuda", q_scale=2.0)
    out, _ = run(A, di, max_rows=prompt)
    check_against_oracle(oracle, di, out, seqs=[0, batch - 1])


def test_early_cache_launches_match_plain_launches(A, oracle):
    # consecutive calls with programmatic dependent launch (the cache is not
    # written by the kernel before each call) give the same bits as plain ones,
    # also when each call's queries come from the kernel just before it
    di = W.decode_inputs([700, 33, 4100, 5], 28, 4, 128, seed=15, device="cuda", q_scale=2.0, new_row=True)
    outs = {}
    for early in (False, True):
        ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
        res = []
        for m in (0, 1000, 10 ** 6):
            q = torch.empty_like(di.q)
            q.copy_(di.q)  # written by the kernel right before the decode kernel
            p = A.DecodeProblem(q, di.k, di.v, offsets=di.offsets, max_rows=m, k_new=di.k_new, v_new=di.v_new,
                                early_cache=early)
            A.aircache_decode(p, ws)
            res.append(p.out)
        assert A.aircache_get_error(ws) == A.OK
        outs[early] = [r.clone() for r in res]
    for a, b in zip(outs[False], outs[True]):
        assert torch.equal(a, b)
    check_against_oracle(oracle, di, outs[True][1].cpu().numpy().astype(np.float64))


def test_gather_fused_decode_equals_decoding_the_compacted_arena(A):
    # decoding layer l's full cache through aircache_row_index's list attends
    # over the same rows, in the same order, as decoding the compacted arena:
    # the same bits
    for with_prefix in (False, True):
        wl = W.make("ragged", seed=16, device="cuda", layers=3, requests=4)
        s = wl.spec
        npf = [min(x, t) for x, t in zip([3, 0, 60, 11], s.n_text)]
        k, v, npt = W.with_prefix(wl, npf) if with_prefix else (wl.k, wl.v, None)
        prob = A.Problem(wl.q, k, v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text),
                         alpha=s.alpha, r=s.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual,
                         n_prefix=npt)
        res = A.compress(prob)
        ri = A.row_index(prob, res)
        offs = res["out_offsets"]
        rows = offs.cpu().numpy()
        B = s.B
        g = torch.Generator(device="cuda").manual_seed(17)
        qs = torch.randn((s.L, B, s.H_q, s.D), generator=g, device="cuda").to(torch.bfloat16)
        longest = int(np.diff(rows).max())
        for l in range(s.L):
            rb, re = offs[l * B:(l + 1) * B], offs[l * B + 1:(l + 1) * B + 1]
            a = A.decode(A.DecodeProblem(qs[l], res["out_k"], res["out_v"], row_begin=rb, row_end=re,
                                         max_rows=longest))
            b = A.decode(A.DecodeProblem(qs[l], k[l], v[l], row_begin=rb, row_end=re, max_rows=longest,
                                         row_index=ri))
            assert torch.equal(a, b), f"layer {l}"


@pytest.mark.parametrize("max_rows", [0, 1000, 10 ** 6])
def test_gather_decode_of_listed_rows_matches_oracle(A, oracle, max_rows):
    # arbitrary row lists (repeats allowed) over an arena, in every merge mode
    di = W.decode_inputs([3000], 28, 4, 128, seed=18, device="cuda", q_scale=2.0)
    rng = np.random.default_rng(19)
    lens = [1, 70, 129, 1500]
    lists = [rng.integers(0, 3000, n) for n in lens]
    ri = torch.tensor(np.concatenate(lists), dtype=torch.int32, device="cuda")
    offs = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64, device="cuda")
    q = torch.randn((len(lens), 28, 128), generator=torch.Generator(device="cuda").manual_seed(20),
                    device="cuda").to(torch.bfloat16)
    out = A.decode(A.DecodeProblem(q, di.k, di.v, offsets=offs, max_rows=max_rows, row_index=ri))
    out = out.cpu().numpy().astype(np.float64)
    kb, vb, qb = W.host_bits(di.k), W.host_bits(di.v), W.host_bits(q)
    for s_, rows in enumerate(lists):
        ref = oracle.decode(qb[s_], kb[rows], vb[rows])
        assert np.all(np.abs(out[s_] - ref) <= tolerance(qb[s_], kb[rows], vb[rows], ref)), f"sequence {s_}"


def test_gather_row_outside_the_arena_is_a_device_error(A):
    di = W.decode_inputs([100], 8, 2, 64, seed=21, device="cuda")
    ri = torch.tensor([0, 5, 100, 7], dtype=torch.int32, device="cuda")  # 100 is past the arena
    offs = torch.tensor([0, 4], dtype=torch.int64, device="cuda")
    prob = A.DecodeProblem(di.q[:1], di.k, di.v, offsets=offs, max_rows=4, row_index=ri)
    ws = prob.new_workspace()
    A.aircache_decode(prob, ws)
    assert A.aircache_get_error(ws) == A.ERR_DEVICE_BOUNDS
    assert np.isfinite(prob.out.cpu().numpy()).all()


def test_row_index_lists_the_compacted_positions(A):
    wl = W.make("ragged", seed=22, device="cuda", layers=2, requests=3)
    s = wl.spec
    npf = [0, 9, s.n_text[2]]
    k, v, npt = W.with_prefix(wl, npf)
    prob = A.Problem(wl.q, k, v, wl.cu_seqlens, wl.cu_visual, max(s.n_visual), max(s.n_text), alpha=s.alpha,
                     r=s.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual, n_prefix=npt)
    res = A.compress(prob)
    ri = A.row_index(prob, res).cpu().numpy()
    cu_s, cu_v, _ = W.offsets(s)
    keep, idx, offs = res["keep"].cpu().numpy(), res["idx"].cpu().numpy(), res["out_offsets"].cpu().numpy()
    for l in range(s.L):
        for b in range(s.B):
            u = l * s.B + b
            kk, nv, nt, p_ = int(keep[u]), s.n_visual[b], s.n_text[b], npf[b]
            vis = cu_s[b] + p_ + idx[l, cu_v[b]:cu_v[b] + kk]
            txt = cu_s[b] + np.array([j if j < p_ else nv + j for j in range(nt)])
            assert np.array_equal(ri[offs[u]:offs[u + 1]], np.concatenate([vis, txt]))
