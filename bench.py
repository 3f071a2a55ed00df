#!/usr/bin/env python
"""Benchmark of the fused AirCache compression (one-shot visual KV compression
after prefill) on GB300.

One step = one aircache_compress call over the whole workload (elite window,
cross-modal scores, layer budgets, top-k, gather-compact), inputs resident in
HBM.  Default workload: the 7B LVLM-shaped batch (1 request, 28 layers,
H_q=28, H_kv=4, D=128, N_v=7290, N_t=128, bf16, alpha=0.9, r=0.10).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank compresses its own
copy of the workload (requests are independent: weak scaling, no collective on
the data path); the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "visual KV tokens compressed/sec on 1 GB300; fused-compress HBM GB/s vs 8 TB/s"
UNIT = "visual KV tokens/s"
L2_FLUSH_BYTES = 256 << 20
DESCRIPTIONS = {
    "7b": "7B LVLM-shaped (Qwen2-7B-like GQA): 1 request, L=28, H_q=28, H_kv=4, D=128, "
          "N_v=7290 visual + N_t=128 text, bf16, 10% heavy visual keys, alpha=0.9, r=0.10",
    "tiny": "tiny: 1 request, L=2, H_q=H_kv=4, D=64, N_v=64, N_t=16, fp32, alpha=0.9, r=0.25",
    "llama_mha": "Llama-7B MHA-shaped batch: 8 requests, L=32, H=32, D=128, N_v=2880, N_t=512, bf16, r=0.10",
    "video_r01": "video-shaped: 4 requests, L=28, H_q=28, H_kv=4, D=128, N_v=12544, N_t=256, bf16, r=0.01",
    "video_r10": "video-shaped: 4 requests, L=28, H_q=28, H_kv=4, D=128, N_v=12544, N_t=256, bf16, r=0.10",
    "ragged": "ragged serving batch: 32 requests, L=28, H_q=28, H_kv=4, D=128, N_v~U[576,9000], "
              "N_t~U[32,1024], bf16, r=0.05",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="7b")
    ap.add_argument("--window-mode", type=int, default=0,
                    help="ablation observation window: 0 elite (the method), 1 last 16, 2 last 32, 3 all text, "
                         "4 the last 32 visual tokens (seeded visual queries)")
    ap.add_argument("--budget-mode", type=int, default=0,
                    help="ablation budget: 0 strength + skewness (the method), 1 uniform, 2 PyramidKV-style, "
                         "3 strength only, 4 skewness only")
    ap.add_argument("--head-sets", action="store_true",
                    help="one visual index set per KV head (group-wise top-k) instead of one per layer")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-s", type=float, default=1.5, help="untimed back-to-back load before timing")
    ap.add_argument("--cpu-sample-s", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="--prefill only: use the workload's first N layers (a small case for profiling)")
    ap.add_argument("--prefill", action="store_true",
                    help="time the causal prefill attention of every layer alone, with the AirCache scoring "
                         "fused in (aircache_prefill_compress), and followed by aircache_compress")
    ap.add_argument("--decode", action="store_true",
                    help="measure the decode consumer instead: one decode step of attention over the full and "
                         "the compressed cache, per decode configuration (one JSON line each)")
    ap.add_argument("--decode-configs", default="8x2048,8x32768,16x16384",
                    help="comma-separated BATCHxPROMPT list for --decode")
    ap.add_argument("--decode-ratios", default="0.1,0.5", help="retention ratios r for --decode")
    ap.add_argument("--decode-layers", type=int, default=28,
                    help="layers of the decode workload (28 = the 7B shape; fewer only for small profiling runs)")
    ap.add_argument("--timeline", action="store_true",
                    help="device timeline of aircache_compress on the measurement build of the library (each "
                         "kernel's CTAs stamp their entry and exit): per kernel, when its CTAs start and end")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = {"score_pass1": "stream.cu", "decode_kernel": "decode.cu"}


def kernel_sources_hash(kernel):
    """Hash of the translation unit that holds `kernel`, every shared header and
    the C ABI header: what the kernel's DRAM traffic depends on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lvlm_kv_cache_gb300", "csrc")
    files = [os.path.join(csrc, KERNEL_SOURCES.get(kernel, ""))]
    files += [os.path.join(csrc, f) for f in sorted(os.listdir(csrc)) if f.endswith(".cuh")]
    files.append(os.path.join(ROOT, "include", "aircache.h"))
    for f in files:
        if not os.path.isfile(f):
            return None
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(config, kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current sources of that kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(config, {}).get(kernel)
    if not e or e.get("sources") != kernel_sources_hash(kernel):
        return None
    return float(e["dram_bytes_per_launch_full"])


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    if int(parts[0]) != self.gpu_index and self.gpu_index is not None:
                        continue
                    rows.append(parts)
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        mx = max(float(r[2]) for r in rows)
        loaded = [s for s in sm if s > 0.5 * mx] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows)}


def max_over_ranks(x, dist, device):
    """The max of a per-rank float over all ranks (the bench's only collective)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, steps, total_ms):
    """Units processed by all ranks per second, timed by the slowest rank."""
    return world * units_per_rank * steps / (total_ms / 1e3)


def unit_lengths(spec):
    return [(spec.n_visual[b], spec.n_text[b]) for b in range(spec.B)]


def algorithmic_bytes(spec, n_tk, keep, esize):
    """Per-kernel algorithmic bytes of one compression (each input read once,
    each output written once; intermediates such as stored logits and
    partials are not counted) and the whole-path total of the per-(request,
    layer) formula 2*H_kv*D*(N_v+N_t) + 2*H_q*D*(1+N_tk) + 8*H_kv*D*(keep+N_t)
    (bf16; esize-scaled) + the I_v workspace.  bf16 units take the streaming
    path (pass 1 reads the unit's keys and elite query rows; pass 2, or pass 2k
    when g * N_tk > 64, writes I_v and the moment records, and the CTA that
    completes a unit reads its records back and writes its layer statistics;
    each selection CTA reads its request's layer statistics for the budget);
    other units the wide kernel.  The first kernel zeroes the call's block of
    counters."""
    row = spec.H_kv * spec.D * esize
    qrow = spec.H_q * spec.D * esize
    g = spec.H_q // spec.H_kv
    units = spec.L * spec.B
    zero = 52 + 4 * (spec.B + 4 * units)  # the call's zeroed block
    k = {"zero_block": zero, "elite_window": 0, "score_pass1": 0, "score_pass2": 0, "score_pass2k": 0,
         "score_wide": 0, "budget_select": 0, "select_topk": 0, "gather_compact": 0}
    path = zero
    for l in range(spec.L):
        for b, (nv, nt) in enumerate(unit_lengths(spec)):
            u = l * spec.B + b
            t, kp = int(n_tk[u]), int(keep[u])
            k["elite_window"] += nt * row + qrow + 4 * t
            if esize == 2:
                k["score_pass1"] += (nv + t) * row + t * qrow
                # I_v written, plus one 48-byte moment record per key block
                # (256 keys in pass 2, 128 in pass 2k), written and read back
                # once by the merge, and the unit's 16-byte layer statistics
                recs = -(-nv // (256 if g * t <= 64 else 128))
                k["score_pass2" if g * t <= 64 else "score_pass2k"] += 4 * nv + 96 * recs + 16
                k["budget_select"] += 16 * spec.L + 4 * nv + 4 * kp
                iv_passes = 2  # written, read by the selection
            else:
                k["score_wide"] += (nv + t) * row + t * qrow + 4 * nv
                recs, iv_passes = 0, 3  # written, read for the moments and by the selection
                k["select_topk"] += 4 * nv + 4 * kp
            k["gather_compact"] += 2 * 2 * (kp + nt) * row + 4 * kp
            path += ((nv + nt) * row + (1 + t) * qrow + 2 * 2 * (kp + nt) * row + 4 * nv * iv_passes
                     + 96 * recs + (16 + 16 * spec.L if recs else 0) + 8 * kp)
    return k, path


def oracle_sample(wl, budget_s, device_for_copy=None, window_mode=0, budget_mode=0):
    """Time the oracle (single thread) on whole requests of the workload until
    budget_s is spent (at least one request).  Returns (tokens, seconds, requests)."""
    from lvlm_kv_cache_gb300 import workloads as W
    from oracle import oracle as O

    spec = wl.spec
    cu_s, cu_v, cu_t = W.offsets(spec)
    tokens, elapsed, done = 0, 0.0, 0
    for b in range(spec.B):
        s0, s1 = cu_s[b], cu_s[b + 1]
        t0, t1 = cu_t[b], cu_t[b + 1]
        nv, nt = spec.n_visual[b], spec.n_text[b]
        q = W.host_bits(wl.q[:, t0:t1])
        k = W.host_bits(wl.k[:, s0:s1])
        v = W.host_bits(wl.v[:, s0:s1])
        t = time.perf_counter()
        res = O.request([q[l] for l in range(spec.L)], [k[l] for l in range(spec.L)], nv, spec.alpha, spec.r,
                        window_mode, budget_mode)
        for l in range(spec.L):
            O.compact(k[l], nv, nt, res["idx"][l])
            O.compact(v[l], nv, nt, res["idx"][l])
        elapsed += time.perf_counter() - t
        tokens += nv * spec.L
        done += 1
        if elapsed >= budget_s:
            break
    return tokens, elapsed, done


# ------------------------------------------------------------------ decode consumer

DECODE_METRIC = "decode attention step time (every layer, one new token per request), full vs compressed cache"


def decode_oracle_sample(q, ranges, budget_s):
    """Time the oracle's decode on sequences (query row index, first row, end
    row, K arena, V arena) until budget_s is spent; returns (rows, seconds,
    sequences)."""
    from oracle import oracle as O

    rows, secs, n = 0, 0.0, 0
    for (qi, r0, r1, kk, vv) in ranges:
        qb = W_host(q[qi])
        kb, vb = W_host(kk[r0:r1]), W_host(vv[r0:r1])
        t = time.perf_counter()
        O.decode(qb, kb, vb)
        secs += time.perf_counter() - t
        rows += r1 - r0
        n += 1
        if secs >= budget_s:
            break
    return rows, secs, n


def W_host(t):
    from lvlm_kv_cache_gb300 import workloads as W

    return W.host_bits(t)


def run_decode(args, local):
    """One decode step = 28 per-layer aircache_decode calls (a CUDA graph of
    them, as a decoder replays it), over (a) the full prefill cache and (b) the
    cache aircache_compress left, for each BATCHxPROMPT and ratio r.  L2 is
    flushed before every timed step (outside the events)."""
    import dataclasses

    import torch

    from lvlm_kv_cache_gb300 import aircache as A
    from lvlm_kv_cache_gb300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peak, peak_kind = load_peaks()
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        flush_buf.zero_()
        torch.sum(flush_buf.view(torch.int64), dim=(0,), out=flush_sink)

    ratios = [float(x) for x in args.decode_ratios.split(",") if x]
    for cfg in [c for c in args.decode_configs.split(",") if c]:
        B, P = (int(x) for x in cfg.lower().split("x"))
        n_t = 128
        base = W.spec("7b")
        spec = dataclasses.replace(base, B=B, L=args.decode_layers, n_visual=[P - n_t] * B, n_text=[n_t] * B)
        wl = W.generate(spec, seed=0, device=dev)
        L, H_q, H_kv, D = spec.L, spec.H_q, spec.H_kv, spec.D
        gen = torch.Generator(device=dev)
        gen.manual_seed(1)
        qdec = torch.randn((L, B, H_q, D), generator=gen, device=dev).to(torch.bfloat16)
        cu64 = wl.cu_seqlens.to(torch.int64)

        def timed(probs, ws):
            for pr in probs:  # eager once: sets the kernel attributes before capture
                A.aircache_decode(pr, ws)
            torch.cuda.synchronize()
            st = A.aircache_get_error(ws)
            if st != 0:
                raise RuntimeError(f"decode device error {st}")
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for pr in probs:
                    A.aircache_decode(pr, ws)
            for _ in range(max(args.warmup, 3)):
                flush_l2()
                g.replay()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for s_, e_ in ev:
                flush_l2()
                s_.record()
                g.replay()
                e_.record()
            torch.cuda.synchronize()
            st = A.aircache_get_error(ws)
            if st != 0:
                raise RuntimeError(f"decode device error {st}")
            return statistics.median(s_.elapsed_time(e_) for s_, e_ in ev)

        # the decode kernels start while the previous layer's finishes (their
        # caches were written long before: AIRCACHE_DECODE_EARLY_CACHE holds)
        full_probs = [A.DecodeProblem(qdec[l], wl.k[l], wl.v[l], offsets=cu64, max_rows=P, early_cache=True)
                      for l in range(L)]
        ws = torch.zeros(max(p.workspace_size() for p in full_probs), dtype=torch.uint8, device=dev)
        sampler = ClockSampler(local)
        sampler.start()
        full_ms = timed(full_probs, ws)
        full_rows = L * B * P
        kv_row_bytes = H_kv * D * 2 * 2
        full_bytes = full_rows * kv_row_bytes + L * B * H_q * D * (2 + 4)
        results = []
        for r in ratios:
            s_r = dataclasses.replace(spec, r=r)
            prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, P - n_t, n_t, s_r.alpha, r,
                             total_tokens=wl.total_tokens, total_visual=wl.total_visual)
            out = A.compress(prob)
            offs = out["out_offsets"]
            rows_h = offs.cpu().numpy()
            longest = int((rows_h[1:] - rows_h[:-1]).max())
            comp_probs = [A.DecodeProblem(qdec[l], out["out_k"], out["out_v"], row_begin=offs[l * B:(l + 1) * B],
                                          row_end=offs[l * B + 1:(l + 1) * B + 1], max_rows=longest,
                                          early_cache=True)
                          for l in range(L)]
            need = max(p.workspace_size() for p in comp_probs)
            ws_c = ws if ws.numel() >= need else torch.zeros(need, dtype=torch.uint8, device=dev)
            comp_ms = timed(comp_probs, ws_c)
            comp_rows = int(rows_h[-1])
            comp_bytes = comp_rows * kv_row_bytes + L * B * H_q * D * (2 + 4)
            # int8 storage of the compressed cache (one aircache_quantize_int8 call, timed on its own)
            kc, vc = out["out_k"][:comp_rows], out["out_v"][:comp_rows]
            k8 = torch.empty(kc.shape, dtype=torch.int8, device=dev)
            v8 = torch.empty(vc.shape, dtype=torch.int8, device=dev)
            ks = torch.empty((L * B, H_kv), dtype=torch.float32, device=dev)
            vs = torch.empty((L * B, H_kv), dtype=torch.float32, device=dev)
            qt = []
            for it in range(max(args.warmup, 3) + 5):
                flush_l2()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                A.aircache_quantize_int8(kc, vc, offs, k8, v8, ks, vs)
                e1.record()
                torch.cuda.synchronize()
                if it >= max(args.warmup, 3):
                    qt.append(e0.elapsed_time(e1))
            q_ms = statistics.median(qt)
            q_bytes = comp_rows * kv_row_bytes * 3 // 2 + 2 * L * B * H_kv * 4  # bf16 read + int8 written
            q8_probs = [A.DecodeProblem(qdec[l], k8, v8, row_begin=offs[l * B:(l + 1) * B],
                                        row_end=offs[l * B + 1:(l + 1) * B + 1], max_rows=longest,
                                        k_scale=ks[l * B:(l + 1) * B], v_scale=vs[l * B:(l + 1) * B],
                                        early_cache=True)
                        for l in range(L)]
            need8 = max(p.workspace_size() for p in q8_probs)  # the int8 launch plan may split differently
            ws_8 = ws_c if ws_c.numel() >= need8 else torch.zeros(need8, dtype=torch.uint8, device=dev)
            q8_ms = timed(q8_probs, ws_8)
            q8_bytes = comp_rows * kv_row_bytes // 2 + L * B * H_q * D * (2 + 4) + 2 * L * B * H_kv * 4
            # gather-fused: the same rows read from the full cache through the row list
            ri = A.row_index(prob, out)
            ga_probs = [A.DecodeProblem(qdec[l], wl.k[l], wl.v[l], row_begin=offs[l * B:(l + 1) * B],
                                        row_end=offs[l * B + 1:(l + 1) * B + 1], max_rows=longest,
                                        early_cache=True, row_index=ri)
                        for l in range(L)]
            ga_ms = timed(ga_probs, ws_c)
            results.append({"r": r, "ms": comp_ms, "rows": comp_rows, "algorithmic_bytes": comp_bytes,
                            "gather_fused": {"ms": ga_ms, "gbs": comp_bytes / (ga_ms * 1e-3) / 1e9,
                                             "reduction": 1.0 - ga_ms / full_ms},
                            "gbs": comp_bytes / (comp_ms * 1e-3) / 1e9,
                            "frac": comp_bytes / (comp_ms * 1e-3) / 1e9 / peak,
                            "splits": comp_probs[0].splits(), "reduction": 1.0 - comp_ms / full_ms,
                            "int8": {"ms": q8_ms, "algorithmic_bytes": q8_bytes,
                                     "gbs": q8_bytes / (q8_ms * 1e-3) / 1e9, "reduction": 1.0 - q8_ms / full_ms,
                                     "quantize_ms": q_ms, "quantize_gbs": q_bytes / (q_ms * 1e-3) / 1e9}})
            del out, prob, k8, v8
        clocks = sampler.stop()
        full_gbs = full_bytes / (full_ms * 1e-3) / 1e9
        line = {
            "metric": DECODE_METRIC, "value": results[0]["ms"] if results else full_ms, "unit": "ms",
            "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"7B LVLM-shaped decode: batch {B}, prompt {P} ({P - n_t} visual + {n_t} text), "
                                   f"L={L}, H_q=28, H_kv=4, D=128, bf16; caches from aircache_compress",
                       "batch": B, "prompt": P,
                       "step": f"{L} aircache_decode calls (one per layer, num_seqs = batch, "
                               "AIRCACHE_DECODE_EARLY_CACHE) replayed as a CUDA graph",
                       "l2": "flushed before every timed step outside the events"},
            "full": {"ms": full_ms, "rows": full_rows, "algorithmic_bytes": full_bytes, "gbs": full_gbs,
                     "frac": full_gbs / peak, "splits": full_probs[0].splits()},
            "compressed": results,
            "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": full_gbs, "peak": peak,
                         "unit": "GB/s", "frac": full_gbs / peak, "peak_kind": peak_kind,
                         "traffic": recorded_traffic(f"decode_{B}x{P}", "decode_kernel"),
                         "note": "full-cache step: one decode_kernel launch per layer, bytes and time per launch"},
            "gpu_launches": L,
            "clocks": clocks,
        }
        if not args.no_cpu_baseline:
            ranges = [(b, int(cu64[b]), int(cu64[b + 1]), wl.k[0], wl.v[0]) for b in range(B)]
            rows, secs, n = decode_oracle_sample(qdec[0], ranges, args.cpu_sample_s / 2)
            ms_step = secs / rows * full_rows * 1e3
            line["cpu_baseline"] = {"value": ms_step, "unit": "ms per full-cache step (extrapolated)", "cores": 1,
                                    "host_cores": os.cpu_count(),
                                    "kind": "oracle",
                                    "sample": f"{n} (layer 0, request) sequence(s) of {P} rows in {secs:.2f} s, "
                                              f"single thread, scaled by rows to the {L}x{B} sequences of a step"}
        print(json.dumps(line), flush=True)
        del wl, full_probs, ws
        torch.cuda.empty_cache()


TIMELINE_UNITS = ("elite", "stream", "select", "compact")
TIMELINE_KERNELS = {0: "elite_window", 1: "score_pass1", 2: "score_pass2", 3: "score_pass2k",
                    5: "budget_select", 6: "gather_compact"}


def run_timeline(args, local):
    """Device timeline of aircache_compress on the measurement build of the
    library (libaircache_timeline.so, compiled with -DAIRCACHE_TIMELINE: every
    CTA of each compression kernel records its first thread's entry time and
    its warps' latest exit time with globaltimer).  L2 flushed before every
    call (outside it).  Per kernel: CTAs, first and last CTA entry, median and
    last CTA exit, in microseconds from the call's first entry, each the median
    over --steps calls.  The exit stamps add an atomic per warp, so spans read a
    few percent longer than the product build's."""
    os.environ["AIRCACHE_TIMELINE"] = "1"  # before the binding loads its library
    import ctypes

    import numpy as np
    import torch

    from lvlm_kv_cache_gb300 import build

    build.build(timeline=True)
    from lvlm_kv_cache_gb300 import aircache as A
    from lvlm_kv_cache_gb300 import workloads as W

    if not A.LIB_PATH.endswith("libaircache_timeline.so"):
        raise RuntimeError("the binding was loaded before --timeline selected the measurement build")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = A.lib()
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)
    wl = W.make(args.config, device=dev)
    spec = wl.spec
    prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(spec.n_visual), max(spec.n_text),
                     spec.alpha, spec.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual)
    ws = prob.new_workspace()
    out = A.alloc_outputs(prob)
    for _ in range(max(3, args.warmup)):
        A.compress(prob, ws=ws, out=out)
    torch.cuda.synchronize()
    shape = (8, 4096, 2)
    rows = {k: [] for k in TIMELINE_KERNELS}
    spans = []
    for _ in range(args.steps):
        for u in TIMELINE_UNITS:
            if getattr(lib, "aircache_timeline_clear_" + u)() != 0:
                raise RuntimeError("timeline table clear failed")
        flush_buf.zero_()
        torch.sum(flush_buf.view(torch.int64), dim=(0,), out=flush_sink)
        torch.cuda.synchronize()
        A.compress(prob, ws=ws, out=out)
        torch.cuda.synchronize()
        tab = np.zeros(shape, np.uint64)
        for u in TIMELINE_UNITS:
            buf = np.zeros(shape, np.uint64)
            if getattr(lib, "aircache_timeline_read_" + u)(buf.ctypes.data_as(ctypes.c_void_p)) != 0:
                raise RuntimeError("timeline table read failed")
            tab = np.maximum(tab, buf)
        starts = tab[:, :, 0].astype(np.int64)
        t0 = starts[starts > 0].min()
        last = 0.0
        for k in TIMELINE_KERNELS:
            ok = starts[k] > 0
            if not ok.any():
                continue
            st = (starts[k][ok] - t0) / 1000.0
            en = (tab[k, :, 1].astype(np.int64)[ok] - t0) / 1000.0
            rows[k].append((int(ok.sum()), st.min(), st.max(), float(np.median(en)), en.max()))
            last = max(last, en.max())
        spans.append(last)
    kernels = []
    for k, name in TIMELINE_KERNELS.items():
        if not rows[k]:
            continue
        r = np.array(rows[k])
        kernels.append({"name": name, "ctas": int(r[0, 0]), "start_first_us": round(float(np.median(r[:, 1])), 2),
                        "start_last_us": round(float(np.median(r[:, 2])), 2),
                        "end_median_us": round(float(np.median(r[:, 3])), 2),
                        "end_last_us": round(float(np.median(r[:, 4])), 2)})
    print(json.dumps({"metric": "device timeline of one aircache_compress call (measurement build)",
                      "unit": "us", "value": round(float(np.median(spans)), 2), "higher_is_better": False,
                      "steps": args.steps, "data": "synthetic",
                      "config": {"workload": DESCRIPTIONS.get(args.config, args.config), "name": args.config,
                                 "l2": "flushed before every call outside it"},
                      "kernels": kernels}), flush=True)


def run_prefill(args, local):
    """The scoring fused into prefill: (a) aircache_prefill (causal attention of
    every layer), (b) aircache_prefill_compress (the same attention, and the
    whole compression from its logits), (c) aircache_prefill then
    aircache_compress (the scoring streams the keys again).  L2 is flushed before
    every timed call (outside the events); medians of the timed calls."""
    import torch

    from lvlm_kv_cache_gb300 import aircache as A
    from lvlm_kv_cache_gb300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        flush_buf.zero_()
        torch.sum(flush_buf.view(torch.int64), dim=(0,), out=flush_sink)

    wl = W.make(args.config, device=dev, layers=args.layers or None)
    spec = wl.spec
    qv = W.visual_queries(wl, 1)
    cu_s, cu_v, cu_t = W.offsets(spec)
    q = torch.empty((spec.L, wl.total_tokens, spec.H_q, spec.D), dtype=spec.dtype, device=dev)
    for b in range(spec.B):
        nv = cu_v[b + 1] - cu_v[b]
        q[:, cu_s[b]:cu_s[b] + nv] = qv[:, cu_v[b]:cu_v[b + 1]]
        q[:, cu_s[b] + nv:cu_s[b + 1]] = wl.q[:, cu_t[b]:cu_t[b + 1]]
    del qv
    prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(spec.n_visual), max(spec.n_text),
                     spec.alpha, spec.r)
    attn = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    ws = prob.new_workspace()
    out = A.alloc_outputs(prob)

    def plain():
        A.aircache_prefill(prob, q, attn, ws)

    def fused():
        A.aircache_prefill_compress(prob, q, attn, ws, out["out_k"], out["out_v"], out["out_offsets"],
                                    out["keep"], out["idx"], out["iv"])

    def separate():
        plain()
        A.aircache_compress(prob, ws, out["out_k"], out["out_v"], out["out_offsets"], out["keep"], out["idx"],
                            out["iv"])

    def compress_only():
        A.aircache_compress(prob, ws, out["out_k"], out["out_v"], out["out_offsets"], out["keep"], out["idx"],
                            out["iv"])

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for it in range(max(args.warmup, 3) + args.steps):
            flush_l2()
            torch.cuda.synchronize()
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if it >= max(args.warmup, 3):
                ts.append(e0.elapsed_time(e1))
        assert A.aircache_get_error(ws) == 0
        return statistics.median(ts)

    sampler = ClockSampler(local)
    sampler.start()
    t_plain = timed(plain)
    t_fused = timed(fused)
    t_sep = timed(separate)
    t_comp = timed(compress_only)
    clocks = sampler.stop()
    flops = sum((n := cu_s[b + 1] - cu_s[b]) * (n + 1) // 2 for b in range(spec.B)) * spec.H_q * spec.L * spec.D * 4
    tflops = flops / (t_plain * 1e-3) / 1e12
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak, peak_kind = 1900.0, "fallback"
    if os.path.exists(peaks_path):
        with open(peaks_path) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured (burst)"
    line = {
        "metric": "prefill with the AirCache scoring fused in: time over the plain prefill", "unit": "ms",
        "value": t_fused, "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
        "warmup": max(args.warmup, 3), "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS.get(args.config, args.config) + "; queries of every prompt row "
                               "(seeded visual-token queries, then the text queries)",
                   "name": args.config, "layers": spec.L,
                   "l2": "flushed before every timed call outside the events"},
        "prefill_ms": t_plain, "prefill_compress_ms": t_fused, "prefill_then_compress_ms": t_sep,
        "compress_ms": t_comp,
        "fused_overhead": (t_fused - t_plain) / t_plain, "separate_overhead": (t_sep - t_plain) / t_plain,
        "causal_flops": flops,
        "roofline": {"bound": "tensor", "kernel": "prefill_kernel", "achieved": tflops, "peak": peak,
                     "unit": "TFLOP/s", "frac": tflops / peak, "peak_kind": peak_kind, "traffic": None},
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores: each step is a bounded
    sample (whole requests) of the same workload."""
    if rank != 0:
        return
    from lvlm_kv_cache_gb300 import workloads as W

    spec = W.spec(args.config)
    wl = W.generate(spec, seed=0, device="cpu")
    for _ in range(args.warmup):
        oracle_sample(wl, 0.0, window_mode=args.window_mode, budget_mode=args.budget_mode)
    tok, secs = 0, 0.0
    for _ in range(args.steps):
        t, s, _ = oracle_sample(wl, 0.0, window_mode=args.window_mode, budget_mode=args.budget_mode)
        tok += t
        secs += s
    value = tok / secs
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS.get(args.config, args.config), "name": args.config,
                   "sample": "one request (all layers) per step",
                   "inputs": "the same recipe and shapes drawn by the CPU generator (same seed, other values "
                             "than the GPU arm's device generator draws)",
                   "variant": {"window_mode": args.window_mode, "budget_mode": args.budget_mode}},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
                         "sample": "request 0 of the workload, all layers, per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.timeline:
        return run_timeline(args, local)
    if args.prefill:
        return run_prefill(args, local)
    if args.decode:
        return run_decode(args, local)

    import torch

    from lvlm_kv_cache_gb300 import aircache as A
    from lvlm_kv_cache_gb300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    wl = W.make(args.config, seed=rank, device=dev)
    spec = wl.spec
    esize = 2 if spec.dtype == torch.bfloat16 else 4
    prob = A.Problem(wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(spec.n_visual), max(spec.n_text),
                     spec.alpha, spec.r, total_tokens=wl.total_tokens, total_visual=wl.total_visual,
                     window_mode=args.window_mode, budget_mode=args.budget_mode, head_sets=args.head_sets,
                     q_visual=W.visual_queries(wl, seed=rank + 1) if args.window_mode == 4 else None)
    ws = prob.new_workspace()
    out = A.alloc_outputs(prob)
    L, B, TV = prob.L, prob.B, prob.total_visual
    # elite sizes (for the byte accounting) from the staged scorer, outside timing
    iv_s = torch.empty((L, TV), dtype=torch.float32, device=dev)
    el_s = torch.empty((L * B, prob.max_text), dtype=torch.int32, device=dev)
    ntk_s = torch.empty(L * B, dtype=torch.int32, device=dev)
    # (the staged scorer takes one index set per layer; the elite sizes do not depend on it)
    prob_s = prob if not (args.head_sets or args.window_mode == 4) else A.Problem(
        wl.q, wl.k, wl.v, wl.cu_seqlens, wl.cu_visual, max(spec.n_visual), max(spec.n_text), spec.alpha, spec.r,
        total_tokens=wl.total_tokens, total_visual=wl.total_visual,
        window_mode=args.window_mode if args.window_mode != 4 else 0, budget_mode=args.budget_mode)
    ws_s = ws if prob_s is prob else prob_s.new_workspace()
    A.aircache_score(prob_s, ws_s, iv_s, el_s, ntk_s)
    assert A.aircache_get_error(ws_s) == 0

    def step():
        A.aircache_compress(prob, ws, out["out_k"], out["out_v"], out["out_offsets"], out["keep"],
                            out["idx"], out["iv"])

    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read it back: the write evicts the
        # step's data, the read evicts the write's dirty lines, so no write-back
        # of the flush itself lands inside the next timed step
        flush_buf.zero_()
        torch.sum(flush_buf.view(torch.int64), dim=(0,), out=flush_sink)

    for _ in range(max(args.warmup, 3)):
        step()
    st = A.aircache_get_error(ws)
    if st != 0:
        raise RuntimeError(f"device error {st}: {A.status_string(st)}")
    n_tk = ntk_s.cpu().numpy()
    if args.window_mode == 4:  # 32 window rows per unit (their keys are visual keys: a slight overcount)
        import numpy as np

        n_tk = np.minimum(32, np.tile(np.asarray(spec.n_visual), spec.L))
    keep = out["keep"].cpu().numpy()
    kbytes, path_bytes = algorithmic_bytes(spec, n_tk, keep, esize)

    vis_idx = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    try:
        gpu_index = int(vis_idx[local]) if vis_idx != [""] else local
    except ValueError:
        gpu_index = None
    sampler = ClockSampler(gpu_index)
    sampler.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:
        for _ in range(20):
            flush_l2()
            step()
        torch.cuda.synchronize()

    # ---- timed region: K steps, L2 flushed before each (outside the events)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2()
        starts[i].record()
        step()
        ends[i].record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    st = A.aircache_get_error(ws)
    if st != 0:
        raise RuntimeError(f"device error {st}: {A.status_string(st)}")

    units = spec.L * sum(spec.n_visual)  # visual KV rows (token x layer) per step per rank
    ms_per_step = total_ms / args.steps
    value = whole_job_rate(world, units, args.steps, total_ms)

    # ---- per-kernel durations on the launching stream
    nk = prob.launches()
    names = A.kernel_names(prob)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    for row in ev:  # torch creates the CUDA event on first record
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2()
        A.aircache_compress_profile(prob, ws, out["out_k"], out["out_v"], out["out_offsets"], out["keep"],
                                    ev[i], out["idx"], out["iv"])
    torch.cuda.synchronize()
    per_kernel = {n: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
                  for j, n in enumerate(names)}
    peak, peak_kind = load_peaks()
    kernels = []
    for n in names:
        ms = per_kernel[n]
        gbs = kbytes[n] / (ms * 1e-3) / 1e9 if ms > 0 else None
        kernels.append({"name": n, "ms": ms, "algorithmic_bytes": kbytes[n], "gbs": gbs,
                        "frac": gbs / peak if gbs else None})
    dom = max(kernels, key=lambda k: k["ms"])
    roof = {"bound": "hbm", "kernel": dom["name"], "achieved": dom["gbs"], "peak": peak, "unit": "GB/s",
            "frac": dom["frac"], "peak_kind": peak_kind,
            "traffic": recorded_traffic(args.config, dom["name"])}
    path_gbs = path_bytes / (ms_per_step * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if esize == 2 else "f32",
        "data": "synthetic",
        "config": {"workload": DESCRIPTIONS.get(args.config, args.config), "name": args.config,
                   "requests_per_rank": spec.B, "layers": spec.L, "seed": "rank",
                   "variant": {"window_mode": args.window_mode, "budget_mode": args.budget_mode,
                               "head_sets": bool(args.head_sets)},
                   "l2": "flushed before every timed step outside the events: 256 MB written, then read back "
                         "(so the flush's own dirty lines are not written back inside the step)"},
        "requests_per_s": world * spec.B * args.steps / (total_ms / 1e3),
        "visual_tokens_per_s": world * sum(spec.n_visual) * args.steps / (total_ms / 1e3),
        "fused_compress": {"algorithmic_bytes": path_bytes, "gbs": path_gbs,
                           "frac_of_8tbs": path_gbs / 8000.0, "frac_of_measured": path_gbs / peak},
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": nk * args.steps,
        "clocks": clocks,
    }

    # ---- end to end through the public API, host buffers, copies timed
    if not args.no_e2e:
        hq = wl.q.cpu().pin_memory()
        hk = wl.k.cpu().pin_memory()
        hv = wl.v.cpu().pin_memory()
        hcs = wl.cu_seqlens.cpu().pin_memory()
        hcv = wl.cu_visual.cpu().pin_memory()
        ok_h = torch.empty(out["out_k"].shape, dtype=out["out_k"].dtype).pin_memory()
        ov_h = torch.empty_like(ok_h).pin_memory()
        of_h = torch.empty(out["out_offsets"].shape, dtype=torch.int64).pin_memory()
        # the values stay in pinned host memory: only the compaction reads them,
        # the kept visual rows and the text rows, in place over the host link.
        # Two buffer sets, double-buffered across steps: step i+1's inputs
        # cross the link while step i computes and its compacted rows come
        # back (three streams; every step's copies and compute are inside the
        # timed region, which ends when the last step's rows are on the host)
        sets = []
        for j in range(2):
            dq = wl.q if j == 0 else torch.empty_like(wl.q)
            dk = wl.k if j == 0 else torch.empty_like(wl.k)
            dcs = wl.cu_seqlens if j == 0 else torch.empty_like(wl.cu_seqlens)
            dcv = wl.cu_visual if j == 0 else torch.empty_like(wl.cu_visual)
            pj = A.Problem(dq, dk, hv, dcs, dcv, max(spec.n_visual), max(spec.n_text), spec.alpha, spec.r,
                           total_tokens=wl.total_tokens, total_visual=wl.total_visual,
                           window_mode=args.window_mode, budget_mode=args.budget_mode, head_sets=args.head_sets,
                           q_visual=prob.q_visual if args.window_mode == 4 else None)
            oj = out if j == 0 else A.alloc_outputs(pj)
            hj = (ok_h, ov_h, of_h) if j == 0 else (torch.empty_like(ok_h).pin_memory(),
                                                   torch.empty_like(ov_h).pin_memory(),
                                                   torch.empty_like(of_h).pin_memory())
            sets.append({"q": dq, "k": dk, "cs": dcs, "cv": dcv, "prob": pj, "out": oj, "host": hj,
                         "in_done": torch.cuda.Event(), "comp_done": torch.cuda.Event(),
                         "out_done": torch.cuda.Event()})
        s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        v_read = int(out["out_offsets"][-1]) * spec.H_kv * spec.D * esize  # value rows the compaction reads
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hcs, hcv)) + v_read
        d2h = sum(t.numel() * t.element_size() for t in (ok_h, ov_h, of_h))
        for st in sets:  # every event starts recorded, so the first waits are no-ops
            for e in ("in_done", "comp_done", "out_done"):
                st[e].record()

        def e2e_step(i):
            st = sets[i % 2]
            with torch.cuda.stream(s_in):
                s_in.wait_event(st["comp_done"])  # the step before on this set has read its inputs
                st["q"].copy_(hq, non_blocking=True)
                st["k"].copy_(hk, non_blocking=True)
                st["cs"].copy_(hcs, non_blocking=True)
                st["cv"].copy_(hcv, non_blocking=True)
                st["in_done"].record()
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(st["in_done"])
                s_comp.wait_event(st["out_done"])  # the step before on this set has its rows back
                o = st["out"]
                A.aircache_compress(st["prob"], ws, o["out_k"], o["out_v"], o["out_offsets"], o["keep"],
                                    o["idx"], o["iv"])
                st["comp_done"].record()
            with torch.cuda.stream(s_out):
                s_out.wait_event(st["comp_done"])
                for hb, db in zip(st["host"], (st["out"]["out_k"], st["out"]["out_v"], st["out"]["out_offsets"])):
                    hb.copy_(db, non_blocking=True)
                st["out_done"].record()

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 20))
        s_ev = torch.cuda.Event(enable_timing=True)
        e_ev = torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        s_ev.record(s_in)
        for i in range(n_e2e):
            e2e_step(i)
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_comp)
        e_ev.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s_ev.elapsed_time(e_ev), dist, dev)
        # every set's rows equal, bit for bit, those of the call with every value in device memory
        step()
        torch.cuda.synchronize()
        rows_e = int(out["out_offsets"][-1])
        for st in sets:
            hk_, hv_, ho_ = st["host"]
            if not (int(ho_[-1]) == rows_e and torch.equal(hk_[:rows_e], out["out_k"][:rows_e].cpu())
                    and torch.equal(hv_[:rows_e], out["out_v"][:rows_e].cpu())):
                raise RuntimeError("the end-to-end steps (values read in place from host memory) gave other "
                                   "rows than the device-resident call")
        line["e2e"] = {"value": whole_job_rate(world, units, n_e2e, e2e_ms), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
                       "ms_per_step": e2e_ms / n_e2e,
                       "inputs": "q, k and the offsets copied from pinned host memory; the values stay "
                                 "there and the compaction reads the rows it keeps in place "
                                 "(counted in h2d_bytes_per_step); two buffer sets, so one step's "
                                 "inputs cross the link while the step before computes and copies back"}

    # ---- CPU baseline: the oracle on the host cores, rank 0 at N=1 only
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok, secs, nreq = oracle_sample(wl, args.cpu_sample_s, window_mode=args.window_mode,
                                        budget_mode=args.budget_mode)
        line["cpu_baseline"] = {"value": tok / secs, "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{nreq} whole request(s) x {spec.L} layers "
                                          f"({tok} visual KV rows) in {secs:.2f} s, single thread"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
