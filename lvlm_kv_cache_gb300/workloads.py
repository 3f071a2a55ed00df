"""Seeded synthetic inputs shaped like post-prefill LVLM KV caches.

This module only draws random tensors and lays them out; it holds none of the
compression method's arithmetic, so both the CUDA path and the CPU oracle can be
fed from it.  Layout (the prompt layout X = Concat(X_v, X_t) of the AirCache
notes, "Key design 1"): per request, the visual tokens come first, then the text
tokens; requests are packed one after another (FlashAttention-style varlen).

    k, v : [L, total_tokens, H_kv, D]   post-RoPE keys / values, every layer
    q    : [L, total_text,   H_q,  D]   post-RoPE queries of the text tokens
    cu_seqlens[b] : first token of request b in k/v        (int32, [B+1])
    cu_visual[b]  : first I_v slot of request b            (int32, [B+1])
    the text rows of request b in q start at cu_seqlens[b] - cu_visual[b].

Configurations (seed 0 unless stated):

tiny        B=1, L=2, H_q=H_kv=4, D=64, N_v=64, N_t=16, fp32, entries N(0,1)/sqrt(D);
            6 visual keys per layer shifted by +2.0 along the unit mean direction
            of their KV group's text queries; alpha=0.9, r=0.25.
7b          B=1, L=28, H_q=28, H_kv=4, D=128, N_v=7290, N_t=128, bf16 N(0,1);
            10% of visual keys per layer shifted by 1.5 * s_l * sigma_K * sqrt(D)
            along that direction, s_l ~ U(0.5, 2) per layer; alpha=0.9, r=0.10.
llama_mha   B=8, L=32, H_q=H_kv=32, D=128, N_v=2880, N_t=512, bf16 N(0,1), every
            token's key row scaled by exp(N(0, 0.5^2)); 5% heavy visual keys with
            the 7b rule; alpha=0.9, r=0.10.
video_r01 / video_r10
            B=4, L=28, H_q=28, H_kv=4, D=128, N_v=12544 (64 frames x 196
            patches), N_t=256, bf16; visual keys follow k_i = 0.8 k_{i-1} + 0.6 e_i
            along the raster order of each frame (restarted per frame), no heavy
            keys; alpha=0.9, r=0.01 / 0.10.
ragged      B=32, L=28, H_q=28, H_kv=4, D=128, N_v ~ U[576, 9000], N_t ~ U[32, 1024]
            (seeded integers), bf16 N(0,1), 10% heavy keys (7b rule); alpha=0.9,
            r=0.05.

Decode steps (decode_inputs): S sequences of given lengths packed into one
arena [rows, H_kv, D] (sequence s owns rows offsets[s]..offsets[s+1]-1), one
query row [H_q, D] per sequence, bf16 N(0,1) entries (queries times q_scale),
optional extra arena rows after the last sequence filled with NaN, and an
optional new (k, v) row per sequence.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass
class Spec:
    name: str
    B: int
    L: int
    H_q: int
    H_kv: int
    D: int
    n_visual: list
    n_text: list
    dtype: torch.dtype
    alpha: float
    r: float
    entry_std: float = 1.0          # std of Q/K/V entries
    heavy_count: int = 0            # fixed number of heavy visual keys per layer
    heavy_frac: float = 0.0         # or a fraction of N_v
    heavy_bias: float = 0.0         # shift = bias * s_l * entry_std * sqrt(D)
    layer_scale: tuple = (1.0, 1.0)  # s_l ~ U(lo, hi)
    key_norm_sigma: float = 0.0     # per-token key scale exp(N(0, sigma^2))
    frames: int = 0                 # AR(1) visual keys: frames x patches
    ar_rho: float = 0.0


def _spec(name: str) -> Spec:
    rng = np.random.default_rng(0)  # only for the ragged lengths (platform independent)
    if name == "tiny":
        return Spec("tiny", 1, 2, 4, 4, 64, [64], [16], torch.float32, 0.9, 0.25,
                    entry_std=1.0 / math.sqrt(64), heavy_count=6, heavy_bias=2.0)
    if name == "7b":
        return Spec("7b", 1, 28, 28, 4, 128, [7290], [128], torch.bfloat16, 0.9, 0.10,
                    heavy_frac=0.10, heavy_bias=1.5, layer_scale=(0.5, 2.0))
    if name == "llama_mha":
        return Spec("llama_mha", 8, 32, 32, 32, 128, [2880] * 8, [512] * 8, torch.bfloat16,
                    0.9, 0.10, heavy_frac=0.05, heavy_bias=1.5, layer_scale=(0.5, 2.0),
                    key_norm_sigma=0.5)
    if name in ("video_r01", "video_r10"):
        r = 0.01 if name == "video_r01" else 0.10
        return Spec(name, 4, 28, 28, 4, 128, [12544] * 4, [256] * 4, torch.bfloat16, 0.9, r,
                    frames=64, ar_rho=0.8)
    if name == "ragged":
        nv = rng.integers(576, 9001, size=32).tolist()
        nt = rng.integers(32, 1025, size=32).tolist()
        return Spec("ragged", 32, 28, 28, 4, 128, nv, nt, torch.bfloat16, 0.9, 0.05,
                    heavy_frac=0.10, heavy_bias=1.5, layer_scale=(0.5, 2.0))
    raise KeyError(f"unknown workload {name!r}")


CONFIG_NAMES = ("tiny", "7b", "llama_mha", "video_r01", "video_r10", "ragged")


def spec(name: str, layers: int | None = None, requests: int | None = None) -> Spec:
    """The named configuration, optionally cut to its first `layers` layers and
    first `requests` requests (smaller parity cases of the same shape)."""
    s = _spec(name)
    if layers is not None:
        s.L = int(layers)
    if requests is not None:
        s.B = int(requests)
        s.n_visual = s.n_visual[: s.B]
        s.n_text = s.n_text[: s.B]
    return s


@dataclasses.dataclass
class Workload:
    spec: Spec
    q: torch.Tensor          # [L, total_text, H_q, D]
    k: torch.Tensor          # [L, total_tokens, H_kv, D]
    v: torch.Tensor          # [L, total_tokens, H_kv, D]
    cu_seqlens: torch.Tensor  # int32 [B+1]
    cu_visual: torch.Tensor   # int32 [B+1]

    @property
    def total_tokens(self) -> int:
        return int(self.k.shape[1])

    @property
    def total_text(self) -> int:
        return int(self.q.shape[1])

    @property
    def total_visual(self) -> int:
        return int(sum(self.spec.n_visual))


def offsets(spec: Spec):
    """Host lists (cu_seqlens, cu_visual, text_offsets)."""
    cu_s, cu_v, cu_t = [0], [0], [0]
    for nv, nt in zip(spec.n_visual, spec.n_text):
        cu_s.append(cu_s[-1] + nv + nt)
        cu_v.append(cu_v[-1] + nv)
        cu_t.append(cu_t[-1] + nt)
    return cu_s, cu_v, cu_t


def generate(s: Spec, seed: int = 0, device="cpu") -> Workload:
    """Draw the workload on `device` (deterministic for a given seed and device)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    side = np.random.default_rng(seed + 1)  # heavy indices and layer scales
    cu_s, cu_v, cu_t = offsets(s)
    T, TT = cu_s[-1], cu_t[-1]
    g = s.H_q // s.H_kv
    q = torch.empty((s.L, TT, s.H_q, s.D), dtype=s.dtype, device=dev)
    k = torch.empty((s.L, T, s.H_kv, s.D), dtype=s.dtype, device=dev)
    v = torch.empty((s.L, T, s.H_kv, s.D), dtype=s.dtype, device=dev)
    for l in range(s.L):
        ql = torch.randn((TT, s.H_q, s.D), generator=gen, device=dev) * s.entry_std
        kl = torch.randn((T, s.H_kv, s.D), generator=gen, device=dev) * s.entry_std
        vl = torch.randn((T, s.H_kv, s.D), generator=gen, device=dev) * s.entry_std
        if s.key_norm_sigma > 0:
            f = torch.exp(torch.randn((T, 1, 1), generator=gen, device=dev) * s.key_norm_sigma)
            kl = kl * f
        s_l = float(side.uniform(*s.layer_scale)) if s.layer_scale[0] != s.layer_scale[1] \
            else s.layer_scale[0]
        for b in range(s.B):
            nv = s.n_visual[b]
            t0 = cu_s[b]
            if s.frames:
                patches = nv // s.frames
                vis = kl[t0:t0 + nv].reshape(s.frames, patches, s.H_kv, s.D)
                eps = vis.clone()
                for i in range(1, patches):
                    vis[:, i] = s.ar_rho * vis[:, i - 1] + math.sqrt(1 - s.ar_rho ** 2) * eps[:, i]
                kl[t0:t0 + nv] = vis.reshape(nv, s.H_kv, s.D)
            n_heavy = s.heavy_count or int(round(s.heavy_frac * nv))
            if n_heavy:
                tq = ql[cu_t[b]:cu_t[b + 1]]                      # [N_t, H_q, D]
                dirs = tq.reshape(-1, s.H_kv, g, s.D).mean(dim=(0, 2))  # [H_kv, D]
                dirs = dirs / dirs.norm(dim=-1, keepdim=True).clamp_min(1e-12)
                heavy = torch.as_tensor(np.sort(side.choice(nv, n_heavy, replace=False)),
                                        device=dev, dtype=torch.long)
                shift = s.heavy_bias * s_l * s.entry_std * math.sqrt(s.D)
                kl[t0 + heavy] += shift * dirs
        q[l] = ql.to(s.dtype)
        k[l] = kl.to(s.dtype)
        v[l] = vl.to(s.dtype)
    return Workload(
        s, q, k, v,
        torch.tensor(cu_s, dtype=torch.int32, device=dev),
        torch.tensor(cu_v, dtype=torch.int32, device=dev),
    )


def make(name: str, seed: int = 0, device="cpu", layers=None, requests=None) -> Workload:
    return generate(spec(name, layers, requests), seed, device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """A host numpy view of a tensor as the oracle reads it: float32 as is,
    bf16 as raw uint16 bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(f"unsupported dtype {t.dtype}")


def visual_queries(wl: Workload, seed: int = 0) -> torch.Tensor:
    """Seeded post-RoPE queries of the visual tokens, [L, total_visual, H_q, D]
    (the entries' distribution of the text queries), for the visual window."""
    s = wl.spec
    gen = torch.Generator(device=wl.q.device)
    gen.manual_seed(seed)
    q = torch.randn((s.L, wl.total_visual, s.H_q, s.D), generator=gen, device=wl.q.device) * s.entry_std
    return q.to(s.dtype)


def with_prefix(wl: Workload, n_prefix) -> tuple:
    """The same tokens with the first n_prefix[b] text tokens of request b moved
    before its visual span (prompt order [prefix text][visual][other text]).
    Returns (k, v, n_prefix int32 tensor on the workload's device); q (text rows
    in text order), cu_seqlens and cu_visual are unchanged."""
    s = wl.spec
    cu_s, cu_v, _ = offsets(s)
    perm = np.arange(cu_s[-1])
    for b in range(s.B):
        s0, nv, nt, npf = cu_s[b], s.n_visual[b], s.n_text[b], int(n_prefix[b])
        if not 0 <= npf <= nt:
            raise ValueError("0 <= n_prefix <= N_t")
        # new row r of the request takes old (visual-first) row perm[r]
        old = np.concatenate([np.arange(nv, nv + npf), np.arange(nv), np.arange(nv + npf, nv + nt)])
        perm[s0:s0 + nv + nt] = s0 + old
    idx = torch.as_tensor(perm, device=wl.k.device)
    k = wl.k[:, idx].contiguous()
    v = wl.v[:, idx].contiguous()
    return k, v, torch.tensor([int(x) for x in n_prefix], dtype=torch.int32, device=wl.k.device)


@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor        # [S, H_q, D]
    k: torch.Tensor        # [rows, H_kv, D]
    v: torch.Tensor
    offsets: torch.Tensor  # int64 [S+1]
    k_new: torch.Tensor | None = None  # [S, H_kv, D]
    v_new: torch.Tensor | None = None


def decode_inputs(lengths, h_q, h_kv, d, seed=0, device="cpu", q_scale=1.0, nan_tail=0, new_row=False,
                  dtype=torch.bfloat16) -> DecodeInputs:
    """Seeded inputs of one decode step over ragged cached rows (see the module docstring)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    S = len(lengths)
    offs = np.zeros(S + 1, np.int64)
    offs[1:] = np.cumsum(np.asarray(lengths, np.int64))
    rows = int(offs[-1]) + int(nan_tail)
    q = (torch.randn((S, h_q, d), generator=gen, device=dev) * q_scale).to(dtype)
    k = torch.randn((max(rows, 1), h_kv, d), generator=gen, device=dev).to(dtype)
    v = torch.randn((max(rows, 1), h_kv, d), generator=gen, device=dev).to(dtype)
    if nan_tail:
        k[int(offs[-1]):] = float("nan")
        v[int(offs[-1]):] = float("nan")
    kn = vn = None
    if new_row:
        kn = torch.randn((S, h_kv, d), generator=gen, device=dev).to(dtype)
        vn = torch.randn((S, h_kv, d), generator=gen, device=dev).to(dtype)
    return DecodeInputs(q, k, v, torch.as_tensor(offs, device=dev), kn, vn)
