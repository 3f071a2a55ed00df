"""Thin ctypes binding of the AirCache C ABI (include/aircache.h).

Argument marshalling only: every step of the compression runs in the CUDA
library ``libaircache.so`` built from ``csrc/``.  If that library is missing the
binding raises; there is no fallback path.

Tensors are torch CUDA tensors; the functions take the same arguments as the C
entry points (device buffers are tensors, the stream is a torch stream or None
for the current one) and raise ``AirCacheError`` on a non-zero status.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# AIRCACHE_TIMELINE=1 selects the measurement build whose kernels record their
# entry and exit times (build.build(timeline=True)); the default is the product build
LIB_PATH = os.path.join(HERE, "libaircache_timeline.so" if os.environ.get("AIRCACHE_TIMELINE") == "1"
                        else "libaircache.so")

OK = 0
DECODE_EARLY_CACHE = 1
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
ERR_DEVICE_TIMEOUT = -5
ERR_DEVICE_BOUNDS = -6
ERR_ELITE_OVERFLOW = -7
ERR_CAPACITY = -8

F32, BF16, INT8 = 0, 1, 2
MAX_LAYERS = 256
# test hook of the variant word: the first kernel's bounded wait runs out (see aircache.h)
VARIANT_WAIT_TEST = 1 << 24


class AirCacheError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({status_string(status)})")


class ProblemStruct(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32),
        ("num_requests", ctypes.c_int32),
        ("h_q", ctypes.c_int32),
        ("h_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("max_visual", ctypes.c_int32),
        ("max_text", ctypes.c_int32),
        ("max_elite", ctypes.c_int32),
        ("variant", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64),
        ("total_visual", ctypes.c_int64),
        ("cu_seqlens", ctypes.c_void_p),
        ("cu_visual", ctypes.c_void_p),
        ("q_text", ctypes.POINTER(ctypes.c_void_p)),
        ("k", ctypes.POINTER(ctypes.c_void_p)),
        ("v", ctypes.POINTER(ctypes.c_void_p)),
        ("q_stride_tok", ctypes.c_int64),
        ("q_stride_head", ctypes.c_int64),
        ("kv_stride_tok", ctypes.c_int64),
        ("kv_stride_head", ctypes.c_int64),
        ("alpha", ctypes.c_double),
        ("r", ctypes.c_double),
        ("n_prefix", ctypes.c_void_p),
        ("q_visual", ctypes.POINTER(ctypes.c_void_p)),
    ]


_lib = None


class DecodeProblemStruct(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32), ("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("kv_rows", ctypes.c_int64), ("max_rows", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("row_begin", ctypes.c_void_p), ("row_end", ctypes.c_void_p),
        ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
        ("q_stride_seq", ctypes.c_int64), ("q_stride_head", ctypes.c_int64),
        ("kv_stride_row", ctypes.c_int64), ("kv_stride_head", ctypes.c_int64),
        ("new_stride_seq", ctypes.c_int64), ("new_stride_head", ctypes.c_int64),
        ("out", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("flags", ctypes.c_int32), ("reserved1", ctypes.c_int32),
        ("row_index", ctypes.c_void_p), ("index_len", ctypes.c_int64),
    ]


class QuantProblemStruct(ctypes.Structure):
    _fields_ = [
        ("num_units", ctypes.c_int32), ("h_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("reserved0", ctypes.c_int32), ("reserved1", ctypes.c_int32),
        ("rows", ctypes.c_int64), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("kv_stride_row", ctypes.c_int64), ("kv_stride_head", ctypes.c_int64),
        ("offsets", ctypes.c_void_p), ("k8", ctypes.c_void_p), ("v8", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
    ]


def lib():
    """The loaded CUDA library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing; build it with `python -m lvlm_kv_cache_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(ProblemStruct)
        vp, sz, i64, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64, ctypes.c_int
        L.aircache_workspace_size.argtypes = [P]
        L.aircache_workspace_size.restype = sz
        L.aircache_compress_bound.argtypes = [P]
        L.aircache_compress_bound.restype = i64
        L.aircache_score.argtypes = [P, vp, sz, vp, vp, vp, vp]
        L.aircache_score.restype = i32
        L.aircache_budget.argtypes = [P, vp, vp, sz, vp, vp, vp]
        L.aircache_budget.restype = i32
        L.aircache_budget_noalloc.argtypes = [P, vp, vp, vp, vp, vp]
        L.aircache_budget_noalloc.restype = i32
        L.aircache_select.argtypes = [P, vp, vp, vp, sz, vp, vp]
        L.aircache_select.restype = i32
        L.aircache_compact.argtypes = [P, vp, vp, vp, sz, vp, vp, vp, i64, vp]
        L.aircache_compact.restype = i32
        L.aircache_compress.argtypes = [P, vp, sz, vp, vp, vp, i64, vp, vp, vp, vp]
        L.aircache_compress.restype = i32
        L.aircache_get_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
        L.aircache_get_error.restype = i32
        L.aircache_status_string.argtypes = [i32]
        L.aircache_status_string.restype = ctypes.c_char_p
        L.aircache_compress_launches.argtypes = [P]
        L.aircache_compress_launches.restype = i32
        L.aircache_compress_profile.argtypes = [P, vp, sz, vp, vp, vp, i64, vp, vp, vp,
                                                ctypes.POINTER(ctypes.c_void_p), i32, vp]
        L.aircache_compress_profile.restype = i32
        pv = ctypes.POINTER(ctypes.c_void_p)
        L.aircache_prefill.argtypes = [P, pv, i64, i64, pv, i64, i64, vp, sz, vp]
        L.aircache_prefill.restype = i32
        L.aircache_prefill_compress.argtypes = [P, pv, i64, i64, pv, i64, i64, vp, sz, vp, vp, vp, i64, vp, vp,
                                                vp, vp]
        L.aircache_prefill_compress.restype = i32
        L.aircache_kernel_name.argtypes = [P, i32]
        L.aircache_kernel_name.restype = ctypes.c_char_p
        L.aircache_row_index.argtypes = [P, vp, vp, vp, vp, sz, vp, i64, vp]
        L.aircache_row_index.restype = i32
        L.aircache_quantize_int8.argtypes = [ctypes.POINTER(QuantProblemStruct), vp, vp]
        L.aircache_quantize_int8.restype = i32
        DP = ctypes.POINTER(DecodeProblemStruct)
        L.aircache_decode_workspace_size.argtypes = [DP]
        L.aircache_decode_workspace_size.restype = sz
        L.aircache_decode_splits.argtypes = [DP]
        L.aircache_decode_splits.restype = i32
        L.aircache_decode.argtypes = [DP, vp, sz, vp]
        L.aircache_decode.restype = i32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().aircache_status_string(int(status)).decode()
    except ImportError:
        return "library not loaded"


def _check(status: int, where: str):
    if status != OK:
        raise AirCacheError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Problem:
    """A compression problem over torch tensors (kept alive by this object).

    q, k, v: either stacked tensors [L, T, H, D] or lists of per-layer [T, H, D]
    tensors (same strides for every layer); q holds the text rows only.
    cu_seqlens, cu_visual: int32 device tensors [B+1].
    max_visual, max_text: host maxima over the requests.
    """

    def __init__(self, q, k, v, cu_seqlens, cu_visual, max_visual, max_text, alpha=0.9, r=0.1,
                 max_elite=0, total_tokens=None, total_visual=None, window_mode=0, budget_mode=0,
                 n_prefix=None, head_sets=False, q_visual=None, wait_test=False):
        qs = list(q.unbind(0)) if torch.is_tensor(q) else list(q)
        ks = list(k.unbind(0)) if torch.is_tensor(k) else list(k)
        vs = list(v.unbind(0)) if torch.is_tensor(v) else list(v)
        L = len(qs)
        if not (len(ks) == len(vs) == L) or L < 1 or L > MAX_LAYERS:
            raise ValueError("q, k, v must have the same number of layers (1..256)")
        dt = qs[0].dtype
        if dt not in (torch.float32, torch.bfloat16) or any(t.dtype != dt for t in qs + ks + vs):
            raise TypeError("q, k, v must all be float32 or all bfloat16")
        self.dtype = dt
        self.layers = (qs, ks, vs)  # keep alive
        B = cu_seqlens.numel() - 1
        T = int(total_tokens) if total_tokens is not None else int(ks[0].shape[0])
        TV = int(total_visual) if total_visual is not None else None
        if TV is None:
            TV = int(cu_visual[-1].item())
        self.B, self.L = B, L
        self.head_sets = bool(head_sets)
        self.h_q, self.h_kv, self.d = int(qs[0].shape[1]), int(ks[0].shape[1]), int(ks[0].shape[2])
        self.total_tokens, self.total_visual = T, TV
        self.cu_seqlens, self.cu_visual = cu_seqlens, cu_visual
        arr = ctypes.c_void_p * L
        self._q = arr(*[t.data_ptr() for t in qs])
        self._k = arr(*[t.data_ptr() for t in ks])
        self._v = arr(*[t.data_ptr() for t in vs])
        self.c = ProblemStruct(
            num_layers=L, num_requests=B, h_q=self.h_q, h_kv=self.h_kv, head_dim=self.d,
            dtype=BF16 if dt == torch.bfloat16 else F32,
            max_visual=int(max_visual), max_text=int(max_text), max_elite=int(max_elite),
            variant=int(window_mode) | (int(budget_mode) << 8) | ((1 << 16) if head_sets else 0)
            | (VARIANT_WAIT_TEST if wait_test else 0),
            total_tokens=T, total_visual=TV,
            cu_seqlens=cu_seqlens.data_ptr(), cu_visual=cu_visual.data_ptr(),
            q_text=ctypes.cast(self._q, ctypes.POINTER(ctypes.c_void_p)),
            k=ctypes.cast(self._k, ctypes.POINTER(ctypes.c_void_p)),
            v=ctypes.cast(self._v, ctypes.POINTER(ctypes.c_void_p)),
            q_stride_tok=qs[0].stride(0), q_stride_head=qs[0].stride(1),
            kv_stride_tok=ks[0].stride(0), kv_stride_head=ks[0].stride(1),
            alpha=float(alpha), r=float(r),
            n_prefix=n_prefix.data_ptr() if n_prefix is not None else None,
        )
        if q_visual is not None:  # window 4: the visual tokens' queries, per layer [total_visual, H_q, D]
            qvs = list(q_visual.unbind(0)) if torch.is_tensor(q_visual) else list(q_visual)
            if len(qvs) != L or any(t.stride() != qs[0].stride() for t in qvs):
                raise ValueError("q_visual: one tensor per layer with q's strides")
            self._qv = arr(*[t.data_ptr() for t in qvs])
            self.c.q_visual = ctypes.cast(self._qv, ctypes.POINTER(ctypes.c_void_p))
            self.q_visual = qvs  # keep alive
        self.n_prefix = n_prefix  # keep alive
        for t in ks + vs + qs:
            if t.stride(2) != 1:
                raise ValueError("head_dim must be contiguous")
        if any(t.stride() != ks[0].stride() for t in ks + vs) or any(t.stride() != qs[0].stride() for t in qs):
            raise ValueError("every layer must share the same strides")

    @property
    def ref(self):
        return ctypes.byref(self.c)

    def workspace_size(self) -> int:
        n = lib().aircache_workspace_size(self.ref)
        if n == 0:
            raise AirCacheError(ERR_INVALID_ARG, "aircache_workspace_size")
        return int(n)

    def compress_bound(self) -> int:
        n = lib().aircache_compress_bound(self.ref)
        if n < 0:
            raise AirCacheError(ERR_INVALID_ARG, "aircache_compress_bound")
        return int(n)

    def launches(self) -> int:
        return int(lib().aircache_compress_launches(self.ref))

    @property
    def max_text(self):
        return self.c.max_text

    def new_workspace(self, device=None) -> torch.Tensor:
        """A 256-byte-aligned device workspace (torch allocations are 512-B aligned)."""
        dev = device or self.layers[1][0].device
        return torch.empty(self.workspace_size(), dtype=torch.uint8, device=dev)


# ------------------------------------------------------------------ entry points

def aircache_score(prob: Problem, ws, iv, elite, n_tk, stream=None):
    _check(lib().aircache_score(prob.ref, _ptr(ws), ws.numel(), _ptr(iv), _ptr(elite), _ptr(n_tk),
                                _stream(stream)), "aircache_score")


def aircache_budget(prob: Problem, iv, ws, stats, keep, stream=None):
    _check(lib().aircache_budget(prob.ref, _ptr(iv), _ptr(ws), ws.numel(), _ptr(stats), _ptr(keep),
                                 _stream(stream)), "aircache_budget")


def aircache_budget_noalloc(prob: Problem, iv, stats, keep, device_status=None, stream=None):
    """aircache_budget with the library's fixed device scratch instead of a
    workspace (for callers that cannot allocate; at most
    AIRCACHE_NOALLOC_MAX_UNITS layer-request pairs; calls must not overlap)."""
    _check(lib().aircache_budget_noalloc(prob.ref, _ptr(iv), _ptr(stats), _ptr(keep), _ptr(device_status),
                                         _stream(stream)), "aircache_budget_noalloc")


def aircache_select(prob: Problem, iv, keep, ws, idx, stream=None):
    _check(lib().aircache_select(prob.ref, _ptr(iv), _ptr(keep), _ptr(ws), ws.numel(), _ptr(idx),
                                 _stream(stream)), "aircache_select")


def aircache_compact(prob: Problem, idx, keep, ws, out_k, out_v, out_offsets, stream=None):
    cap = out_k.shape[0]
    _check(lib().aircache_compact(prob.ref, _ptr(idx), _ptr(keep), _ptr(ws), ws.numel(), _ptr(out_k),
                                  _ptr(out_v), _ptr(out_offsets), cap, _stream(stream)),
           "aircache_compact")


def aircache_compress(prob: Problem, ws, out_k, out_v, out_offsets, keep, idx=None, iv=None, stream=None):
    cap = out_k.shape[0]
    _check(lib().aircache_compress(prob.ref, _ptr(ws), ws.numel(), _ptr(out_k), _ptr(out_v),
                                   _ptr(out_offsets), cap, _ptr(keep), _ptr(idx), _ptr(iv),
                                   _stream(stream)), "aircache_compress")


def _layer_array(ts):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return arr, ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))


def aircache_prefill(prob: Problem, q_all, attn_out, ws, stream=None):
    """Causal prefill attention of every layer: q_all [L][T][H_q][D] (every
    prompt row), attn_out [L][T][H_q][D] bf16 (written)."""
    qs = list(q_all.unbind(0)) if torch.is_tensor(q_all) else list(q_all)
    os_ = list(attn_out.unbind(0)) if torch.is_tensor(attn_out) else list(attn_out)
    qa, qp = _layer_array(qs)
    oa, op = _layer_array(os_)
    _check(lib().aircache_prefill(prob.ref, qp, qs[0].stride(0), qs[0].stride(1), op, os_[0].stride(0),
                                  os_[0].stride(1), _ptr(ws), ws.numel(), _stream(stream)), "aircache_prefill")


def aircache_prefill_compress(prob: Problem, q_all, attn_out, ws, out_k, out_v, out_offsets, keep, idx=None,
                              iv=None, stream=None):
    """The prefill attention and, from its own logits, the whole compression."""
    qs = list(q_all.unbind(0)) if torch.is_tensor(q_all) else list(q_all)
    os_ = list(attn_out.unbind(0)) if torch.is_tensor(attn_out) else list(attn_out)
    qa, qp = _layer_array(qs)
    oa, op = _layer_array(os_)
    cap = out_k.shape[0]
    _check(lib().aircache_prefill_compress(prob.ref, qp, qs[0].stride(0), qs[0].stride(1), op, os_[0].stride(0),
                                           os_[0].stride(1), _ptr(ws), ws.numel(), _ptr(out_k), _ptr(out_v),
                                           _ptr(out_offsets), cap, _ptr(keep), _ptr(idx), _ptr(iv),
                                           _stream(stream)), "aircache_prefill_compress")


def prefill_compress(prob: Problem, q_all, attn_out=None, ws=None, out=None, stream=None, check=True):
    """aircache_prefill_compress with allocated outputs; returns (attn_out, out dict)."""
    ws = prob.new_workspace() if ws is None else ws
    out = alloc_outputs(prob) if out is None else out
    if attn_out is None:
        attn_out = torch.empty(q_all.shape, dtype=torch.bfloat16, device=q_all.device)
    aircache_prefill_compress(prob, q_all, attn_out, ws, out["out_k"], out["out_v"], out["out_offsets"],
                              out["keep"], out["idx"], out["iv"], stream)
    if check:
        st = aircache_get_error(ws, stream)
        if st != OK:
            raise AirCacheError(st, "aircache_prefill_compress (device)")
    return attn_out, out


def aircache_compress_profile(prob: Problem, ws, out_k, out_v, out_offsets, keep, events, idx=None,
                              iv=None, stream=None):
    """aircache_compress recording torch.cuda.Event objects around each kernel
    (len(events) == prob.launches() + 1)."""
    cap = out_k.shape[0]
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().aircache_compress_profile(prob.ref, _ptr(ws), ws.numel(), _ptr(out_k), _ptr(out_v),
                                           _ptr(out_offsets), cap, _ptr(keep), _ptr(idx), _ptr(iv),
                                           arr, len(events), _stream(stream)),
           "aircache_compress_profile")


def kernel_names(prob: "Problem"):
    """Names of the kernels one aircache_compress call on `prob` launches, in order."""
    n = prob.launches()
    return [lib().aircache_kernel_name(prob.ref, i).decode() for i in range(n)]


def aircache_get_error(ws, stream=None) -> int:
    st = ctypes.c_int32(0)
    _check(lib().aircache_get_error(_ptr(ws), _stream(stream), ctypes.byref(st)), "aircache_get_error")
    return int(st.value)


# ------------------------------------------------------------------ conveniences

def alloc_outputs(prob: Problem, device=None):
    """Device buffers for aircache_compress: out_k, out_v ([bound, H_kv, D]),
    out_offsets [L*B+1], keep [L*B], idx and iv [L, total_visual]."""
    dev = device or prob.layers[1][0].device
    rows = prob.compress_bound()
    L, B = prob.L, prob.B
    return {
        "out_k": torch.empty((rows, prob.h_kv, prob.d), dtype=prob.dtype, device=dev),
        "out_v": torch.empty((rows, prob.h_kv, prob.d), dtype=prob.dtype, device=dev),
        "out_offsets": torch.empty(L * B + 1, dtype=torch.int64, device=dev),
        "keep": torch.empty(L * B, dtype=torch.int32, device=dev),
        "idx": torch.empty((L, prob.h_kv, prob.total_visual) if prob.head_sets else (L, prob.total_visual),
                           dtype=torch.int32, device=dev),
        "iv": torch.empty((L, prob.total_visual), dtype=torch.float32, device=dev),
    }


def compress(prob: Problem, ws=None, out=None, stream=None, check=True):
    """One fused compression; returns the output dict (see alloc_outputs).
    With check=True the device error word is read (this synchronises)."""
    ws = prob.new_workspace() if ws is None else ws
    out = alloc_outputs(prob) if out is None else out
    aircache_compress(prob, ws, out["out_k"], out["out_v"], out["out_offsets"], out["keep"],
                      out["idx"], out["iv"], stream)
    if check:
        st = aircache_get_error(ws, stream)
        if st != OK:
            raise AirCacheError(st, "aircache_compress (device)")
    return out


def compress_host(q, k, v, cu_seqlens, cu_visual, max_visual, max_text, alpha=0.9, r=0.1,
                  device="cuda", stream=None):
    """End-to-end from HOST tensors: copies q, k and the offsets to the device,
    compresses, and copies the compacted cache and its offsets back.  Values in
    page-locked memory (v.is_pinned()) stay on the host: only the compaction
    reads them, and only the rows it keeps; other values are copied first.
    Returns (out_k, out_v, out_offsets) as host tensors trimmed to the rows used."""
    dq = q.to(device, non_blocking=True)
    dk = k.to(device, non_blocking=True)
    dv = v if v.is_pinned() else v.to(device, non_blocking=True)
    dcs = cu_seqlens.to(device, non_blocking=True)
    dcv = cu_visual.to(device, non_blocking=True)
    prob = Problem(dq, dk, dv, dcs, dcv, max_visual, max_text, alpha, r,
                   total_tokens=k.shape[1], total_visual=int(cu_visual[-1]))
    out = compress(prob, stream=stream)
    offs = out["out_offsets"].cpu()
    rows = int(offs[-1])
    return out["out_k"][:rows].cpu(), out["out_v"][:rows].cpu(), offs


def math_bound(L, B, total_text, total_visual, r):
    """The compress_bound formula, for host-side sizing without the library."""
    return L * total_text + math.ceil(r * L * total_visual) + B * (2 * L + 1)


# ------------------------------------------------------------------ decode

class DecodeProblem:
    """One decode step over cached rows (see aircache_decode in the header).

    q: [S, H_q, D] bf16 (one query row per sequence); k, v: arenas
    [rows, H_kv, D] bf16, or int8 codes with k_scale, v_scale [S, H_kv] fp32;
    row_begin, row_end: int64 device tensors [S] (or one offsets tensor [S+1]
    via ``offsets=``); k_new, v_new: optional [S, H_kv, D] bf16; out: fp32
    [S, H_q, D] (allocated when None).  max_rows: the expected longest range
    (sizes the split; not a limit).  early_cache: AIRCACHE_DECODE_EARLY_CACHE
    (programmatic dependent launch; the kernel launched just before on the
    stream must not write the ranges or the cached rows)."""

    def __init__(self, q, k, v, row_begin=None, row_end=None, max_rows=0, k_new=None, v_new=None,
                 out=None, offsets=None, k_scale=None, v_scale=None, early_cache=False, row_index=None):
        if offsets is not None:
            row_begin, row_end = offsets[:-1], offsets[1:]
        S, h_q, d = (int(x) for x in q.shape)
        h_kv = int(k.shape[1])
        if out is None:
            out = torch.empty((S, h_q, d), dtype=torch.float32, device=q.device)
        for t in (q, k, v) + ((k_new, v_new) if k_new is not None else ()):
            if t.stride(-1) != 1:
                raise ValueError("head_dim must be contiguous")
        if k.stride() != v.stride() or (k_new is not None and k_new.stride() != v_new.stride()):
            raise ValueError("k and v (and k_new and v_new) must share strides")
        if row_begin.dtype != torch.int64 or row_end.dtype != torch.int64:
            raise TypeError("row ranges are int64")
        if not out.is_contiguous() or tuple(out.shape) != (S, h_q, d) or out.dtype != torch.float32:
            raise ValueError("out must be a dense fp32 [S, H_q, D] tensor")
        q8 = k.dtype == torch.int8
        if q8 and (k_scale is None or v_scale is None or not k_scale.is_contiguous() or not v_scale.is_contiguous()):
            raise ValueError("int8 caches need contiguous k_scale and v_scale [S, H_kv]")
        if row_index is not None and (row_index.dtype != torch.int32 or not row_index.is_contiguous()):
            raise TypeError("row_index is a contiguous int32 tensor")
        self.keep = (q, k, v, row_begin, row_end, k_new, v_new, out, k_scale, v_scale, row_index)
        self.out = out
        self.c = DecodeProblemStruct(
            num_seqs=S, h_q=h_q, h_kv=h_kv, head_dim=d,
            dtype=BF16 if q.dtype == torch.bfloat16 else F32, kv_dtype=INT8 if q8 else BF16,
            kv_rows=int(k.shape[0]), max_rows=int(max_rows),
            q=q.data_ptr(), k=k.data_ptr(), v=v.data_ptr(),
            row_begin=row_begin.data_ptr(), row_end=row_end.data_ptr(),
            k_new=k_new.data_ptr() if k_new is not None else None,
            v_new=v_new.data_ptr() if v_new is not None else None,
            q_stride_seq=q.stride(0), q_stride_head=q.stride(1),
            kv_stride_row=k.stride(0), kv_stride_head=k.stride(1),
            new_stride_seq=k_new.stride(0) if k_new is not None else 0,
            new_stride_head=k_new.stride(1) if k_new is not None else 0,
            out=out.data_ptr(),
            k_scale=k_scale.data_ptr() if q8 else None, v_scale=v_scale.data_ptr() if q8 else None,
            flags=DECODE_EARLY_CACHE if early_cache else 0, reserved1=0,
            row_index=row_index.data_ptr() if row_index is not None else None,
            index_len=row_index.numel() if row_index is not None else 0,
        )

    @property
    def ref(self):
        return ctypes.byref(self.c)

    def workspace_size(self) -> int:
        n = lib().aircache_decode_workspace_size(self.ref)
        if n == 0:
            raise AirCacheError(ERR_INVALID_ARG, "aircache_decode_workspace_size")
        return int(n)

    def splits(self) -> int:
        return int(lib().aircache_decode_splits(self.ref))

    def new_workspace(self, device=None) -> torch.Tensor:
        """A zeroed decode workspace (zeroed once; every call leaves it zeroed
        again, apart from a recorded device error)."""
        return torch.zeros(self.workspace_size(), dtype=torch.uint8, device=device or self.out.device)


def aircache_decode(prob: DecodeProblem, ws, stream=None):
    _check(lib().aircache_decode(prob.ref, _ptr(ws), ws.numel(), _stream(stream)), "aircache_decode")


def decode(prob: DecodeProblem, ws=None, stream=None, check=True):
    """One decode step; returns prob.out.  check=True reads the device error word (synchronises)."""
    ws = prob.new_workspace() if ws is None else ws
    aircache_decode(prob, ws, stream)
    if check:
        st = aircache_get_error(ws, stream)
        if st != OK:
            raise AirCacheError(st, "aircache_decode (device)")
    return prob.out


# ------------------------------------------------------------------ int8 storage

def aircache_quantize_int8(k, v, offsets, k8, v8, k_scale, v_scale, status=None, stream=None):
    """int8 codes and per-(unit, KV head) scales of the bf16 arenas k, v
    ([rows, H_kv, D]); units are offsets[u] .. offsets[u+1]-1 (int64 device)."""
    c = QuantProblemStruct(
        num_units=offsets.numel() - 1, h_kv=int(k.shape[1]), head_dim=int(k.shape[2]),
        dtype=BF16 if k.dtype == torch.bfloat16 else F32, reserved0=0, reserved1=0,
        rows=int(k.shape[0]), k=k.data_ptr(), v=v.data_ptr(),
        kv_stride_row=k.stride(0), kv_stride_head=k.stride(1), offsets=offsets.data_ptr(),
        k8=k8.data_ptr(), v8=v8.data_ptr(), k_scale=k_scale.data_ptr(), v_scale=v_scale.data_ptr())
    if k.stride() != v.stride() or k.stride(2) != 1:
        raise ValueError("k and v must share strides, head_dim contiguous")
    _check(lib().aircache_quantize_int8(ctypes.byref(c), _ptr(status), _stream(stream)), "aircache_quantize_int8")


def quantize_int8(k, v, offsets, stream=None, check=True):
    """Allocates and returns (k8, v8, k_scale, v_scale) for the arenas k, v."""
    U = offsets.numel() - 1
    k8 = torch.empty(k.shape, dtype=torch.int8, device=k.device)
    v8 = torch.empty(v.shape, dtype=torch.int8, device=v.device)
    ks = torch.empty((U, k.shape[1]), dtype=torch.float32, device=k.device)
    vs = torch.empty((U, k.shape[1]), dtype=torch.float32, device=k.device)
    st = torch.zeros(1, dtype=torch.int32, device=k.device) if check else None
    aircache_quantize_int8(k, v, offsets, k8, v8, ks, vs, st, stream)
    if check and int(st.item()) != OK:
        raise AirCacheError(int(st.item()), "aircache_quantize_int8 (device)")
    return k8, v8, ks, vs


def aircache_row_index(prob: Problem, keep, idx, out_offsets, ws, row_index, stream=None):
    _check(lib().aircache_row_index(prob.ref, _ptr(keep), _ptr(idx), _ptr(out_offsets), _ptr(ws), ws.numel(),
                                    _ptr(row_index), row_index.numel(), _stream(stream)), "aircache_row_index")


def row_index(prob: Problem, out, ws=None, stream=None, check=True):
    """The compacted rows' prompt positions (int32 [rows]) for a gather-fused
    decode from the full cache; `out` is aircache_compress's output dict."""
    ws = prob.new_workspace() if ws is None else ws
    rows = int(out["out_offsets"][-1])
    ri = torch.empty(max(rows, 1), dtype=torch.int32, device=out["keep"].device)
    aircache_row_index(prob, out["keep"], out["idx"], out["out_offsets"], ws, ri, stream)
    if check:
        st = aircache_get_error(ws, stream)
        if st != OK:
            raise AirCacheError(st, "aircache_row_index (device)")
    return ri
