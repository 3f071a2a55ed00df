"""AirCache oracle, Python side -- TEST INFRASTRUCTURE ONLY.

ctypes bindings for the plain fp64 C oracle in ``aircache_oracle.c``.  Only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use
this module; the product library never imports it, and it imports nothing from
the product.

Arrays are numpy, token-major ``[tokens, heads, D]`` with D contiguous.  fp32
tensors are passed as ``float32``; bf16 tensors as their raw bits in ``uint16``
(the C side decodes them exactly).  Every function works on one request (and,
where stated, one layer); the formulas and their sources are documented in the
C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "aircache_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1


class _View(ctypes.Structure):
    _fields_ = [
        ("base", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("stride_tok", ctypes.c_int64),
        ("stride_head", ctypes.c_int64),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, strict fp64, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "aircache_oracle.h"))
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
             "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        # A test may point this at a deliberately altered build of the oracle.
        path = os.environ.get("AIRCACHE_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        V = ctypes.POINTER(_View)
        L.oracle_elite.argtypes = [V, V, i32, i32, i32, i32, i32, i32, f64, vp, vp]
        L.oracle_elite.restype = i32
        L.oracle_score.argtypes = [V, V, i32, i32, i32, i32, i32, i32, vp, i32, vp, vp, vp]
        L.oracle_score.restype = i32
        L.oracle_stats.argtypes = [vp, i32, vp]
        L.oracle_stats.restype = i32
        L.oracle_budget.argtypes = [vp, vp, i32, i32, f64, vp, vp]
        L.oracle_budget.restype = i32
        L.oracle_select.argtypes = [vp, i32, i32, vp]
        L.oracle_select.restype = i32
        L.oracle_compact.argtypes = [V, i32, i32, i32, i32, i32, vp, i32, vp]
        L.oracle_compact.restype = i64
        L.oracle_request.argtypes = [V, V, i32, i32, i32, i32, i32, i32, f64, f64,
                                     vp, vp, vp, vp, vp, vp]
        L.oracle_request.restype = i32
        L.oracle_decode.argtypes = [V, V, V, i32, i32, i32, i64, vp]
        L.oracle_decode.restype = i32
        L.oracle_quant_code.argtypes = [ctypes.c_float, ctypes.c_float]
        L.oracle_quant_code.restype = i32
        L.oracle_quantize_int8.argtypes = [V, i64, i32, i32, vp, vp]
        L.oracle_quantize_int8.restype = i32
        L.oracle_window.argtypes = [i32, i32, vp]
        L.oracle_window.restype = i32
        L.oracle_budget_variant.argtypes = [vp, vp, i32, i32, f64, i32, vp, vp]
        L.oracle_budget_variant.restype = i32
        L.oracle_request_variant.argtypes = [V, V, i32, i32, i32, i32, i32, i32, i32, f64, f64, i32, i32,
                                             vp, vp, vp, vp, vp, vp, vp, vp, V]
        L.oracle_window_visual.argtypes = [i32, vp]
        L.oracle_window_visual.restype = i32
        L.oracle_score_visual_window.argtypes = [V, V, i32, i32, i32, i32, i32, vp, i32, vp]
        L.oracle_score_visual_window.restype = i32
        L.oracle_compact_heads.argtypes = [V, i32, i32, i32, i32, i32, vp, i32, vp]
        L.oracle_compact_heads.restype = i64
        L.oracle_request_variant.restype = i32
        _lib = L
    return _lib


def _view(a: np.ndarray) -> _View:
    if a.ndim != 3:
        raise ValueError("expected a [tokens, heads, D] array")
    if a.dtype == np.float32:
        dt = F32
    elif a.dtype == np.uint16:
        dt = BF16
    else:
        raise TypeError("oracle arrays are float32 or uint16 (bf16 bits)")
    es = a.itemsize
    if a.size == 0:  # no element is read: any strides will do
        return _View(a.ctypes.data, dt, 0, a.shape[1] * a.shape[2], a.shape[2])
    if a.strides[2] != es:
        raise ValueError("D must be contiguous")
    return _View(a.ctypes.data, dt, 0, a.strides[0] // es, a.strides[1] // es)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def elite(q: np.ndarray, k: np.ndarray, n_v: int, alpha: float, n_p: int = 0):
    """Elite window of one (request, layer): q = this request's text queries
    [N_t, H_q, D]; k = this request's keys [N_v+N_t, H_kv, D] in prompt order
    (n_p prefix text rows, the visual rows, the other text rows; reading R18).
    Returns (elite positions (text-relative, ascending), head-mean row P)."""
    n_t, h_q, d = q.shape
    h_kv = k.shape[1]
    P = np.zeros(n_t, np.float64)
    el = np.zeros(n_t, np.int32)
    n = lib().oracle_elite(ctypes.byref(_view(q)), ctypes.byref(_view(k)), h_q, h_kv, d,
                           n_v, n_t, int(n_p), float(alpha), _ptr(P), _ptr(el))
    if n < 0:
        raise ValueError("oracle_elite rejected its arguments")
    return el[:n].copy(), P


def score(q: np.ndarray, k: np.ndarray, n_v: int, elite_idx: np.ndarray, n_p: int = 0):
    """I_v of one (request, layer) for a given elite set.
    Returns (I_v [N_v] fp64, elite-key mass [H_q, N_tk])."""
    n_t, h_q, d = q.shape
    h_kv = k.shape[1]
    el = np.ascontiguousarray(elite_idx, dtype=np.int32)
    iv = np.zeros(n_v, np.float64)
    mass = np.zeros(h_q * len(el), np.float64)
    rc = lib().oracle_score(ctypes.byref(_view(q)), ctypes.byref(_view(k)), h_q, h_kv, d,
                            n_v, n_t, int(n_p), _ptr(el), len(el), _ptr(iv), _ptr(mass), None)
    if rc != 0:
        raise ValueError("oracle_score rejected its arguments")
    return iv, mass.reshape(h_q, len(el))


def score_heads(q: np.ndarray, k: np.ndarray, n_v: int, elite_idx: np.ndarray, n_p: int = 0):
    """I_v and the per-KV-head I_v^(h) [H_kv, N_v] of one (request, layer) for a
    given elite set (reading R19)."""
    n_t, h_q, d = q.shape
    h_kv = k.shape[1]
    el = np.ascontiguousarray(elite_idx, dtype=np.int32)
    iv = np.zeros(n_v, np.float64)
    ivh = np.zeros((h_kv, n_v), np.float64)
    rc = lib().oracle_score(ctypes.byref(_view(q)), ctypes.byref(_view(k)), h_q, h_kv, d,
                            n_v, n_t, int(n_p), _ptr(el), len(el), _ptr(iv), None, _ptr(ivh))
    if rc != 0:
        raise ValueError("oracle_score rejected its arguments")
    return iv, ivh


def compact_heads(src: np.ndarray, n_v: int, n_t: int, idx_heads, n_p: int = 0) -> np.ndarray:
    """Compaction with one visual index set per KV head (reading R19): idx_heads
    [H_kv, keep]; dense [keep+N_t, H_kv, D]."""
    h_kv, d = src.shape[1], src.shape[2]
    ih = np.asarray(idx_heads, dtype=np.int32)
    keep = ih.shape[1]
    full = np.zeros((h_kv, n_v), np.int32)
    full[:, :keep] = ih
    out = np.zeros((keep + n_t, h_kv, d), src.dtype)
    n = lib().oracle_compact_heads(ctypes.byref(_view(src)), h_kv, d, n_v, n_t, int(n_p), _ptr(full), keep,
                                   _ptr(out))
    assert n == keep + n_t
    return out


def stats(iv: np.ndarray):
    """(s_t, s_k, mu, sigma) of one I_v vector."""
    v = np.ascontiguousarray(iv, dtype=np.float64)
    out = np.zeros(4, np.float64)
    if lib().oracle_stats(_ptr(v), len(v), _ptr(out)) != 0:
        raise ValueError("oracle_stats needs N_v >= 3")
    return tuple(float(x) for x in out)


def budget(s_t, s_k, n_v: int, r: float):
    """Per-layer (r_l, keep) of one request from its per-layer strength/skewness."""
    st = np.ascontiguousarray(s_t, dtype=np.float64)
    sk = np.ascontiguousarray(s_k, dtype=np.float64)
    L = len(st)
    rl = np.zeros(L, np.float64)
    keep = np.zeros(L, np.int32)
    if lib().oracle_budget(_ptr(st), _ptr(sk), L, n_v, float(r), _ptr(rl), _ptr(keep)) != 0:
        raise ValueError("oracle_budget rejected its arguments")
    return rl, keep


def decode(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """One decode step of attention: q [H_q, D] (one query row), k, v
    [rows, H_kv, D] (the cached rows).  Returns o [H_q, D] in fp64."""
    h_q, d = q.shape
    h_kv = k.shape[1]
    qv = _view(np.ascontiguousarray(q).reshape(1, h_q, d))
    out = np.zeros((h_q, d), np.float64)
    rc = lib().oracle_decode(ctypes.byref(qv), ctypes.byref(_view(k)), ctypes.byref(_view(v)), h_q, h_kv, d,
                             int(k.shape[0]), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return out


def quant_code(x: float, s: float) -> int:
    """The symmetric int8 step clip(round(x / s), -127, 127) in fp32 (reading R17)."""
    return int(lib().oracle_quant_code(float(x), float(s)))


def quantize_int8(src: np.ndarray):
    """Per-head int8 codes of one compacted unit src [rows, H_kv, D] (fp32 or
    bf16 bits).  Returns (codes int8 [rows, H_kv, D], scales fp32 [H_kv])."""
    rows, h_kv, d = src.shape
    codes = np.zeros((rows, h_kv, d), np.int8)
    scales = np.zeros(h_kv, np.float32)
    rc = lib().oracle_quantize_int8(ctypes.byref(_view(src)), rows, h_kv, d, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("oracle_quantize_int8 rejected its arguments")
    return codes, scales


def window(n_t: int, mode: int) -> np.ndarray:
    """Observation window of an ablation variant (1: last 16 text tokens,
    2: last 32, 3: every text token), text-relative, ascending."""
    pos = np.zeros(max(int(n_t), 1), np.int32)
    n = lib().oracle_window(int(n_t), int(mode), _ptr(pos))
    if n < 0:
        raise ValueError("oracle_window rejected its arguments")
    return pos[:n].copy()


def budget_variant(s_t, s_k, n_v: int, r: float, mode: int):
    """Per-layer (r_l, keep) under a budget variant (0: the method's own,
    1: uniform, 2: PyramidKV-style, 3: strength only, 4: skewness only)."""
    st = np.ascontiguousarray(s_t, dtype=np.float64)
    sk = np.ascontiguousarray(s_k, dtype=np.float64)
    L = len(st)
    rl = np.zeros(L, np.float64)
    keep = np.zeros(L, np.int32)
    if lib().oracle_budget_variant(_ptr(st), _ptr(sk), L, n_v, float(r), int(mode), _ptr(rl),
                                   _ptr(keep)) != 0:
        raise ValueError("oracle_budget_variant rejected its arguments")
    return rl, keep


def select(iv: np.ndarray, keep: int) -> np.ndarray:
    """Ascending positions of the `keep` largest I_v (ties to the lower index)."""
    v = np.ascontiguousarray(iv, dtype=np.float64)
    idx = np.zeros(max(int(keep), 1), np.int32)
    if lib().oracle_select(_ptr(v), len(v), int(keep), _ptr(idx)) != 0:
        raise ValueError("oracle_select rejected its arguments")
    return idx[: int(keep)].copy()


def compact(src: np.ndarray, n_v: int, n_t: int, idx: np.ndarray, n_p: int = 0) -> np.ndarray:
    """The kept visual rows (visual indices idx), then every text row in text
    order, of one (request, layer) whose rows are in prompt order with n_p
    prefix text rows; dense [keep+N_t, H_kv, D] in the source element type."""
    h_kv, d = src.shape[1], src.shape[2]
    el = np.ascontiguousarray(idx, dtype=np.int32)
    out = np.zeros((len(el) + n_t, h_kv, d), src.dtype)
    n = lib().oracle_compact(ctypes.byref(_view(src)), h_kv, d, n_v, n_t, int(n_p), _ptr(el),
                             len(el), _ptr(out))
    assert n == len(el) + n_t
    return out


def window_visual(n_v: int) -> np.ndarray:
    """R14's visual window: the last min(32, N_v) visual indices."""
    out = np.zeros(32, np.int32)
    n = lib().oracle_window_visual(int(n_v), _ptr(out))
    if n < 0:
        raise ValueError("oracle_window_visual rejected its arguments")
    return out[:n].copy()


def score_visual_window(qv: np.ndarray, k: np.ndarray, n_v: int, pos, n_p: int = 0) -> np.ndarray:
    """I_v of one (request, layer) for the visual window: qv [N_v, H_q, D] the
    visual tokens' queries, k [N_v+N_t, H_kv, D] in prompt order."""
    _, h_q, d = qv.shape
    h_kv = k.shape[1]
    ps = np.ascontiguousarray(pos, dtype=np.int32)
    iv = np.zeros(n_v, np.float64)
    rc = lib().oracle_score_visual_window(ctypes.byref(_view(qv)), ctypes.byref(_view(k)), h_q, h_kv, d, n_v,
                                          int(n_p), _ptr(ps), len(ps), _ptr(iv))
    if rc != 0:
        raise ValueError("oracle_score_visual_window rejected its arguments")
    return iv


def request(q_layers, k_layers, n_v: int, alpha: float, r: float, window_mode: int = 0,
            budget_mode: int = 0, n_p: int = 0, per_head: bool = False, qv_layers=None):
    """The whole one-shot pass for one request over its layers (optionally
    with an ablation window / budget variant).

    q_layers[l]: [N_t, H_q, D]; k_layers[l]: [N_v+N_t, H_kv, D].
    Returns a dict with per-layer iv, elite, n_tk, stats, keep, idx."""
    L = len(q_layers)
    n_t, h_q, d = q_layers[0].shape
    h_kv = k_layers[0].shape[1]
    qv = (_View * L)(*[_view(a) for a in q_layers])
    kv = (_View * L)(*[_view(a) for a in k_layers])
    qvis = (_View * L)(*[_view(a) for a in qv_layers]) if qv_layers is not None else None
    iv = np.zeros((L, n_v), np.float64)
    el = np.zeros((L, max(n_t, 32)), np.int32)
    ntk = np.zeros(L, np.int32)
    st = np.zeros((L, 4), np.float64)
    keep = np.zeros(L, np.int32)
    idx = np.zeros((L, n_v), np.int32)
    ivh = np.zeros((L, h_kv, n_v), np.float64) if per_head else None
    idxh = np.zeros((L, h_kv, n_v), np.int32) if per_head else None
    rc = lib().oracle_request_variant(qv, kv, L, h_q, h_kv, d, n_v, n_t, int(n_p), float(alpha), float(r),
                                      int(window_mode), int(budget_mode), _ptr(iv), _ptr(el),
                                      _ptr(ntk), _ptr(st), _ptr(keep), _ptr(idx),
                                      _ptr(ivh) if per_head else None, _ptr(idxh) if per_head else None, qvis)
    if rc != 0:
        raise ValueError("oracle_request rejected its arguments")
    return {
        "iv": iv,
        "elite": [el[l, : ntk[l]].copy() for l in range(L)],
        "n_tk": ntk,
        "stats": st,
        "keep": keep,
        "idx": [idx[l, : keep[l]].copy() for l in range(L)],
        **({"iv_heads": ivh, "idx_heads": [idxh[l, :, : keep[l]].copy() for l in range(L)]} if per_head else {}),
    }
