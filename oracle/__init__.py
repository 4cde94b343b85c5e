"""float64 CPU oracle for fused softmax attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs anything here, and this
package imports nothing from the product.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, three
passes per query row); this module only compiles it with gcc and marshals
numpy buffers through ctypes.

What it computes: O = softmax(Scale * Q K^T + Mask) V with the visibility and
special-value rules of "Attention" (recursiveai.org OneGPU docs), sections
"What it covers" and "Special values"; see the header of ``attn_oracle.c``
for every reading taken where the pages are silent.

Parity status per function:
  attn     -- pinned by tests/test_oracle.py (brute force, closed forms,
              invariants, torch CPU float64 SDPA, golden fixtures).
  combine  -- pinned by tests/test_oracle.py (split-then-combine equals the
              whole row; closed forms for empty and NaN ranges).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
INT64_MIN = -(2**63)


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so with gcc (no CUDA involved)."""
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Layout(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_int64), ("batch_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64), ("row_stride", ctypes.c_int64)]


class _Problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("q_len", ctypes.c_int32), ("k_len", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float), ("causal", ctypes.c_int32),
                ("causal_offset", ctypes.c_int64), ("masked_rows_zero", ctypes.c_int32),
                ("q", _Layout), ("k", _Layout), ("v", _Layout), ("mask", _Layout),
                ("seg_batch_stride", ctypes.c_int64), ("window_left", ctypes.c_int32),
                ("causal_align", ctypes.c_int32), ("k_lens_kind", ctypes.c_int32),
                ("softcap", ctypes.c_float), ("smooth_softmax", ctypes.c_int32),
                ("head_sink", ctypes.c_void_p), ("kv_int8", ctypes.c_int32),
                ("kv_per_channel", ctypes.c_int32), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.orc_attn_rows.restype = ctypes.c_int
        lib.orc_attn_rows.argtypes = [ctypes.POINTER(_Problem)] + [ctypes.c_void_p] * 6 + [
            ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
        lib.orc_combine.restype = ctypes.c_int
        lib.orc_combine.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
        lib.orc_append_rows.restype = ctypes.c_int
        lib.orc_append_rows.argtypes = ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] +
                                        [ctypes.c_int32] * 5 + [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                                ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32])
        lib.orc_widen.restype = ctypes.c_double
        lib.orc_widen.argtypes = [ctypes.c_int32, ctypes.c_uint32]
        lib.orc_default_scale.restype = ctypes.c_float
        lib.orc_default_scale.argtypes = [ctypes.c_int32]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _storage(a, dtype):
    if a is None:
        return None
    want = np.float32 if dtype == "f32" else np.uint16
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        raise TypeError(f"oracle expects {want} storage for {dtype}, got {a.dtype}")
    return a


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def attn(problem: dict, q, k, v, mask=None, seg=None, k_lens=None, rows=None, nthreads=None, head_sink=None,
         k_scale=None, v_scale=None):
    """O and LSE of the requested query rows, in float64.

    problem: dict with batch, heads, kv_heads, q_len, k_len, head_dim, dtype
      ('f32'|'f16'|'bf16'), scale (0 = default), causal, causal_offset (None =
      k_len - q_len), masked_rows ('nan'|'zero'), q_layout/k_layout/v_layout
      and mask_layout as (offset, batch_stride, head_stride, row_stride) in
      elements, seg_batch_stride; optional window_left (None/-1 = off),
      causal_align ('fixed' | 'klens'), k_lens_kind ('count' | 'last_index'),
      softcap (0 = off), smooth_softmax (bool).
    head_sink: None or float32 [heads] per-head sink logits.
    k_scale, v_scale: float32 scales when problem['kv_dtype'] == 'i8' (k and v are
      then int8 storage): one value (problem['kv_scale'] == 'tensor') or
      kv_heads * head_dim values ('channel').
    q, k, v: raw storage (float32 for f32, uint16 bit patterns for f16/bf16),
      indexed through the layouts.  mask: float32 storage; seg, k_lens: int32.
    rows: None for every (b, h, qi) row in that order, else an int array [n, 3].
    Returns (o [n_rows, head_dim], lse [n_rows]).
    """
    lib = _load()
    p = problem
    dt = p["dtype"]
    kv8 = p.get("kv_dtype") == "i8"
    q = _storage(q, dt)
    if kv8:
        if np.asarray(k).dtype != np.int8 or np.asarray(v).dtype != np.int8:
            raise TypeError("oracle expects int8 key/value storage for kv_dtype 'i8'")
        k, v = np.ascontiguousarray(k), np.ascontiguousarray(v)
    else:
        k, v = _storage(k, dt), _storage(v, dt)
    mask = None if mask is None else np.ascontiguousarray(mask, dtype=np.float32)
    seg = None if seg is None else np.ascontiguousarray(seg, dtype=np.int32)
    k_lens = None if k_lens is None else np.ascontiguousarray(k_lens, dtype=np.int32)
    prob = _Problem()
    prob.batch, prob.heads, prob.kv_heads = p["batch"], p["heads"], p["kv_heads"]
    prob.q_len, prob.k_len, prob.head_dim = p["q_len"], p["k_len"], p["head_dim"]
    prob.dtype = DTYPES[dt]
    prob.scale = float(p.get("scale", 0.0) or 0.0)
    prob.causal = 1 if p.get("causal") else 0
    off = p.get("causal_offset")
    prob.causal_offset = INT64_MIN if off is None else int(off)
    prob.masked_rows_zero = 1 if p.get("masked_rows", "nan") == "zero" else 0
    prob.q = _Layout(*p["q_layout"])
    prob.k = _Layout(*p["k_layout"])
    prob.v = _Layout(*p["v_layout"])
    prob.mask = _Layout(*(p.get("mask_layout") or (0, 0, 0, 0)))
    prob.seg_batch_stride = int(p.get("seg_batch_stride", p["q_len"]))
    w = p.get("window_left")
    prob.window_left = -1 if w is None else int(w)
    prob.causal_align = 1 if p.get("causal_align") in ("klens", 1) else 0
    prob.k_lens_kind = 1 if p.get("k_lens_kind") in ("last_index", 1) else 0
    prob.softcap = float(p.get("softcap") or 0.0)
    prob.smooth_softmax = 1 if p.get("smooth_softmax") else 0
    sink = None if head_sink is None else np.ascontiguousarray(head_sink, dtype=np.float32)
    if sink is not None and sink.shape != (p["heads"],):
        raise ValueError("head_sink must be float32 [heads]")
    prob.head_sink = None if sink is None else sink.ctypes.data
    prob.kv_int8 = 1 if kv8 else 0
    prob.kv_per_channel = 1 if p.get("kv_scale") == "channel" else 0
    scales = []
    if kv8:
        n_sc = p["kv_heads"] * p["head_dim"] if prob.kv_per_channel else 1
        for sc in (k_scale, v_scale):
            sc = np.ascontiguousarray(sc, dtype=np.float32).reshape(-1)
            if sc.size != n_sc:
                raise ValueError(f"expected {n_sc} scales, got {sc.size}")
            scales.append(sc)
        prob.k_scale, prob.v_scale = scales[0].ctypes.data, scales[1].ctypes.data
    if rows is None:
        n_rows = p["batch"] * p["heads"] * p["q_len"]
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
        n_rows = rows_arr.shape[0]
    o = np.empty((n_rows, p["head_dim"]), dtype=np.float64)
    lse = np.empty((n_rows,), dtype=np.float64)
    nt = default_threads() if nthreads is None else int(nthreads)
    rc = lib.orc_attn_rows(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(seg),
                           _ptr(k_lens), n_rows, _ptr(rows_arr), _ptr(o), _ptr(lse), nt)
    if rc != 0:
        raise ValueError(f"oracle rejected the problem (status {rc})")
    return o, lse


def append_rows(problem: dict, k_cache, v_cache, k_new, v_new, k_lens, k_scale=None, v_scale=None):
    """The cache update before a decode step: copies of the BNSH caches with each
    (batch, kv head)'s new row written at position L_b - 1 (see attn_oracle.c).
    k_new / v_new: [batch, kv_heads, head_dim] storage of the problem's dtype;
    caches: storage of the problem's dtype, or int8 when problem['kv_dtype'] == 'i8'.
    Returns (k_cache', v_cache')."""
    lib = _load()
    p = problem
    B, G, D, cap = p["batch"], p["kv_heads"], p["head_dim"], p["k_len"]
    kv8 = p.get("kv_dtype") == "i8"
    per_ch = 1 if p.get("kv_scale") == "channel" else 0
    plus = 1 if p.get("k_lens_kind") in ("last_index", 1) else 0
    k_lens = np.ascontiguousarray(k_lens, dtype=np.int32)
    out = []
    for cache, new, sc in ((k_cache, k_new, k_scale), (v_cache, v_new, v_scale)):
        c = np.array(cache, copy=True, order="C")
        n = _storage(np.ascontiguousarray(new), p["dtype"])
        lay = p["k_layout"]
        elem = 1 if kv8 else (4 if p["dtype"] == "f32" else 2)
        scale = None if sc is None else np.ascontiguousarray(sc, dtype=np.float32).reshape(-1)
        rc = lib.orc_append_rows(c.ctypes.data + lay[0] * elem, lay[1], lay[2], lay[3], cap, B, G, D, elem,
                                 n.ctypes.data, DTYPES[p["dtype"]], k_lens.ctypes.data, plus,
                                 None if scale is None else scale.ctypes.data, per_ch)
        if rc != 0:
            raise ValueError("oracle append rejected its arguments")
        out.append(c)
    return out[0], out[1]


def combine(part_o, part_lse, masked_rows="nan"):
    """Merge per-range partials: part_o [rows, n_splits, D] f32, part_lse [rows, n_splits] f32."""
    lib = _load()
    part_o = np.ascontiguousarray(part_o, dtype=np.float32)
    part_lse = np.ascontiguousarray(part_lse, dtype=np.float32)
    rows, n_splits, d = part_o.shape
    assert part_lse.shape == (rows, n_splits)
    o = np.empty((rows, d), dtype=np.float64)
    lse = np.empty((rows,), dtype=np.float64)
    rc = lib.orc_combine(n_splits, rows, d, _ptr(part_o), _ptr(part_lse),
                         1 if masked_rows == "zero" else 0, _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle combine rejected its arguments (status {rc})")
    return o, lse


def widen(dtype: str, bits: int) -> float:
    """The oracle's exact widening of one stored element to double."""
    return _load().orc_widen(DTYPES[dtype], bits)


def default_scale(head_dim: int) -> float:
    return _load().orc_default_scale(head_dim)
