"""ctypes binding of libattn.so (include/attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  The low-level functions keep the C names (attn_fwd, attn_decode,
attn_combine, ...) and take integer device addresses; ``fwd``, ``decode`` and
``combine`` build the problem struct from torch tensors, allocate the outputs
and the workspace with torch, and call them on torch's current stream.
There is no CPU fallback: if the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn.so")

ATTN_F32, ATTN_F16, ATTN_BF16 = 0, 1, 2
ATTN_MASKED_ROWS_NAN, ATTN_MASKED_ROWS_ZERO = 0, 1
ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_ALIGNMENT = 0, 1, 2, 3
ATTN_ERR_WORKSPACE, ATTN_ERR_CUDA, ATTN_ERR_DEVICE_TIMEOUT = 4, 5, 6
ATTN_OFFSET_DEFAULT = -(2**63)
ATTN_CAUSAL_FIXED, ATTN_CAUSAL_KLENS = 0, 1
ATTN_KLENS_COUNT, ATTN_KLENS_LAST_INDEX = 0, 1
ATTN_KV_AS_Q, ATTN_KV_INT8 = 0, 1
ATTN_KV_SCALE_TENSOR, ATTN_KV_SCALE_CHANNEL = 0, 1
ATTN_INJECT_NONE, ATTN_INJECT_DROP_FIRST_COPY = 0, 1
DTYPE_CODE = {"f32": ATTN_F32, "f16": ATTN_F16, "bf16": ATTN_BF16}
EXPORTS = ("attn_fwd_workspace_size", "attn_fwd", "attn_decode_workspace_size", "attn_decode", "attn_combine",
           "attn_device_status", "attn_status_string", "attn_version", "attn_decode_noalloc",
           "attn_decode_noalloc_max_scratch", "attn_decode_append", "attn_probe_ex2", "attn_test_inject")


class attn_layout(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_int64), ("batch_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64), ("row_stride", ctypes.c_int64)]


class attn_problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("q_len", ctypes.c_int32), ("k_len", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float), ("causal", ctypes.c_int32),
                ("causal_offset", ctypes.c_int64), ("masked_rows", ctypes.c_int32),
                ("q", attn_layout), ("k", attn_layout), ("v", attn_layout), ("o", attn_layout),
                ("mask", attn_layout), ("seg_batch_stride", ctypes.c_int64),
                ("lse_batch_stride", ctypes.c_int64), ("lse_head_stride", ctypes.c_int64),
                ("window_left", ctypes.c_int32), ("causal_align", ctypes.c_int32),
                ("k_lens_kind", ctypes.c_int32), ("softcap", ctypes.c_float),
                ("smooth_softmax", ctypes.c_int32), ("head_sink", ctypes.c_void_p),
                ("kv_dtype", ctypes.c_int32), ("kv_scale_kind", ctypes.c_int32),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("key_splits", ctypes.c_int32)]


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (status {code})")
        self.code = code


_lib = None


def lib():
    """Load libattn.so (raises when it has not been built: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m attention_attn_fwd_02_gb300.build`"
                               " (or __graft_entry__.build()); there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(attn_problem)
        vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
        L.attn_fwd_workspace_size.argtypes, L.attn_fwd_workspace_size.restype = [P], sz
        L.attn_decode_workspace_size.argtypes, L.attn_decode_workspace_size.restype = [P], sz
        L.attn_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.attn_fwd.restype = ctypes.c_int
        L.attn_decode.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.attn_decode.restype = ctypes.c_int
        L.attn_combine.argtypes = [i32, i32, i32, vp, vp, i32, vp, i64, vp, i32, vp]
        L.attn_combine.restype = ctypes.c_int
        L.attn_device_status.argtypes, L.attn_device_status.restype = [vp], ctypes.c_int
        L.attn_status_string.argtypes, L.attn_status_string.restype = [ctypes.c_int], ctypes.c_char_p
        L.attn_version.argtypes, L.attn_version.restype = [], ctypes.c_int
        L.attn_decode_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.attn_decode_noalloc.restype = ctypes.c_int
        L.attn_decode_noalloc_max_scratch.argtypes, L.attn_decode_noalloc_max_scratch.restype = [], sz
        L.attn_decode_append.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.attn_decode_append.restype = ctypes.c_int
        L.attn_probe_ex2.argtypes, L.attn_probe_ex2.restype = [i32, i32, vp, vp], ctypes.c_int
        L.attn_test_inject.argtypes, L.attn_test_inject.restype = [i32], ctypes.c_int
        _lib = L
    return _lib


# ---- the C entry points, same names ---------------------------------------------


def attn_fwd_workspace_size(p: attn_problem) -> int:
    return lib().attn_fwd_workspace_size(ctypes.byref(p))


def attn_decode_workspace_size(p: attn_problem) -> int:
    return lib().attn_decode_workspace_size(ctypes.byref(p))


def attn_fwd(p, q, k, v, o, mask, seg, k_lens, lse, workspace, workspace_bytes, stream) -> int:
    return lib().attn_fwd(ctypes.byref(p), q, k, v, o, mask, seg, k_lens, lse, workspace, workspace_bytes, stream)


def attn_decode(p, q, k_cache, v_cache, o, mask, seg, k_lens, lse, workspace, workspace_bytes, stream) -> int:
    return lib().attn_decode(ctypes.byref(p), q, k_cache, v_cache, o, mask, seg, k_lens, lse, workspace,
                             workspace_bytes, stream)


def attn_decode_noalloc(p, q, k_cache, v_cache, o, mask, seg, k_lens, lse, stream) -> int:
    """attn_decode with the library's fixed device scratch array instead of a caller workspace,
    for callers that cannot allocate device memory (see include/attn.h)."""
    return lib().attn_decode_noalloc(ctypes.byref(p), q, k_cache, v_cache, o, mask, seg, k_lens, lse, stream)


def attn_decode_append(p, q, k_new, v_new, k_cache, v_cache, o, mask, k_lens, lse, workspace, workspace_bytes,
                       stream) -> int:
    return lib().attn_decode_append(ctypes.byref(p), q, k_new, v_new, k_cache, v_cache, o, mask, k_lens, lse,
                                    workspace, workspace_bytes, stream)


def attn_probe_ex2(blocks, iters, sink, stream) -> int:
    """Launch the exponential-throughput micro-kernel (a measurement utility; see include/attn.h)."""
    return lib().attn_probe_ex2(blocks, iters, sink, stream)


def attn_test_inject(fault: int) -> int:
    """Arm the one-shot bounded-wait test fault (a test utility; see include/attn.h)."""
    return lib().attn_test_inject(fault)


def attn_decode_noalloc_max_scratch() -> int:
    return lib().attn_decode_noalloc_max_scratch()


def attn_combine(n_splits, rows, head_dim, part_o, part_lse, out_dtype, o, o_row_stride, lse, masked_rows,
                 stream) -> int:
    return lib().attn_combine(n_splits, rows, head_dim, part_o, part_lse, out_dtype, o, o_row_stride, lse,
                              masked_rows, stream)


def attn_device_status(stream=None) -> int:
    return lib().attn_device_status(stream)


def status_string(code: int) -> str:
    try:
        return lib().attn_status_string(code).decode()
    except RuntimeError:
        return f"status {code}"


def attn_version() -> int:
    return lib().attn_version()


# ---- problem construction ---------------------------------------------------------


def make_problem(d: dict) -> attn_problem:
    """attn_problem from a plain dict (the fields of the struct; layouts as 4-tuples)."""
    p = attn_problem()
    p.batch, p.heads, p.kv_heads = d["batch"], d["heads"], d["kv_heads"]
    p.q_len, p.k_len, p.head_dim = d["q_len"], d["k_len"], d["head_dim"]
    p.dtype = DTYPE_CODE[d["dtype"]] if isinstance(d["dtype"], str) else int(d["dtype"])
    p.scale = float(d.get("scale") or 0.0)
    p.causal = 1 if d.get("causal") else 0
    off = d.get("causal_offset")
    p.causal_offset = ATTN_OFFSET_DEFAULT if off is None else int(off)
    mr = d.get("masked_rows", "nan")
    p.masked_rows = ATTN_MASKED_ROWS_ZERO if mr in ("zero", ATTN_MASKED_ROWS_ZERO) else ATTN_MASKED_ROWS_NAN
    for name in ("q", "k", "v", "o"):
        setattr(p, name, attn_layout(*d[f"{name}_layout"]))
    p.mask = attn_layout(*(d.get("mask_layout") or (0, 0, 0, 0)))
    p.seg_batch_stride = int(d.get("seg_batch_stride", d["q_len"]))
    lb, lh = d.get("lse_layout") or (d["heads"] * d["q_len"], d["q_len"])
    p.lse_batch_stride, p.lse_head_stride = lb, lh
    w = d.get("window_left")
    p.window_left = -1 if w is None else int(w)
    p.causal_align = ATTN_CAUSAL_KLENS if d.get("causal_align") in ("klens", ATTN_CAUSAL_KLENS) else ATTN_CAUSAL_FIXED
    p.k_lens_kind = (ATTN_KLENS_LAST_INDEX if d.get("k_lens_kind") in ("last_index", ATTN_KLENS_LAST_INDEX)
                     else ATTN_KLENS_COUNT)
    p.softcap = float(d.get("softcap") or 0.0)
    p.smooth_softmax = 1 if d.get("smooth_softmax") else 0
    p.head_sink = d.get("head_sink_ptr")      # device address of float32 [heads], or None
    p.kv_dtype = ATTN_KV_INT8 if d.get("kv_dtype") in ("i8", ATTN_KV_INT8) else ATTN_KV_AS_Q
    p.kv_scale_kind = (ATTN_KV_SCALE_CHANNEL if d.get("kv_scale") in ("channel", ATTN_KV_SCALE_CHANNEL)
                       else ATTN_KV_SCALE_TENSOR)
    p.k_scale = d.get("k_scale_ptr")          # device addresses of float32 scales (int8 caches)
    p.v_scale = d.get("v_scale_ptr")
    p.key_splits = int(d.get("key_splits") or 0)   # attn_fwd key ranges: 0 = the library's plan
    return p


def _ptr(t):
    return None if t is None else t.data_ptr()


def _torch():
    import torch
    return torch


def _dtype_name(t):
    torch = _torch()
    return {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[t.dtype]


def _layout4(t, heads_dim: int):
    """(offset, batch, head, row) strides of a 4-D tensor whose dims are [B, S, H, D] (heads_dim=2)
    or [B, H, S, D] (heads_dim=1); offset 0 relative to data_ptr()."""
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("expected a 4-D tensor with contiguous last dimension")
    if heads_dim == 2:
        return (0, t.stride(0), t.stride(2), t.stride(1))
    return (0, t.stride(0), t.stride(1), t.stride(2))


def _check(code, where):
    if code != ATTN_OK:
        raise AttnError(code, where)


def fwd(q, k, v, *, layout="bshd", causal=False, causal_offset=None, scale=0.0, mask=None, seg=None,
        k_lens=None, masked_rows="nan", return_lse=False, out=None, lse=None, stream=None,
        window_left=None, causal_align="fixed", k_lens_kind="count", softcap=0.0, smooth_softmax=False,
        head_sink=None, key_splits=0):
    """O (and LSE) for torch CUDA tensors.  layout 'bshd': Q [B,Sq,H,D], K/V [B,Sk,G,D];
    'bhsd': Q [B,H,Sq,D], K/V [B,G,Sk,D].  mask: float32 broadcastable 4-D [B|1, H|1, Sq|1, Sk]
    with contiguous keys; seg: int32 [B, Sq] or [Sq]; k_lens: int32 [B].  window_left: left
    window of causal local attention (None = off); causal_align: 'fixed' (one offset) or
    'klens' (each entry's diagonal right-aligned to its key length); k_lens_kind: 'count' or
    'last_index' (ONNX seqlens_k, count minus one).  softcap: cap of the scaled scores (0 = off);
    smooth_softmax / head_sink (float32 [H] CUDA tensor): the sink term of the denominator.
    key_splits: key ranges merged in range order (0 = the library's shape-only plan)."""
    torch = _torch()
    hd = 2 if layout == "bshd" else 1
    sd = 1 if layout == "bshd" else 2
    B, Sq, H, D = q.shape[0], q.shape[sd], q.shape[hd], q.shape[3]
    G, Sk = k.shape[hd], k.shape[sd]
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    d = dict(batch=B, heads=H, kv_heads=G, q_len=Sq, k_len=Sk, head_dim=D, dtype=_dtype_name(q), scale=scale,
             causal=causal, causal_offset=causal_offset, masked_rows=masked_rows,
             q_layout=_layout4(q, hd), k_layout=_layout4(k, hd), v_layout=_layout4(v, hd),
             o_layout=_layout4(out, hd), window_left=window_left, causal_align=causal_align,
             k_lens_kind=k_lens_kind, softcap=softcap, smooth_softmax=smooth_softmax,
             head_sink_ptr=_ptr(head_sink), key_splits=key_splits)
    if mask is not None:
        if mask.dtype != torch.float32 or mask.dim() != 4 or mask.stride(3) != 1:
            raise ValueError("mask must be float32, 4-D, keys contiguous")
        d["mask_layout"] = (0, mask.stride(0) if mask.shape[0] > 1 else 0,
                            mask.stride(1) if mask.shape[1] > 1 else 0, mask.stride(2) if mask.shape[2] > 1 else 0)
    if seg is not None:
        d["seg_batch_stride"] = 0 if seg.dim() == 1 else seg.stride(0)
    if return_lse and lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if lse is not None:
        d["lse_layout"] = (lse.stride(0), lse.stride(1))
    p = make_problem(d)
    ws_bytes = attn_fwd_workspace_size(p)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
    st = torch.cuda.current_stream(q.device).cuda_stream if stream is None else stream
    _check(attn_fwd(p, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(mask), _ptr(seg), _ptr(k_lens), _ptr(lse),
                    _ptr(ws), ws_bytes, st), "attn_fwd")
    return (out, lse) if return_lse else out


def decode(q, k_cache, v_cache, k_lens=None, *, scale=0.0, mask=None, masked_rows="nan", return_lse=False,
           out=None, lse=None, workspace=None, stream=None, window_left=None, k_lens_kind="count", softcap=0.0,
           smooth_softmax=False, head_sink=None, k_scale=None, v_scale=None):
    """Single-query decode: q [B, 1, H, D]; caches BNSH [B, G, cap, D]; k_lens int32 [B].
    window_left keeps only the last window_left + 1 valid keys (local attention);
    k_lens_kind 'last_index' takes ONNX seqlens_k (count minus one) as given.
    int8 caches take float32 k_scale / v_scale tensors of 1 (per cache) or
    G * D (per kv head and channel) elements."""
    torch = _torch()
    B, Sq, H, D = q.shape
    G, cap = k_cache.shape[1], k_cache.shape[2]
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    d = dict(batch=B, heads=H, kv_heads=G, q_len=Sq, k_len=cap, head_dim=D, dtype=_dtype_name(q), scale=scale,
             causal=window_left is not None, causal_align="klens", window_left=window_left,
             k_lens_kind=k_lens_kind, softcap=softcap, smooth_softmax=smooth_softmax,
             head_sink_ptr=_ptr(head_sink), masked_rows=masked_rows, q_layout=_layout4(q, 2),
             kv_dtype="i8" if k_cache.dtype == torch.int8 else None,
             kv_scale="channel" if (k_scale is not None and k_scale.numel() > 1) else "tensor",
             k_scale_ptr=_ptr(k_scale), v_scale_ptr=_ptr(v_scale),
             k_layout=_layout4(k_cache, 1), v_layout=_layout4(v_cache, 1), o_layout=_layout4(out, 2))
    if mask is not None:
        d["mask_layout"] = (0, mask.stride(0) if mask.shape[0] > 1 else 0,
                            mask.stride(1) if mask.shape[1] > 1 else 0, mask.stride(2) if mask.shape[2] > 1 else 0)
    if return_lse and lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if lse is not None:
        d["lse_layout"] = (lse.stride(0), lse.stride(1))
    p = make_problem(d)
    ws_bytes = attn_decode_workspace_size(p)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = torch.cuda.current_stream(q.device).cuda_stream if stream is None else stream
    _check(attn_decode(p, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(mask), None, _ptr(k_lens),
                       _ptr(lse), _ptr(workspace), workspace.numel(), st), "attn_decode")
    return (out, lse) if return_lse else out


def combine(part_o, part_lse, *, out_dtype=None, masked_rows="nan", return_lse=False, stream=None):
    """Merge partials: part_o float32 [rows, n_splits, D], part_lse float32 [rows, n_splits]."""
    torch = _torch()
    rows, n, D = part_o.shape
    out_dtype = out_dtype or torch.float32
    out = torch.empty((rows, D), dtype=out_dtype, device=part_o.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=part_o.device) if return_lse else None
    st = torch.cuda.current_stream(part_o.device).cuda_stream if stream is None else stream
    code = {torch.float32: ATTN_F32, torch.float16: ATTN_F16, torch.bfloat16: ATTN_BF16}[out_dtype]
    _check(attn_combine(n, rows, D, _ptr(part_o), _ptr(part_lse), code, _ptr(out), D, _ptr(lse),
                        ATTN_MASKED_ROWS_ZERO if masked_rows == "zero" else ATTN_MASKED_ROWS_NAN, st),
           "attn_combine")
    return (out, lse) if return_lse else out
