"""Seeded synthetic inputs for attention problems.

This module only draws random numbers and lays them out in memory.  It holds
none of the attention arithmetic; the oracle and the CUDA path both read the
buffers it returns, and nothing else passes between them.

Recipe: every tensor comes from ``numpy.random.default_rng([seed, tensor_id])``
(Q = 0, K = 1, V = 2, mask = 3, segment/length draws = 4), drawn as float32
N(0, 1) (times a stated scale) and rounded to the element type with
round-to-nearest-even.  Keys that are structurally hidden from every query
row of their batch entry (beyond that entry's key length) are filled with NaN,
so any read of them shows up in the result.

A problem is described by a plain dict (the fields of the C ABI's problem
struct, layouts as (offset, batch_stride, head_stride, row_stride) tuples in
elements); the storage arrays are float32 for f32 and uint16 bit patterns for
f16/bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

Q_ID, K_ID, V_ID, MASK_ID, LEN_ID = 0, 1, 2, 3, 4

NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}


def rng(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.default_rng([seed, tensor_id])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns.

    Uses PyTorch's multithreaded CPU conversion when it is importable (the same
    rounding, checked bit for bit against the numpy form in the tests)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    try:
        import torch
    except ImportError:
        return f32_to_bf16_bits_numpy(x)
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f32_to_bf16_bits_numpy(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in = x.reshape(-1)
    flat_out = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_in.size, step):
        u = flat_in[s:s + step].view(np.uint32)
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        r = r.astype(np.uint16)
        nan = np.isnan(flat_in[s:s + step])
        r[nan] = 0x7FC0
        flat_out[s:s + step] = r
    return out


def to_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(x32.astype(np.float16)).view(np.uint16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    raise ValueError(dtype)


def normal(seed: int, tensor_id: int, shape, scale: float = 1.0) -> np.ndarray:
    x = rng(seed, tensor_id).standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def layout_of(kind: str, B: int, H: int, S: int, D: int):
    """(shape of the storage tensor, layout tuple) for a contiguous BSHD or BHSD tensor."""
    if kind == "bshd":     # position-first
        return (B, S, H, D), (0, S * H * D, D, H * D)
    if kind == "bhsd":     # head-first
        return (B, H, S, D), (0, H * S * D, S * D, D)
    raise ValueError(kind)


@dataclass
class Case:
    name: str
    problem: dict
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    o_shape: tuple
    mask: np.ndarray | None = None
    seg: np.ndarray | None = None
    k_lens: np.ndarray | None = None
    head_sink: np.ndarray | None = None
    k_scale: np.ndarray | None = None
    v_scale: np.ndarray | None = None
    decode: bool = False
    meta: dict = field(default_factory=dict)


def doc_starts(seed: int, batch: int, seq: int, lo: int = 64, hi: int = 512) -> np.ndarray:
    """Per-token document start: document lengths drawn uniform in [lo, hi] until they cover seq."""
    r = rng(seed, LEN_ID)
    seg = np.zeros((batch, seq), dtype=np.int32)
    for b in range(batch):
        pos = 0
        while pos < seq:
            n = int(r.integers(lo, hi + 1))
            seg[b, pos:min(seq, pos + n)] = pos
            pos += n
    return seg


def make_case(*, name="case", seed=0, dtype="bf16", layout="bshd", batch=1, heads=2, kv_heads=None,
              q_len=16, k_len=None, head_dim=32, causal=False, causal_offset=None, scale=0.0,
              masked_rows="nan", value_scale=1.0, k_lens=None, seg=None, mask=None,
              mask_kind="b11k", nan_fill=True, packed=False, decode=False, window_left=None,
              causal_align="fixed", k_lens_kind="count", softcap=0.0, smooth_softmax=False,
              head_sink=None, kv_dtype=None, kv_scale="channel") -> Case:
    """A general seeded problem.

    k_lens / seg / mask may be arrays (used as given) or None.  window_left,
    causal_align and k_lens_kind are the visibility variants of the problem
    (k_lens holds the values as passed: count - 1 under 'last_index').
    kv_dtype='i8' stores K and V as int8 (uniform in [-127, 127]; rows beyond a
    batch entry's length are -128) with float32 scales per (kv head, channel)
    ('channel', uniform in [0.005, 0.02]) or one per cache ('tensor').  mask_kind names
    the broadcast shape of a given mask: 'b11k' [B,1,1,K], 'bhqk' [B,H,Q,K],
    '11qk' [1,1,Q,K].  packed=True stores Q, K and V as slices of one
    [B, S, H + 2*KVH, D] projection (q_len must equal k_len).  decode=True
    stores K/V as a BNSH cache of capacity k_len and Q as [B, 1, H, D].
    """
    kv_heads = heads if kv_heads is None else kv_heads
    k_len = q_len if k_len is None else k_len
    B, H, G, Sq, Sk, D = batch, heads, kv_heads, q_len, k_len, head_dim
    qx = normal(seed, Q_ID, (B, Sq, H, D) if layout == "bshd" or packed else (B, H, Sq, D), value_scale)
    if decode:
        kshape = vshape = (B, G, Sk, D)
        kv_kind = "bhsd"
    else:
        kv_kind = layout
        kshape = vshape = (B, Sk, G, D) if layout == "bshd" or packed else (B, G, Sk, D)
    kx = normal(seed, K_ID, kshape, value_scale)
    vx = normal(seed, V_ID, vshape, value_scale)
    if k_lens is not None:
        k_lens = np.asarray(k_lens, dtype=np.int32)
        if nan_fill:
            for b in range(B):
                kl = int(min(max(int(k_lens[b]) + (1 if k_lens_kind == "last_index" else 0), 0), Sk))
                if kv_kind == "bshd" or packed:
                    kx[b, kl:] = np.nan
                    vx[b, kl:] = np.nan
                else:
                    kx[b, :, kl:] = np.nan
                    vx[b, :, kl:] = np.nan
    prob = dict(batch=B, heads=H, kv_heads=G, q_len=Sq, k_len=Sk, head_dim=D, dtype=dtype,
                scale=float(scale), causal=bool(causal), causal_offset=causal_offset,
                masked_rows=masked_rows, window_left=window_left, causal_align=causal_align,
                k_lens_kind=k_lens_kind, softcap=float(softcap), smooth_softmax=bool(smooth_softmax))
    if packed:
        assert Sq == Sk and not decode
        W = H + 2 * G
        buf = np.empty((B, Sq, W, D), dtype=np.float32)
        buf[:, :, :H] = qx
        buf[:, :, H:H + G] = kx
        buf[:, :, H + G:] = vx
        st = to_storage(buf, dtype)
        q = k = v = st
        rs, bs = W * D, Sq * W * D
        prob["q_layout"] = (0, bs, D, rs)
        prob["k_layout"] = (H * D, bs, D, rs)
        prob["v_layout"] = (H * D + G * D, bs, D, rs)
    else:
        q, k, v = to_storage(qx, dtype), to_storage(kx, dtype), to_storage(vx, dtype)
        prob["q_layout"] = layout_of("bshd" if (layout == "bshd" or decode) else "bhsd", B, H, Sq, D)[1]
        prob["k_layout"] = layout_of(kv_kind, B, G, Sk, D)[1]
        prob["v_layout"] = layout_of(kv_kind, B, G, Sk, D)[1]
    o_kind = "bshd" if (layout == "bshd" or packed or decode) else "bhsd"
    o_shape, o_layout = layout_of(o_kind, B, H, Sq, D)
    prob["o_layout"] = o_layout
    prob["o_kind"] = o_kind
    if mask is not None:
        mask = np.ascontiguousarray(mask, dtype=np.float32)
        if mask_kind == "b11k":
            prob["mask_layout"] = (0, Sk, 0, 0)
        elif mask_kind == "bhqk":
            prob["mask_layout"] = (0, H * Sq * Sk, Sq * Sk, Sk)
        elif mask_kind == "11qk":
            prob["mask_layout"] = (0, 0, 0, Sk)
        else:
            raise ValueError(mask_kind)
    if seg is not None:
        seg = np.ascontiguousarray(seg, dtype=np.int32)
        prob["seg_batch_stride"] = 0 if seg.ndim == 1 else Sq
    prob["lse_layout"] = (H * Sq, Sq)   # LSE [B, H, q_len] float32
    if head_sink is not None:
        head_sink = np.ascontiguousarray(head_sink, dtype=np.float32)
    k_scale = v_scale = None
    if kv_dtype == "i8":
        assert not packed
        r8 = rng(seed, K_ID + 10)
        k = r8.integers(-127, 128, size=kshape, dtype=np.int8)
        v = r8.integers(-127, 128, size=vshape, dtype=np.int8)
        if k_lens is not None and nan_fill:
            for b in range(B):
                kl = int(min(max(int(k_lens[b]) + (1 if k_lens_kind == "last_index" else 0), 0), Sk))
                if kv_kind == "bshd":
                    k[b, kl:] = -128
                    v[b, kl:] = -128
                else:
                    k[b, :, kl:] = -128
                    v[b, :, kl:] = -128
        n_sc = G * D if kv_scale == "channel" else 1
        k_scale = r8.uniform(0.005, 0.02, size=n_sc).astype(np.float32)
        v_scale = r8.uniform(0.005, 0.02, size=n_sc).astype(np.float32)
        prob["kv_dtype"] = "i8"
        prob["kv_scale"] = kv_scale
    return Case(name=name, problem=prob, q=q, k=k, v=v, o_shape=o_shape, mask=mask, seg=seg,
                k_lens=k_lens, head_sink=head_sink, k_scale=k_scale, v_scale=v_scale, decode=decode)


# ---- the five named workloads -------------------------------------------------


def tiny_f32_mha(seed: int = 1) -> Case:
    """float32 MHA, batch 1, 2 heads, 64 queries and keys, head dim 32, position-first, no mask."""
    return make_case(name="tiny_f32_mha_b1_h2_s64_d32", seed=seed, dtype="f32", layout="bshd",
                     batch=1, heads=2, q_len=64, head_dim=32)


def gqa_doc_causal_bf16(seed: int = 2, batch: int = 4, seq: int = 1024) -> Case:
    """Causal GQA training forward with per-document segments: 12 heads over 4 KV heads, head dim 64."""
    seg = doc_starts(seed, batch, seq)
    return make_case(name=f"gqa_doc_causal_bf16_b{batch}_h12_kv4_s{seq}_d64", seed=seed, dtype="bf16",
                     layout="bshd", batch=batch, heads=12, kv_heads=4, q_len=seq, head_dim=64,
                     causal=True, causal_offset=0, scale=1.0 / 8.0, seg=seg)


def long_causal_gqa_bf16(seed: int = 3, batch: int = 2, seq: int = 4096, heads: int = 32,
                         kv_heads: int = 8) -> Case:
    """Long causal GQA prefill, head-first, head dim 128, per-batch key lengths in [seq/2, seq]."""
    r = rng(seed, LEN_ID)
    k_lens = r.integers(seq // 2, seq + 1, size=batch).astype(np.int32)
    return make_case(name=f"long_causal_gqa_bf16_b{batch}_h{heads}_kv{kv_heads}_s{seq}_d128", seed=seed,
                     dtype="bf16", layout="bhsd", batch=batch, heads=heads, kv_heads=kv_heads,
                     q_len=seq, head_dim=128, causal=True, causal_offset=None, value_scale=0.5,
                     k_lens=k_lens)


def dense_gqa_bf16(seed: int = 3, batch: int = 2, seq: int = 4096, heads: int = 32, kv_heads: int = 8) -> Case:
    """The long GQA prefill's shape without the causal bound or key lengths: every query sees every key
    (a context measurement of the tensor-core kernel's steady state)."""
    return make_case(name=f"dense_gqa_bf16_b{batch}_h{heads}_kv{kv_heads}_s{seq}_d128", seed=seed, dtype="bf16",
                     layout="bhsd", batch=batch, heads=heads, kv_heads=kv_heads, q_len=seq, head_dim=128,
                     causal=False, causal_offset=None, value_scale=0.5)


def masked_gqa_bf16(seed: int = 3, batch: int = 2, seq: int = 4096, heads: int = 32, kv_heads: int = 8) -> Case:
    """The long GQA prefill's shapes with a float32 padding mask [B,1,1,K] instead of the causal bound:
    N(0,1) values, the last key_len/8 keys of each batch entry -inf (a context measurement of the masked
    score path)."""
    r = rng(seed, MASK_ID)
    mask = r.standard_normal((batch, 1, 1, seq)).astype(np.float32)
    mask[:, :, :, seq - seq // 8:] = -np.inf
    return make_case(name=f"masked_gqa_bf16_b{batch}_h{heads}_kv{kv_heads}_s{seq}_d128", seed=seed, dtype="bf16",
                     layout="bhsd", batch=batch, heads=heads, kv_heads=kv_heads, q_len=seq, head_dim=128,
                     causal=False, causal_offset=None, value_scale=0.5, mask=mask, mask_kind="b11k")


def rowmask_gqa_bf16(seed: int = 7, batch: int = 2, seq: int = 4096, heads: int = 32, kv_heads: int = 8) -> Case:
    """The long GQA prefill's shapes with a float32 mask of one row per query, shared by every batch entry
    and head ([1,1,Q,K], 64 MiB): N(0,1) values, the last key_len/8 keys -inf (a context measurement of the
    per-row mask path)."""
    r = rng(seed, MASK_ID)
    mask = r.standard_normal((1, 1, seq, seq)).astype(np.float32)
    mask[:, :, :, seq - seq // 8:] = -np.inf
    return make_case(name=f"rowmask_gqa_bf16_b{batch}_h{heads}_kv{kv_heads}_s{seq}_d128", seed=seed, dtype="bf16",
                     layout="bhsd", batch=batch, heads=heads, kv_heads=kv_heads, q_len=seq, head_dim=128,
                     causal=False, causal_offset=None, value_scale=0.5, mask=mask, mask_kind="11qk")


def short_query_cross_bf16(seed: int = 6, batch: int = 1, heads: int = 32, kv_heads: int = 8, q_len: int = 64,
                           k_len: int = 8192) -> Case:
    """A few queries against a long key axis (bf16, head dim 128, head-first, non-causal): too few blocks
    of query rows to fill the GPU, so the keys are cut into ranges (a context measurement of the split)."""
    return make_case(name=f"short_query_cross_bf16_b{batch}_h{heads}_kv{kv_heads}_q{q_len}_k{k_len}_d128",
                     seed=seed, dtype="bf16", layout="bhsd", batch=batch, heads=heads, kv_heads=kv_heads,
                     q_len=q_len, k_len=k_len, head_dim=128, value_scale=0.5)


def decode_bnsh_bf16(seed: int = 4, batch: int = 64, capacity: int = 8192, heads: int = 32,
                     kv_heads: int = 8, min_len: int = 512) -> Case:
    """Batched single-query decode over a BNSH cache [B, 8, capacity, 128], lengths uniform in [512, capacity]."""
    r = rng(seed, LEN_ID)
    k_lens = r.integers(min_len, capacity + 1, size=batch).astype(np.int32)
    return make_case(name=f"decode_bnsh_bf16_b{batch}_h{heads}_kv{kv_heads}_cap{capacity}_d128", seed=seed,
                     dtype="bf16", batch=batch, heads=heads, kv_heads=kv_heads, q_len=1, k_len=capacity,
                     head_dim=128, k_lens=k_lens, decode=True)


def decode_bnsh_int8(seed: int = 4, batch: int = 64, capacity: int = 8192, heads: int = 32,
                     kv_heads: int = 8, min_len: int = 512) -> Case:
    """The batched decode workload with an int8 BNSH cache and per-(kv head, channel) scales
    (bf16 queries): the same lengths as decode_bnsh_bf16, half the cache bytes."""
    r = rng(seed, LEN_ID)
    k_lens = r.integers(min_len, capacity + 1, size=batch).astype(np.int32)
    return make_case(name=f"decode_bnsh_int8_b{batch}_h{heads}_kv{kv_heads}_cap{capacity}_d128", seed=seed,
                     dtype="bf16", batch=batch, heads=heads, kv_heads=kv_heads, q_len=1, k_len=capacity,
                     head_dim=128, k_lens=k_lens, decode=True, kv_dtype="i8", kv_scale="channel")


def cross_mask_f16(seed: int = 5, batch: int = 8, q_len: int = 512, k_len: int = 2048, heads: int = 16,
                   masked_rows: str = "nan") -> Case:
    """fp16 cross-attention, head dim 256, additive float32 mask [B,1,1,K]: N(0,1), 10% of keys -inf,
    the last batch entry fully -inf."""
    r = rng(seed, MASK_ID)
    mask = r.standard_normal((batch, 1, 1, k_len)).astype(np.float32)
    n_hidden = int(math.floor(0.1 * k_len))
    for b in range(batch):
        idx = r.choice(k_len, size=n_hidden, replace=False)
        mask[b, 0, 0, idx] = -np.inf
    mask[batch - 1] = -np.inf
    return make_case(name=f"cross_mask_f16_b{batch}_h{heads}_q{q_len}_k{k_len}_d256_{masked_rows}",
                     seed=seed, dtype="f16", layout="bshd", batch=batch, heads=heads, q_len=q_len,
                     k_len=k_len, head_dim=256, scale=1.0 / 16.0, mask=mask, mask_kind="b11k",
                     masked_rows=masked_rows)


def visible_pairs(case: Case) -> int:
    """Exact count of structurally visible (query, key) pairs with a finite mask, summed over (b, h).

    Work measure only (4 * head_dim flops per pair); no attention arithmetic.
    """
    p = case.problem
    B, H, Sq, Sk = p["batch"], p["heads"], p["q_len"], p["k_len"]
    off = p["causal_offset"] if p["causal_offset"] is not None else Sk - Sq
    plus = 1 if p.get("k_lens_kind") == "last_index" else 0
    w = p.get("window_left")
    total = 0
    qi = np.arange(Sq, dtype=np.int64)
    for b in range(B):
        kl = Sk if case.k_lens is None else min(max(int(case.k_lens[b]) + plus, 0), Sk)
        hi = np.full(Sq, kl, dtype=np.int64)
        lo = np.zeros(Sq, dtype=np.int64)
        if p["causal"]:
            diag = qi + (kl - Sq if p.get("causal_align") == "klens" else off)
            hi = np.minimum(hi, np.maximum(diag + 1, 0))
            if w is not None and w >= 0:
                lo = np.maximum(lo, diag - w)
        if case.seg is not None:
            s = case.seg if case.seg.ndim == 1 else case.seg[b]
            lo = np.maximum(lo, np.clip(s.astype(np.int64), 0, Sk))
        if case.mask is None:
            total += H * int(np.maximum(hi - lo, 0).sum())
            continue
        ml = p["mask_layout"]
        flat = case.mask.reshape(-1)
        finite = np.isfinite(flat)
        for h in range(H):
            for q in range(Sq):
                base = ml[0] + b * ml[1] + h * ml[2] + q * ml[3]
                if hi[q] > lo[q]:
                    total += int(finite[base + lo[q]: base + hi[q]].sum())
    return total
