"""Helpers shared by the tests: exact widening with numpy, canonical <-> strided
storage, and the comparison rules.  Nothing here computes attention."""
from __future__ import annotations

import numpy as np

from attention_attn_fwd_02_gb300 import workloads as wl


def widen(storage: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of stored elements (numpy's own conversions)."""
    if dtype == "f32":
        return storage.astype(np.float64)
    if dtype == "f16":
        return storage.view(np.float16).astype(np.float64)
    u = storage.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def representable(x64: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the element type and return them widened back (exact values)."""
    return widen(wl.to_storage(x64.astype(np.float32), dtype), dtype)


def canonical_problem(Qc, Kc, Vc, dtype, layout="bhsd", **kw):
    """Storage + problem dict for canonical Q [B,H,Sq,D], K/V [B,G,Sk,D] (values already representable)."""
    B, H, Sq, D = Qc.shape
    G, Sk = Kc.shape[1], Kc.shape[2]
    if layout == "bhsd":
        qs, ks, vs = Qc, Kc, Vc
    else:
        qs, ks, vs = (np.ascontiguousarray(x.transpose(0, 2, 1, 3)) for x in (Qc, Kc, Vc))
    prob = dict(batch=B, heads=H, kv_heads=G, q_len=Sq, k_len=Sk, head_dim=D, dtype=dtype,
                scale=kw.get("scale", 0.0), causal=kw.get("causal", False),
                causal_offset=kw.get("causal_offset"), masked_rows=kw.get("masked_rows", "nan"),
                q_layout=wl.layout_of(layout, B, H, Sq, D)[1],
                k_layout=wl.layout_of(layout, B, G, Sk, D)[1],
                v_layout=wl.layout_of(layout, B, G, Sk, D)[1],
                mask_layout=kw.get("mask_layout"), seg_batch_stride=kw.get("seg_batch_stride", Sq))
    conv = (lambda x: wl.to_storage(x.astype(np.float32), dtype))
    return prob, conv(qs), conv(ks), conv(vs)


def brute_force(Qc, Kc, Vc, scale, visible, mask=None):
    """Materialise every score with an explicit visibility test and take the
    softmax without subtracting a maximum (tiny, moderate scores only).

    visible(b, q, k) -> bool; mask(b, h, q, k) -> float or None.  Returns
    O [B,H,Sq,D] and LSE [B,H,Sq] with NaN rows for no visible key (LSE -inf).
    """
    B, H, Sq, D = Qc.shape
    G, Sk = Kc.shape[1], Kc.shape[2]
    grp = H // G
    O = np.zeros((B, H, Sq, D))
    L = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            g = h // grp
            for q in range(Sq):
                w = []
                for k in range(Sk):
                    if not visible(b, q, k):
                        continue
                    s = scale * float(np.dot(Qc[b, h, q], Kc[b, g, k]))
                    if mask is not None:
                        s += mask(b, h, q, k)
                    if s == -np.inf:
                        continue
                    w.append((np.exp(np.longdouble(s)), k))
                if not w:
                    O[b, h, q] = np.nan
                    L[b, h, q] = -np.inf
                    continue
                den = sum(x for x, _ in w)
                for d in range(D):
                    O[b, h, q, d] = float(sum(x * np.longdouble(Vc[b, g, k, d]) for x, k in w) / den)
                L[b, h, q] = float(np.log(den))
    return O, L


def row_classes(o_rows: np.ndarray) -> np.ndarray:
    """0 = finite row, 1 = all-NaN row, 2 = all-zero row (for hidden rows under MaskedRows = Zero),
    3 = mixed (never valid)."""
    nan = np.isnan(o_rows)
    cls = np.full(o_rows.shape[0], 3, dtype=np.int8)
    cls[np.all(np.isfinite(o_rows), axis=1)] = 0
    cls[np.all(nan, axis=1)] = 1
    return cls
