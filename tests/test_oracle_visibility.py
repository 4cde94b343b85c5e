"""Pins for the oracle's visibility variants (CPU, no GPU): the sliding window
(left window w over the causal diagonal), the causal bound right-aligned to
each batch entry's key length (chunked prefill), and key lengths given as the
last valid index (ONNX seqlens_k).  Source: "com.microsoft.GroupQueryAttention"
(webgpu-kernels README), attributes local_window_size and causal, input
seqlens_k, and its chunked-prefill variants.

Each variant is checked against a brute force whose visibility test is written
out here independently, against closed forms (a window of 0 keeps the diagonal
key alone, so the row returns that key's V exactly), and against equivalent
problems the oracle already answers through other code (a window is the same
as per-row segment starts; right alignment is one scalar offset per batch
entry; last-index lengths are counts minus one).
"""
from __future__ import annotations

import zlib

import numpy as np
import pytest

import oracle
from tutil import brute_force, canonical_problem, representable

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rand_canon(seed, B, H, G, Sq, Sk, D, dtype):
    r = np.random.default_rng(seed)
    Q = representable(r.standard_normal((B, H, Sq, D)), dtype)
    K = representable(r.standard_normal((B, G, Sk, D)), dtype)
    V = representable(r.standard_normal((B, G, Sk, D)), dtype)
    return Q, K, V


def run(prob, q, k, v, **kw):
    o, lse = oracle.attn(prob, q, k, v, **kw)
    B, H, Sq, D = prob["batch"], prob["heads"], prob["q_len"], prob["head_dim"]
    return o.reshape(B, H, Sq, D), lse.reshape(B, H, Sq)


def close(o, ref, lse, ref_l, tol=1e-12):
    assert np.array_equal(np.isnan(o), np.isnan(ref))
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_l))
    f = np.isfinite(ref)
    assert np.all(np.abs(o[f] - ref[f]) <= tol * (1 + np.abs(ref[f])))
    fl = np.isfinite(ref_l)
    assert np.all(np.abs(lse[fl] - ref_l[fl]) <= tol * (1 + np.abs(ref_l[fl])))


VARIANTS = [
    # dtype, layout, B, H, G, Sq, Sk, D, offset, window, align, lens, last_index, seg
    ("f32", "bhsd", 2, 2, 1, 6, 9, 3, None, 2, "fixed", True, False, False),
    ("bf16", "bshd", 3, 2, 2, 4, 8, 2, None, 0, "klens", True, False, False),
    ("f16", "bhsd", 2, 4, 2, 5, 7, 3, 1, 3, "fixed", False, False, True),
    ("f32", "bshd", 3, 2, 1, 3, 9, 4, None, -1, "klens", True, True, False),
    ("bf16", "bhsd", 2, 2, 2, 6, 6, 2, -2, 1, "fixed", True, True, True),
    ("f32", "bhsd", 2, 3, 3, 4, 10, 2, None, 4, "klens", True, True, False),
]


@pytest.mark.parametrize("case", VARIANTS, ids=[f"v{i}" for i in range(len(VARIANTS))])
def test_brute_force_visibility_variants(case):
    dtype, layout, B, H, G, Sq, Sk, D, off, window, align, use_lens, last_index, use_seg = case
    r = np.random.default_rng(zlib.crc32(repr(case).encode()))
    Q, K, V = rand_canon(int(r.integers(1 << 30)), B, H, G, Sq, Sk, D, dtype)
    scale = 0.6
    k_lens = r.integers(-1, Sk + 2, size=B).astype(np.int32) if use_lens else None
    seg = r.integers(-1, Sk, size=(B, Sq)).astype(np.int32) if use_seg else None
    stored = None if k_lens is None else (k_lens - 1 if last_index else k_lens).astype(np.int32)

    def count(b):
        return Sk if k_lens is None else min(max(int(k_lens[b]), 0), Sk)

    def vis(b, q, k):
        if k >= count(b):
            return False
        o_b = count(b) - Sq if align == "klens" else ((Sk - Sq) if off is None else off)
        if k > q + o_b:
            return False
        if window >= 0 and k < q + o_b - window:
            return False
        if seg is not None and k < min(max(int(seg[b, q]), 0), Sk):
            return False
        return True

    prob, qs, ks, vs = canonical_problem(Q, K, V, dtype, layout, scale=scale, causal=True, causal_offset=off)
    prob.update(window_left=window, causal_align=align, k_lens_kind="last_index" if last_index else "count")
    o, lse = run(prob, qs, ks, vs, seg=seg, k_lens=stored)
    ref_o, ref_l = brute_force(Q, K, V, float(np.float32(scale)), vis)
    close(o, ref_o, lse, ref_l)


def test_window_zero_returns_the_diagonal_value_exactly():
    B, H, G, Sq, Sk, D = 2, 4, 2, 7, 11, 5
    Q, K, V = rand_canon(3, B, H, G, Sq, Sk, D, "bf16")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "bf16", "bhsd", causal=True, causal_offset=2)
    prob["window_left"] = 0
    o, lse = run(prob, qs, ks, vs)
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                k = i + 2
                if k < Sk:
                    assert np.array_equal(o[b, h, i], V[b, h // 2, k])
                    assert lse[b, h, i] == pytest.approx(float(np.float32(oracle.default_scale(D))) *
                                                         float(np.dot(Q[b, h, i], K[b, h // 2, k])), abs=1e-12)
                else:
                    assert np.all(np.isnan(o[b, h, i])) and np.isneginf(lse[b, h, i])


def test_window_equals_segment_starts():
    B, H, G, Sq, Sk, D, w, off = 2, 2, 1, 9, 14, 4, 3, 4
    Q, K, V = rand_canon(5, B, H, G, Sq, Sk, D, "f16")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f16", "bshd", causal=True, causal_offset=off)
    k_lens = np.array([12, 7], dtype=np.int32)
    win = dict(prob, window_left=w)
    o1, l1 = run(win, qs, ks, vs, k_lens=k_lens)
    seg = np.tile(np.arange(Sq, dtype=np.int32) + off - w, (B, 1))
    o2, l2 = run(prob, qs, ks, vs, k_lens=k_lens, seg=seg)
    assert np.array_equal(o1, o2, equal_nan=True) and np.array_equal(l1, l2, equal_nan=True)


def test_large_window_equals_no_window():
    B, H, G, Sq, Sk, D = 1, 2, 2, 8, 8, 3
    Q, K, V = rand_canon(7, B, H, G, Sq, Sk, D, "f32")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bhsd", causal=True)
    o1, l1 = run(dict(prob, window_left=Sk), qs, ks, vs)
    o2, l2 = run(prob, qs, ks, vs)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_last_index_lengths_equal_counts_minus_one():
    B, H, G, Sq, Sk, D = 3, 2, 1, 5, 9, 3
    Q, K, V = rand_canon(9, B, H, G, Sq, Sk, D, "bf16")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "bf16", "bhsd", causal=True, causal_offset=3)
    counts = np.array([9, 0, 4], dtype=np.int32)
    o1, l1 = run(prob, qs, ks, vs, k_lens=counts)
    o2, l2 = run(dict(prob, k_lens_kind="last_index"), qs, ks, vs, k_lens=counts - 1)
    assert np.array_equal(o1, o2, equal_nan=True) and np.array_equal(l1, l2, equal_nan=True)
    assert np.all(np.isnan(o1[1])) and np.all(np.isneginf(l1[1]))   # a zero count hides every key


def test_right_aligned_bound_is_one_offset_per_batch_entry():
    B, H, G, Sq, Sk, D = 3, 2, 2, 4, 10, 3
    Q, K, V = rand_canon(11, B, H, G, Sq, Sk, D, "f16")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f16", "bhsd", causal=True)
    k_lens = np.array([10, 6, 3], dtype=np.int32)
    o, l = run(dict(prob, causal_align="klens"), qs, ks, vs, k_lens=k_lens)
    for b in range(B):
        one = dict(prob, batch=1, causal_offset=int(k_lens[b]) - Sq)
        sl = slice(b, b + 1)
        conv = (lambda x: np.ascontiguousarray(x[sl]))
        ob, lb = run(one, conv(qs.reshape(B, H, Sq, D)), conv(ks.reshape(B, G, Sk, D)),
                     conv(vs.reshape(B, G, Sk, D)), k_lens=k_lens[sl])
        assert np.array_equal(o[b], ob[0], equal_nan=True) and np.array_equal(l[b], lb[0], equal_nan=True)


def test_right_aligned_without_lengths_is_the_default_offset():
    B, H, G, Sq, Sk, D = 2, 2, 1, 5, 9, 2
    Q, K, V = rand_canon(13, B, H, G, Sq, Sk, D, "bf16")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "bf16", "bshd", causal=True)
    o1, l1 = run(dict(prob, causal_align="klens"), qs, ks, vs)
    o2, l2 = run(prob, qs, ks, vs)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
