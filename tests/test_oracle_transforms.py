"""Pins for the oracle's score transforms (CPU, no GPU): soft-capping and the
softmax sink ("com.microsoft.GroupQueryAttention" (webgpu-kernels README),
attributes softcap and smooth_softmax, input head_sink).

Readings pinned here: a cap c > 0 replaces the scaled dot product s by
c * tanh(s / c) before the additive mask; a sink logit sigma_h joins every row's
denominator as exp(sigma_h) with nothing in the numerator (sigma_h = 0 under
smooth_softmax without per-head values); LSE is the log of the whole
denominator.  Checks: a brute force written out here (numpy tanh, explicit
extra denominator term), closed forms (zero queries give equal weights, so
O = n/(n + e^sigma) * mean(V) and LSE = log(n + e^sigma); a sink with no
visible key gives O = 0 and LSE = sigma), and invariants (shifting every
visible score and the sink by one constant leaves O unchanged; capped scores
stay inside (-c, c)).
"""
from __future__ import annotations

import math
import zlib

import numpy as np
import pytest

import oracle
from tutil import canonical_problem, representable

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rand_canon(seed, B, H, G, Sq, Sk, D, dtype, scale=1.0):
    r = np.random.default_rng(seed)
    Q = representable(r.standard_normal((B, H, Sq, D)) * scale, dtype)
    K = representable(r.standard_normal((B, G, Sk, D)) * scale, dtype)
    V = representable(r.standard_normal((B, G, Sk, D)), dtype)
    return Q, K, V


def run(prob, q, k, v, **kw):
    o, lse = oracle.attn(prob, q, k, v, **kw)
    B, H, Sq, D = prob["batch"], prob["heads"], prob["q_len"], prob["head_dim"]
    return o.reshape(B, H, Sq, D), lse.reshape(B, H, Sq)


def brute(Q, K, V, scale, cap, sink, causal_off, mask=None):
    """Scores, cap, mask, then exp without max subtraction (moderate scores);
    sink: None or per-head logits joining the denominator."""
    B, H, Sq, D = Q.shape
    G, Sk = K.shape[1], K.shape[2]
    O = np.zeros((B, H, Sq, D))
    L = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            g = h // (H // G)
            for i in range(Sq):
                num = np.zeros(D, dtype=np.longdouble)
                den = np.longdouble(0)
                for k in range(Sk):
                    if causal_off is not None and k > i + causal_off:
                        continue
                    s = scale * float(np.dot(Q[b, h, i], K[b, g, k]))
                    if cap:
                        s = cap * math.tanh(s / cap)
                    if mask is not None:
                        s += float(mask[b, 0, 0, k])
                    if s == -math.inf:
                        continue
                    w = np.exp(np.longdouble(s))
                    num += w * V[b, g, k].astype(np.longdouble)
                    den += w
                if sink is not None:
                    den += np.exp(np.longdouble(sink[h]))
                if den == 0:
                    O[b, h, i] = np.nan
                    L[b, h, i] = -np.inf
                else:
                    O[b, h, i] = (num / den).astype(np.float64)
                    L[b, h, i] = float(np.log(den))
    return O, L


CASES = [
    # dtype, B, H, G, Sq, Sk, D, cap, sink ('none' | 'smooth' | 'heads'), causal offset, mask
    ("f32", 2, 2, 1, 5, 7, 4, 2.5, "none", None, False),
    ("bf16", 1, 4, 2, 4, 6, 3, 0.0, "heads", 2, False),
    ("f16", 2, 2, 2, 3, 8, 4, 1.5, "smooth", None, True),
    ("f32", 2, 4, 1, 6, 6, 2, 4.0, "heads", 0, True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"t{i}" for i in range(len(CASES))])
def test_brute_force_softcap_and_sink(case):
    dtype, B, H, G, Sq, Sk, D, cap, sink_kind, off, use_mask = case
    r = np.random.default_rng(zlib.crc32(repr(case).encode()))
    Q, K, V = rand_canon(int(r.integers(1 << 30)), B, H, G, Sq, Sk, D, dtype, scale=1.3)
    scale = 0.8
    mask = None
    if use_mask:
        mask = r.standard_normal((B, 1, 1, Sk)).astype(np.float32)
        mask[r.random(mask.shape) < 0.3] = -np.inf
    sink = None
    if sink_kind == "heads":
        sink = (r.standard_normal(H) * 2).astype(np.float32)
    prob, qs, ks, vs = canonical_problem(Q, K, V, dtype, "bhsd", scale=scale, causal=off is not None,
                                         causal_offset=off, mask_layout=(0, Sk, 0, 0) if use_mask else None)
    prob.update(softcap=cap, smooth_softmax=sink_kind == "smooth")
    o, lse = run(prob, qs, ks, vs, mask=mask, head_sink=sink)
    ref_sink = None if sink_kind == "none" else (sink if sink is not None else np.zeros(H, dtype=np.float32))
    ref_o, ref_l = brute(Q, K, V, float(np.float32(scale)), cap, ref_sink, off, mask)
    assert np.array_equal(np.isnan(o), np.isnan(ref_o))
    f = np.isfinite(ref_o)
    assert np.all(np.abs(o[f] - ref_o[f]) <= 1e-12 * (1 + np.abs(ref_o[f])))
    fl = np.isfinite(ref_l)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_l))
    assert np.all(np.abs(lse[fl] - ref_l[fl]) <= 1e-12 * (1 + np.abs(ref_l[fl])))


def test_sink_closed_form_with_zero_queries():
    B, H, G, Sq, Sk, D = 1, 3, 1, 4, 6, 5
    _, K, V = rand_canon(3, B, H, G, Sq, Sk, D, "bf16")
    Q = np.zeros((B, H, Sq, D))
    prob, qs, ks, vs = canonical_problem(Q, K, V, "bf16", "bshd", causal=True, causal_offset=1)
    sink = np.array([0.0, 1.5, -2.0], dtype=np.float32)
    o, lse = run(prob, qs, ks, vs, head_sink=sink)
    for h in range(H):
        for i in range(Sq):
            n = min(i + 2, Sk)
            den = n + math.exp(float(sink[h]))
            ref = V[0, 0, :n].sum(axis=0) / den
            assert np.allclose(o[0, h, i], ref, rtol=0, atol=1e-14)
            assert lse[0, h, i] == pytest.approx(math.log(den), abs=1e-14)


def test_smooth_softmax_equals_zero_sinks_and_fully_hidden_rows_give_zero():
    B, H, G, Sq, Sk, D = 2, 2, 2, 5, 5, 3
    Q, K, V = rand_canon(5, B, H, G, Sq, Sk, D, "f16")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f16", "bhsd", causal=True, causal_offset=-2)
    o1, l1 = run(dict(prob, smooth_softmax=True), qs, ks, vs)
    o2, l2 = run(prob, qs, ks, vs, head_sink=np.zeros(H, dtype=np.float32))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # rows 0 and 1 see no key (offset -2): O = 0, LSE = sigma = 0, in both masked-rows modes
    for mr in ("nan", "zero"):
        o, l = run(dict(prob, masked_rows=mr), qs, ks, vs, head_sink=np.full(H, 0.75, dtype=np.float32))
        assert np.all(o[:, :, :2] == 0) and np.all(l[:, :, :2] == np.float64(np.float32(0.75)))
        assert np.all(np.isfinite(o[:, :, 2:]))


def test_shifting_scores_and_sink_together_leaves_o_unchanged():
    B, H, G, Sq, Sk, D = 1, 2, 1, 4, 7, 4
    Q, K, V = rand_canon(7, B, H, G, Sq, Sk, D, "f32")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bhsd", mask_layout=(0, Sk, 0, 0))
    sink = np.array([0.25, -1.0], dtype=np.float32)   # the shifted values stay exact in float32
    zero = np.zeros((B, 1, 1, Sk), dtype=np.float32)
    c = np.float32(2.0)
    o1, l1 = run(prob, qs, ks, vs, mask=zero, head_sink=sink)
    o2, l2 = run(prob, qs, ks, vs, mask=zero + c, head_sink=sink + c)
    assert np.allclose(o1, o2, rtol=1e-13, atol=1e-14)
    assert np.allclose(l2 - l1, float(c), atol=1e-13)


def test_non_finite_sinks():
    B, H, G, Sq, Sk, D = 1, 3, 3, 2, 4, 2
    Q, K, V = rand_canon(9, B, H, G, Sq, Sk, D, "bf16")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "bf16", "bhsd")
    o, l = run(prob, qs, ks, vs, head_sink=np.array([np.nan, np.inf, -np.inf], dtype=np.float32))
    assert np.all(np.isnan(o[0, :2])) and np.all(np.isnan(l[0, :2]))          # NaN / +inf sink: NaN rows
    o0, l0 = run(prob, qs, ks, vs)
    assert np.array_equal(o[0, 2], o0[0, 2]) and np.array_equal(l[0, 2], l0[0, 2])   # -inf sink: no term


def test_capped_scores_stay_inside_the_cap():
    B, H, G, Sq, Sk, D, cap = 1, 2, 2, 3, 9, 8, 0.5
    Q, K, V = rand_canon(11, B, H, G, Sq, Sk, D, "f32", scale=3.0)
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bshd", scale=1.0)
    _, lse = run(dict(prob, softcap=cap), qs, ks, vs)
    # every capped score lies in (-cap, cap), so LSE lies in (log n - cap, log n + cap)
    assert np.all(lse > math.log(Sk) - cap) and np.all(lse < math.log(Sk) + cap)
    _, raw = run(prob, qs, ks, vs)
    assert np.any(raw > math.log(Sk) + cap)                                  # uncapped scores exceed it


def test_a_sink_far_above_every_score_dominates_without_overflow():
    B, H, G, Sq, Sk, D = 1, 2, 1, 3, 5, 4
    Q, K, V = rand_canon(13, B, H, G, Sq, Sk, D, "f32")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bshd")
    o, l = run(prob, qs, ks, vs, head_sink=np.array([800.0, -800.0], dtype=np.float32))
    # head 0: the sink's weight is 1 up to e^(score - 800): O ~ 0 and LSE = 800 to double precision
    assert np.all(np.abs(o[0, 0]) < 1e-300) and np.allclose(l[0, 0], 800.0, rtol=0, atol=1e-12)
    o0, l0 = run(prob, qs, ks, vs)
    assert np.allclose(o[0, 1], o0[0, 1], rtol=1e-15, atol=0) and np.allclose(l[0, 1], l0[0, 1], atol=1e-15)
