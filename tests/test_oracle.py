"""Pins for the float64 CPU oracle (runs without a GPU).

Each test checks the oracle against something other than itself: numpy's own
type conversions, a brute-force softmax without max subtraction, PyTorch's CPU
float64 scaled_dot_product_attention, closed forms, invariants, and the worked
examples the pages print (tests/golden/).  A plausible slip in the oracle -- a
dropped mask term, a wrong head index, a transposed operand, an off-by-one in
the causal bound, a missing special case -- fails at least one of them.
"""
from __future__ import annotations

import math
import os
import zlib

import numpy as np
import pytest

import oracle
from attention_attn_fwd_02_gb300 import workloads as wl
from tutil import brute_force, canonical_problem, representable, row_classes, widen

GOLD = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def run(prob, q, k, v, **kw):
    o, lse = oracle.attn(prob, q, k, v, **kw)
    B, H, Sq, D = prob["batch"], prob["heads"], prob["q_len"], prob["head_dim"]
    return o.reshape(B, H, Sq, D), lse.reshape(B, H, Sq)


def rand_canon(seed, B, H, G, Sq, Sk, D, dtype, scale=1.0):
    r = np.random.default_rng(seed)
    Q = representable(r.standard_normal((B, H, Sq, D)) * scale, dtype)
    K = representable(r.standard_normal((B, G, Sk, D)) * scale, dtype)
    V = representable(r.standard_normal((B, G, Sk, D)) * scale, dtype)
    return Q, K, V


def assert_rows_close(o, ref, lse, ref_lse, rtol):
    assert np.array_equal(np.isnan(o), np.isnan(ref))
    assert np.array_equal(np.isnan(lse), np.isnan(ref_lse))
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    f = np.isfinite(ref)
    assert np.all(np.abs(o[f] - ref[f]) <= rtol * (1 + np.abs(ref[f])))
    fl = np.isfinite(ref_lse)
    assert np.all(np.abs(lse[fl] - ref_lse[fl]) <= rtol * (1 + np.abs(ref_lse[fl])))


# ---- storage widening -----------------------------------------------------------


def test_widen_f16_all_patterns_match_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.widen("f16", int(b)) for b in bits])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m])
    assert np.array_equal(np.signbit(got[m]), np.signbit(ref[m]))


def test_widen_bf16_all_patterns_match_float32_upper_half():
    bits = np.arange(1 << 16, dtype=np.uint32)
    ref = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    got = np.array([oracle.widen("bf16", int(b)) for b in bits])
    m = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[m], ref[m])


def test_default_scale_is_float_nearest_inverse_sqrt():
    for d in (1, 2, 31, 32, 64, 96, 128, 200, 256):
        s = oracle.default_scale(d)
        exact = 1.0 / math.sqrt(d)
        f = np.float32(s)
        assert abs(float(f) - exact) <= 0.5 * float(np.spacing(f)) * (1 + 1e-12)


# ---- brute force on tiny shapes ---------------------------------------------------


CASES = [
    # dtype, layout, B, H, G, Sq, Sk, D, causal, offset, use_seg, use_lens, mask_kind
    ("f32", "bhsd", 1, 2, 2, 5, 5, 3, False, None, False, False, None),
    ("f32", "bshd", 2, 2, 1, 4, 7, 4, True, None, False, False, None),
    ("bf16", "bhsd", 2, 4, 2, 6, 6, 2, True, 0, True, False, None),
    ("f16", "bshd", 2, 2, 2, 3, 7, 4, False, None, False, True, "bhqk"),
    ("f32", "bshd", 2, 4, 1, 5, 6, 3, True, 2, True, True, "b11k"),
    ("bf16", "bhsd", 1, 3, 3, 6, 4, 1, True, -1, False, False, "11qk"),
    ("f16", "bhsd", 2, 2, 1, 6, 6, 4, True, 3, True, True, "bhqk"),
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
@pytest.mark.parametrize("masked_rows", ["nan", "zero"])
def test_brute_force_tiny(case, masked_rows):
    dtype, layout, B, H, G, Sq, Sk, D, causal, off, use_seg, use_lens, mask_kind = case
    r = np.random.default_rng(zlib.crc32(repr(case).encode()))
    Q, K, V = rand_canon(int(r.integers(1 << 30)), B, H, G, Sq, Sk, D, dtype)
    scale = 0.7
    seg = r.integers(-1, Sk + 1, size=(B, Sq)).astype(np.int32) if use_seg else None
    k_lens = r.integers(-1, Sk + 2, size=B).astype(np.int32) if use_lens else None
    mask = None
    mfun = None
    mlay = None
    if mask_kind is not None:
        shape = {"bhqk": (B, H, Sq, Sk), "b11k": (B, 1, 1, Sk), "11qk": (1, 1, Sq, Sk)}[mask_kind]
        mask = r.standard_normal(shape).astype(np.float32)
        mask[r.random(shape) < 0.25] = -np.inf
        mlay = {"bhqk": (0, H * Sq * Sk, Sq * Sk, Sk), "b11k": (0, Sk, 0, 0), "11qk": (0, 0, 0, Sk)}[mask_kind]
        mfun = (lambda b, h, q, k: float(mask[b if shape[0] > 1 else 0, h if shape[1] > 1 else 0,
                                             q if shape[2] > 1 else 0, k]))
    eff_off = (Sk - Sq) if off is None else off

    def vis(b, q, k):
        if k_lens is not None and k >= min(max(int(k_lens[b]), 0), Sk):
            return False
        if causal and k > q + eff_off:
            return False
        if seg is not None and k < min(max(int(seg[b, q]), 0), Sk):
            return False
        return True

    prob, qs, ks, vs = canonical_problem(Q, K, V, dtype, layout, scale=scale, causal=causal,
                                         causal_offset=off, masked_rows=masked_rows, mask_layout=mlay)
    o, lse = run(prob, qs, ks, vs, mask=mask, seg=seg, k_lens=k_lens)
    ref_o, ref_l = brute_force(Q, K, V, float(np.float32(scale)), vis, mfun)
    if masked_rows == "zero":
        ref_o[np.isnan(ref_o)] = 0.0
    assert_rows_close(o, ref_o, lse, ref_l, 1e-12)


# ---- PyTorch CPU float64 SDPA on larger shapes ----------------------------------------


@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
def test_matches_torch_sdpa_float64(layout):
    torch = pytest.importorskip("torch")
    B, H, G, Sq, Sk, D = 2, 6, 2, 33, 47, 24
    dtype = "bf16"
    Q, K, V = rand_canon(11, B, H, G, Sq, Sk, D, dtype)
    r = np.random.default_rng(12)
    off = 9
    k_lens = np.array([40, 13], dtype=np.int32)
    seg = np.sort(r.integers(0, 20, size=(B, Sq)), axis=1).astype(np.int32)
    mask = r.standard_normal((B, H, Sq, Sk)).astype(np.float32)
    mask[r.random(mask.shape) < 0.1] = -np.inf
    scale = float(np.float32(0.3))
    prob, qs, ks, vs = canonical_problem(Q, K, V, dtype, layout, scale=scale, causal=True,
                                         causal_offset=off,
                                         mask_layout=(0, H * Sq * Sk, Sq * Sk, Sk))
    o, lse = run(prob, qs, ks, vs, mask=mask, seg=seg, k_lens=k_lens)
    qi = np.arange(Sq)[:, None]
    kk = np.arange(Sk)[None, :]
    add = np.empty((B, H, Sq, Sk))
    for b in range(B):
        vis = (kk < k_lens[b]) & (kk <= qi + off) & (kk >= seg[b][:, None])
        add[b] = np.where(vis[None], mask[b].astype(np.float64), -np.inf)
    Kr = np.repeat(K, H // G, axis=1)
    Vr = np.repeat(V, H // G, axis=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q), torch.from_numpy(Kr), torch.from_numpy(Vr),
        attn_mask=torch.from_numpy(add), scale=scale).numpy()
    has = np.isfinite(add).any(axis=-1)
    assert has.sum() > 100 and (~has).sum() > 0
    assert np.all(np.abs(o[has] - ref[has]) <= 1e-12 * (1 + np.abs(ref[has])))
    ref_lse = np.log(np.exp(scale * np.einsum("bhqd,bhkd->bhqk", Q, Kr) + add).sum(-1))
    assert np.allclose(lse[has], ref_lse[has], rtol=1e-12, atol=1e-12)
    assert np.all(np.isnan(o[~has])) and np.all(np.isneginf(lse[~has]))


# ---- closed forms -----------------------------------------------------------------------


def test_zero_query_gives_mean_of_visible_values_and_log_count():
    B, H, G, Sq, Sk, D = 2, 4, 2, 9, 13, 8
    _, K, V = rand_canon(3, B, H, G, Sq, Sk, D, "f32")
    Q = np.zeros((B, H, Sq, D))
    k_lens = np.array([13, 7], dtype=np.int32)
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bshd", causal=True, causal_offset=2)
    o, lse = run(prob, qs, ks, vs, k_lens=k_lens)
    for b in range(B):
        for h in range(H):
            for q in range(Sq):
                n = min(int(k_lens[b]), q + 2 + 1)
                mean = V[b, h // 2, :n].mean(axis=0)
                assert np.allclose(o[b, h, q], mean, rtol=1e-14, atol=1e-14)
                assert abs(lse[b, h, q] - math.log(n)) < 1e-14


def test_zero_query_with_mask_gives_softmax_of_mask():
    B, H, Sq, Sk, D = 1, 2, 3, 11, 5
    _, K, V = rand_canon(4, B, H, H, Sq, Sk, D, "f32")
    Q = np.zeros((B, H, Sq, D))
    mask = np.random.default_rng(5).standard_normal((B, 1, 1, Sk)).astype(np.float32) * 3
    mask[0, 0, 0, [2, 5]] = -np.inf
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bhsd", mask_layout=(0, Sk, 0, 0))
    o, lse = run(prob, qs, ks, vs, mask=mask)
    w = np.exp(mask[0, 0, 0].astype(np.float64))
    for h in range(H):
        ref = (w[:, None] * V[0, h]).sum(0) / w.sum()
        assert np.allclose(o[0, h], ref[None], rtol=1e-13, atol=1e-14)
        assert np.allclose(lse[0, h], math.log(w.sum()), rtol=1e-14)


def test_one_hot_values_recover_probabilities():
    B, H, Sq, Sk = 1, 2, 6, 8
    D = Sk
    Q, K, _ = rand_canon(6, B, H, H, Sq, Sk, D, "f32")
    V = np.broadcast_to(np.eye(Sk), (B, H, Sk, D)).copy()
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bhsd", causal=True, causal_offset=1)
    o, lse = run(prob, qs, ks, vs)
    assert np.allclose(o.sum(-1), 1.0, rtol=0, atol=1e-14)
    sc = float(np.float32(1 / math.sqrt(D)))
    for h in range(H):
        for q in range(Sq):
            assert np.all(o[0, h, q, q + 2:] == 0.0)            # causally hidden keys get weight 0
            s = sc * (Q[0, h, q] @ K[0, h, :q + 2].T)
            p = np.exp(s - s.max())
            assert np.allclose(o[0, h, q, :q + 2], p / p.sum(), rtol=1e-13, atol=1e-15)


def test_constant_values_give_that_value():
    B, H, Sq, Sk, D = 2, 2, 7, 9, 6
    Q, K, _ = rand_canon(7, B, H, H, Sq, Sk, D, "bf16")
    V = np.full((B, H, Sk, D), 1.0)
    prob, qs, ks, vs = canonical_problem(Q, K, V, "bf16", "bshd", causal=True)
    o, _ = run(prob, qs, ks, vs)
    assert np.all(o == 1.0)
    V2 = np.full((B, H, Sk, D), -0.8125)
    prob, qs, ks, vs = canonical_problem(Q, K, V2, "bf16", "bshd")
    o2, _ = run(prob, qs, ks, vs)
    assert np.allclose(o2, -0.8125, rtol=4e-16, atol=0)


def test_single_visible_key_returns_its_value_row_exactly():
    B, H, Sq, Sk, D = 2, 3, 8, 8, 5
    Q, K, V = rand_canon(8, B, H, H, Sq, Sk, D, "f16")
    seg = np.tile(np.arange(Sq, dtype=np.int32), (B, 1))      # each row's document starts at itself
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f16", "bhsd", causal=True, causal_offset=0)
    o, lse = run(prob, qs, ks, vs, seg=seg)
    sc = float(np.float32(1 / math.sqrt(D)))
    for b in range(B):
        for h in range(H):
            for q in range(Sq):
                assert np.array_equal(o[b, h, q], V[b, h, q])
                assert lse[b, h, q] == sc * float(Q[b, h, q] @ K[b, h, q])


# ---- special values (golden: "Attention", section "Special values") ------------------


def _special_case(name, masked_rows):
    B, H, Sq, Sk, D = 1, 2, 3, 5, 4
    Q, K, V = rand_canon(9, B, H, H, Sq, Sk, D, "f32")
    kw = dict(masked_rows=masked_rows)
    extra = {}
    if name == "all_keys_mask_neg_inf":
        extra["mask"] = np.full((B, 1, 1, Sk), -np.inf, dtype=np.float32)
        kw["mask_layout"] = (0, Sk, 0, 0)
    elif name == "klen_zero":
        K, V = K[:, :, :0], V[:, :, :0]
    elif name == "key_length_zero":
        extra["k_lens"] = np.array([0], dtype=np.int32)
    elif name == "causal_before_first_key":
        kw.update(causal=True, causal_offset=-Sq)
    elif name == "segment_after_causal_bound":
        kw.update(causal=True, causal_offset=0)
        extra["seg"] = np.array([[1, 2, 3]], dtype=np.int32)
    elif name in ("nan_score", "pos_inf_score"):
        m = np.zeros((B, 1, 1, Sk), dtype=np.float32)
        m[0, 0, 0, 3] = np.nan if name == "nan_score" else np.inf
        extra["mask"] = m
        kw["mask_layout"] = (0, Sk, 0, 0)
    elif name == "lone_nan_rest_hidden":
        m = np.full((B, 1, 1, Sk), -np.inf, dtype=np.float32)
        m[0, 0, 0, 1] = np.nan
        extra["mask"] = m
        kw["mask_layout"] = (0, Sk, 0, 0)
    else:
        raise KeyError(name)
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bshd", **kw)
    return run(prob, qs, ks, vs, **extra)


def _golden_special():
    rows = []
    for line in open(os.path.join(GOLD, "special_values.txt")):
        if line.strip() and not line.startswith("#"):
            rows.append(tuple(line.split()))
    return rows


@pytest.mark.parametrize("name,masked_rows,o_class,lse_val", _golden_special())
def test_special_values_golden(name, masked_rows, o_class, lse_val):
    o, lse = _special_case(name, masked_rows)
    if name == "segment_after_causal_bound":
        o, lse = o[:, :, :], lse[:, :, :]        # every row: seg[q] = q + 1 > q + 0
    if o_class == "nan":
        assert np.all(np.isnan(o))
    else:
        assert np.all(o == 0.0)
    if lse_val == "nan":
        assert np.all(np.isnan(lse))
    else:
        assert np.all(np.isneginf(lse))


# ---- grouped heads (golden: "attention_forward ...", section "GQA") ------------------


def test_gqa_mapping_golden_and_repeat_equivalence():
    lines = [l.split() for l in open(os.path.join(GOLD, "gqa_mapping.txt")) if l.strip() and not l.startswith("#")]
    hdr = {l[0]: int(l[1]) for l in lines if not l[0].isdigit()}
    pairs = [(int(a), int(b)) for a, b in (l for l in lines if l[0].isdigit())]
    H, G = hdr["n_heads"], hdr["n_kv_heads"]
    assert H // G == hdr["q_per_group"]
    B, Sq, Sk, D = 1, 5, 6, 4
    Q, K, V = rand_canon(10, B, H, G, Sq, Sk, D, "bf16")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "bf16", "bshd", causal=True)
    o, lse = run(prob, qs, ks, vs)
    # whole problem equals MHA with K/V heads repeated q_per_group times, bit for bit
    Kr, Vr = np.repeat(K, H // G, axis=1), np.repeat(V, H // G, axis=1)
    prob2, qs2, ks2, vs2 = canonical_problem(Q, Kr, Vr, "bf16", "bshd", causal=True)
    o2, lse2 = run(prob2, qs2, ks2, vs2)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    # the page's listed (h, kv_h) pairs: head h alone against kv head kv_h
    for h, g in pairs:
        p1, q1, k1, v1 = canonical_problem(Q[:, h:h + 1], K[:, g:g + 1], V[:, g:g + 1], "bf16", "bshd", causal=True)
        oh, lh = run(p1, q1, k1, v1)
        assert np.array_equal(oh[:, 0], o[:, h]) and np.array_equal(lh[:, 0], lse[:, h])
        other = (g + 1) % G
        p2, q2, k2, v2 = canonical_problem(Q[:, h:h + 1], K[:, other:other + 1], V[:, other:other + 1], "bf16",
                                           "bshd", causal=True)
        assert not np.array_equal(run(p2, q2, k2, v2)[0][:, 0], o[:, h])


# ---- invariants ---------------------------------------------------------------------------


def test_hidden_keys_are_never_read():
    B, H, Sq, Sk, D = 2, 2, 6, 10, 4
    k_lens = np.array([6, 9], dtype=np.int32)
    case = wl.make_case(seed=21, dtype="bf16", layout="bhsd", batch=B, heads=H, q_len=Sq, k_len=Sk,
                        head_dim=D, k_lens=k_lens, causal=True, causal_offset=3, nan_fill=True)
    o, lse = oracle.attn(case.problem, case.q, case.k, case.v, k_lens=case.k_lens)
    assert np.all(np.isfinite(o))
    # permute the hidden (beyond-length) keys and fill with other garbage: no change, bit for bit
    k2, v2 = case.k.copy(), case.v.copy()
    k2[0, :, 6:] = k2[0, :, 6:][:, ::-1]
    v2[0, :, 6:] = 0x7F80                                   # +inf
    o2, lse2 = oracle.attn(case.problem, case.q, k2, v2, k_lens=case.k_lens)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_permuting_mask_hidden_keys_changes_nothing():
    B, H, Sq, Sk, D = 1, 2, 4, 12, 3
    Q, K, V = rand_canon(22, B, H, H, Sq, Sk, D, "f32")
    mask = np.zeros((B, 1, 1, Sk), dtype=np.float32)
    hidden = np.array([1, 4, 7, 10])
    mask[0, 0, 0, hidden] = -np.inf
    kw = dict(mask_layout=(0, Sk, 0, 0))
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bshd", **kw)
    o, lse = run(prob, qs, ks, vs, mask=mask)
    perm = hidden[[2, 3, 0, 1]]
    K2, V2 = K.copy(), V.copy()
    K2[:, :, hidden], V2[:, :, hidden] = K[:, :, perm], V[:, :, perm]
    prob, qs, ks, vs = canonical_problem(Q, K2, V2, "f32", "bshd", **kw)
    o2, lse2 = run(prob, qs, ks, vs, mask=mask)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_mask_shift_and_scale_folding():
    B, H, Sq, Sk, D = 1, 2, 5, 9, 4
    Q, K, V = rand_canon(23, B, H, H, Sq, Sk, D, "f32")
    # multiples of 1/64 so that adding 3 is exact in float32
    mask = (np.round(np.random.default_rng(24).standard_normal((B, H, Sq, Sk)) * 64) / 64).astype(np.float32)
    lay = (0, H * Sq * Sk, Sq * Sk, Sk)
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bhsd", scale=0.5, mask_layout=lay)
    o, lse = run(prob, qs, ks, vs, mask=mask)
    o2, lse2 = run(prob, qs, ks, vs, mask=mask + np.float32(3.0))
    assert np.allclose(o, o2, rtol=1e-13, atol=1e-14)
    assert np.allclose(lse + 3.0, lse2, rtol=1e-14, atol=1e-13)
    # scale * (2Q) == (2 scale) * Q exactly (scalings by two)
    prob2, qs2, ks2, vs2 = canonical_problem(2 * Q, K, V, "f32", "bhsd", scale=0.25, mask_layout=lay)
    o3, lse3 = run(prob2, qs2, ks2, vs2, mask=mask)
    assert np.array_equal(o, o3) and np.array_equal(lse, lse3)


def test_mask_is_added_after_scaling():
    B, H, Sq, Sk, D = 1, 1, 1, 2, 1
    Q = np.array([[[[2.0]]]])
    K = np.array([[[[1.0], [0.0]]]])
    V = np.array([[[[1.0], [0.0]]]])
    mask = np.array([[[[1.0, 0.0]]]], dtype=np.float32)
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bhsd", scale=0.5, mask_layout=(0, Sk, 0, 0))
    o, lse = run(prob, qs, ks, vs, mask=mask)
    s0, s1 = 0.5 * 2.0 + 1.0, 0.0                       # scale * q.k + mask
    assert abs(o[0, 0, 0, 0] - math.exp(s0) / (math.exp(s0) + math.exp(s1))) < 1e-15
    assert abs(lse[0, 0, 0] - math.log(math.exp(s0) + math.exp(s1))) < 1e-15


def test_online_recurrence_agrees_with_three_pass():
    """The page's blocked online recurrence (blocks of 256 keys, correction
    exp(m_old - m_new)), restated here with the guard for a row whose keys are
    all hidden so far, reaches the oracle's result to rounding."""
    B, H, Sq, Sk, D = 1, 2, 3, 1000, 8
    Q, K, V = rand_canon(25, B, H, H, Sq, Sk, D, "bf16", scale=2.0)
    seg = np.array([[0, 300, 700]], dtype=np.int32)
    prob, qs, ks, vs = canonical_problem(Q, K, V, "bf16", "bhsd", seg_batch_stride=Sq)
    o, lse = run(prob, qs, ks, vs, seg=seg)
    sc = float(np.float32(1 / math.sqrt(D)))
    for h in range(H):
        for q in range(Sq):
            m, l, acc = -np.inf, 0.0, np.zeros(D)
            for k0 in range(0, Sk, 256):
                ks_ = np.arange(k0, min(Sk, k0 + 256))
                s = np.where(ks_ >= seg[0, q], sc * (K[0, h, ks_] @ Q[0, h, q]), -np.inf)
                m_new = max(m, s.max())
                if m_new == -np.inf:
                    continue
                p = np.exp(s - m_new)
                corr = math.exp(m - m_new)
                l = l * corr + p.sum()
                acc = acc * corr + p @ V[0, h, ks_]
                m = m_new
            assert np.allclose(o[0, h, q], acc / l, rtol=1e-12, atol=1e-13)
            assert abs(lse[0, h, q] - (m + math.log(l))) < 1e-12


# ---- combine --------------------------------------------------------------------------------


def test_split_then_combine_equals_whole_row():
    B, H, Sq, Sk, D = 1, 2, 4, 37, 6
    Q, K, V = rand_canon(26, B, H, H, Sq, Sk, D, "f32")
    mask = np.random.default_rng(27).standard_normal((B, 1, 1, Sk)).astype(np.float32)
    mask[0, 0, 0, 10:17] = -np.inf                            # range 1 below is entirely hidden
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bshd", mask_layout=(0, Sk, 0, 0))
    o, lse = run(prob, qs, ks, vs, mask=mask)
    cuts = [0, 10, 17, 30, 37]
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        pr, q1, k1, v1 = canonical_problem(Q, K[:, :, a:b], V[:, :, a:b], "f32", "bshd", mask_layout=(0, b - a, 0, 0),
                                           scale=float(np.float32(1 / math.sqrt(D))))
        po, pl = run(pr, q1, k1, v1, mask=np.ascontiguousarray(mask[..., a:b]))
        parts_o.append(np.where(np.isnan(po), 0.0, po))
        parts_l.append(pl)
    po = np.stack(parts_o, axis=3).reshape(B * H * Sq, len(parts_o), D)
    pl = np.stack(parts_l, axis=3).reshape(B * H * Sq, len(parts_l))
    assert np.all(np.isneginf(pl[:, 1]))
    co, cl = oracle.combine(po.astype(np.float32), pl.astype(np.float32))
    assert np.allclose(co, o.reshape(-1, D), rtol=2e-6, atol=2e-6)
    assert np.allclose(cl, lse.reshape(-1), rtol=1e-6, atol=1e-6)


def test_combine_closed_forms():
    D = 3
    a = np.array([1.0, -2.0, 0.5], dtype=np.float32)
    b = np.array([3.0, 4.0, -0.5], dtype=np.float32)
    po = np.stack([np.stack([a, b]), np.stack([a, b]), np.stack([a, b]), np.stack([a, b])])
    pl = np.array([[0.0, 0.0], [-np.inf, 1.5], [-np.inf, -np.inf], [np.nan, 0.0]], dtype=np.float32)
    for mr in ("nan", "zero"):
        o, l = oracle.combine(po, pl, masked_rows=mr)
        assert np.array_equal(o[0], (a.astype(np.float64) + b) / 2) and l[0] == math.log(2.0)
        assert np.array_equal(o[1], b.astype(np.float64)) and l[1] == 1.5
        assert (np.all(np.isnan(o[2])) if mr == "nan" else np.all(o[2] == 0)) and np.isneginf(l[2])
        assert np.all(np.isnan(o[3])) and np.isnan(l[3])
    assert D == 3


# ---- named workloads: small-scale sanity of the generators with the oracle --------------------


def test_named_workload_generators_shapes_and_rules():
    c1 = wl.tiny_f32_mha()
    assert c1.q.shape == (1, 64, 2, 32) and c1.q.dtype == np.float32
    c2 = wl.gqa_doc_causal_bf16(batch=2, seq=1024)
    assert c2.seg.shape == (2, 1024)
    for b in range(2):
        starts = np.unique(c2.seg[b])
        lens = np.diff(np.append(starts, 1024))
        assert np.all(lens[:-1] >= 64) and np.all(lens <= 512)
        assert np.all(c2.seg[b] <= np.arange(1024))
    c5 = wl.cross_mask_f16(batch=3, q_len=4, k_len=40, heads=2)
    assert np.all(np.isneginf(c5.mask[-1]))
    assert all(int(np.isneginf(c5.mask[b]).sum()) == 4 for b in range(2))
    o, lse = oracle.attn(c5.problem, c5.q, c5.k, c5.v, mask=c5.mask)
    o = o.reshape(3, 2, 4, 256)
    assert np.all(np.isnan(o[2])) and np.all(np.isfinite(o[:2]))


def test_oracle_rejects_bad_problems():
    Q, K, V = rand_canon(30, 1, 3, 3, 2, 2, 2, "f32")
    prob, qs, ks, vs = canonical_problem(Q, K, V, "f32", "bhsd")
    prob["kv_heads"] = 2
    with pytest.raises(ValueError):
        oracle.attn(prob, qs, ks, vs)
    prob["kv_heads"] = 3
    with pytest.raises(ValueError):
        oracle.attn(prob, qs, ks, vs, rows=np.array([[0, 3, 0]]))


def test_bf16_rounding_paths_agree_bit_for_bit():
    r = np.random.default_rng(77)
    x = (r.standard_normal(1 << 16) * np.exp(r.uniform(-30, 30, 1 << 16))).astype(np.float32)
    x[:4] = [np.inf, -np.inf, 0.0, -0.0]
    # ties: values exactly halfway between two bfloat16 numbers
    x[4:8] = np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x00008000], dtype=np.uint32).view(np.float32)
    a = wl.f32_to_bf16_bits(x)
    b = wl.f32_to_bf16_bits_numpy(x)
    assert np.array_equal(a, b)
    assert list(a[4:8]) == [0x3F80, 0x3F82, 0xBF80, 0x0000]
