"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Small and medium cases compare every element; the full-size workloads compare
sampled rows the oracle computes one by one.  Bars: float32 per element
|d| <= 2e-6 (1 + |O|); f16/bf16 |d| <= 1.5e-2 absolute; LSE |d| <= 1e-3;
NaN / zero row classes exact; plus the scaled-error bounds of "Attention"
(recursiveai.org OneGPU docs), section "Tolerances".
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from attention_attn_fwd_02_gb300 import attn, build
from attention_attn_fwd_02_gb300 import workloads as wl
from gpu_util import GpuCase, compare, host_storage, oracle_full, torch_mod

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = torch_mod()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    attn.lib()


def run_and_compare(case, lse=True, where=None):
    g = GpuCase(case, lse=lse).run()
    o, l, _ = g.outputs()
    g.check_guards()
    ref_o, ref_l = oracle_full(case)
    st = compare(o, l, ref_o, ref_l if lse else None, case.problem["dtype"], case.problem["masked_rows"],
                 where or case.name)
    assert attn.attn_device_status() == attn.ATTN_OK
    return st, g


# ---- the named workloads (reduced where the full size is sampled below) ---------------------


def test_tiny_f32_mha():
    run_and_compare(wl.tiny_f32_mha())


def test_gqa_doc_causal_bf16_full():
    run_and_compare(wl.gqa_doc_causal_bf16())


def test_long_causal_gqa_bf16_reduced():
    run_and_compare(wl.long_causal_gqa_bf16(batch=2, seq=640, heads=8, kv_heads=2))


@pytest.mark.parametrize("cap", [1024, 8192])
def test_decode_bnsh_bf16_reduced(cap):
    run_and_compare(wl.decode_bnsh_bf16(batch=4, capacity=cap, heads=32, kv_heads=8, min_len=1), lse=True)


@pytest.mark.parametrize("masked_rows", ["nan", "zero"])
def test_cross_mask_f16_reduced(masked_rows):
    c = wl.cross_mask_f16(batch=3, q_len=130, k_len=300, heads=2, masked_rows=masked_rows)
    st, _ = run_and_compare(c)
    assert st["nan_rows"] == (2 * 130 if masked_rows == "nan" else 0)


# ---- edge sweep ---------------------------------------------------------------------------

EDGE = [
    # dtype, layout, B, H, G, Sq, Sk, D, causal, offset, seg, lens, mask, masked_rows, packed
    ("f32", "bshd", 1, 1, 1, 1, 1, 1, False, None, False, False, None, "nan", False),
    ("f32", "bhsd", 2, 3, 1, 33, 65, 31, True, None, False, False, None, "nan", False),
    ("f32", "bshd", 1, 4, 2, 129, 127, 33, True, 5, True, True, "bhqk", "zero", False),
    ("f32", "bshd", 2, 2, 2, 7, 0, 16, False, None, False, False, None, "nan", False),
    ("f32", "bshd", 2, 2, 2, 7, 0, 16, False, None, False, False, None, "zero", False),
    ("bf16", "bshd", 2, 8, 1, 200, 200, 64, True, 0, True, False, None, "nan", False),
    ("bf16", "bhsd", 1, 6, 3, 129, 1000, 128, True, None, False, True, "b11k", "nan", False),
    ("bf16", "bshd", 2, 4, 4, 128, 128, 96, True, -3, False, False, None, "zero", False),
    ("f16", "bshd", 1, 2, 2, 65, 257, 256, False, None, False, True, "b11k", "nan", False),
    ("f16", "bhsd", 2, 32, 1, 17, 300, 2, True, 100, True, True, None, "nan", False),
    ("bf16", "bshd", 2, 4, 2, 150, 150, 64, True, None, False, False, None, "nan", True),
    ("f16", "bshd", 1, 2, 1, 127, 127, 200, False, None, False, False, "11qk", "zero", True),
    ("bf16", "bhsd", 3, 2, 2, 1, 513, 128, False, None, False, True, None, "nan", False),
    ("f32", "bhsd", 1, 2, 2, 300, 300, 256, True, None, False, False, None, "nan", False),
    # float32 at odd head dims around the thread-per-row splits (CUDA-core path)
    ("f32", "bshd", 2, 2, 1, 45, 70, 63, True, None, False, True, None, "nan", False),
    ("f32", "bhsd", 1, 3, 3, 33, 100, 65, False, None, False, False, "bhqk", "nan", False),
    ("f32", "bshd", 1, 2, 2, 40, 40, 127, True, 0, True, False, None, "zero", False),
    ("f32", "bhsd", 2, 2, 1, 20, 77, 129, False, None, False, True, "b11k", "nan", False),
    ("f32", "bshd", 1, 2, 1, 30, 50, 255, True, None, False, False, None, "nan", False),
    # float32 at head_dim 8 x threads-per-row (the chunked form: 16-byte shared-memory loads)
    ("f32", "bhsd", 2, 4, 2, 70, 150, 64, True, None, True, True, "bhqk", "nan", False),
    ("f32", "bshd", 1, 2, 1, 1, 300, 128, False, None, False, True, "b11k", "zero", False),
    ("f32", "bshd", 2, 3, 3, 40, 33, 32, True, 2, False, False, "11qk", "nan", False),
    ("bf16", "bhsd", 2, 4, 2, 70, 90, 32, True, None, True, True, "bhqk", "nan", False),
    ("f16", "bshd", 1, 4, 1, 1, 200, 32, False, None, False, True, "b11k", "zero", False),
    # head_dim 256 with two and three key tiles: the last P V may still be two phases behind
    ("bf16", "bhsd", 2, 4, 2, 200, 100, 256, False, None, False, False, None, "nan", False),
    ("f16", "bshd", 1, 3, 1, 260, 190, 256, True, None, False, True, None, "zero", False),
    # masks with a row per query on the tensor-core kernels: rows of 517 floats (not 16-byte aligned,
    # element loads) with a ragged last key tile; aligned rows (vector loads) with segments, and with a
    # ragged last tile; head_dim 256 on CTA pairs
    ("bf16", "bhsd", 2, 4, 2, 300, 517, 128, True, None, False, True, "11qk", "nan", False),
    ("f16", "bshd", 1, 4, 1, 257, 640, 64, False, None, True, False, "bhqk", "zero", False),
    ("bf16", "bhsd", 1, 2, 2, 200, 1000, 128, False, None, False, False, "bhqk", "zero", False),
    ("bf16", "bshd", 1, 2, 1, 260, 300, 256, True, None, False, True, "bhqk", "nan", False),
]


def make_edge(i, e):
    dtype, layout, B, H, G, Sq, Sk, D, causal, off, use_seg, use_lens, mk, mr, packed = e
    r = np.random.default_rng(1000 + i)
    seg = np.sort(r.integers(0, max(1, Sk), size=(B, Sq)), axis=1).astype(np.int32) if use_seg else None
    k_lens = None
    if use_lens:
        k_lens = r.integers(0, Sk + 1, size=B).astype(np.int32)
        k_lens[0] = Sk if B > 1 else k_lens[0]
    mask = None
    if mk is not None:
        shape = {"bhqk": (B, H, Sq, Sk), "b11k": (B, 1, 1, Sk), "11qk": (1, 1, Sq, Sk)}[mk]
        mask = r.standard_normal(shape).astype(np.float32)
        mask[r.random(shape) < 0.2] = -np.inf
    return wl.make_case(name=f"edge{i}", seed=2000 + i, dtype=dtype, layout=layout, batch=B, heads=H, kv_heads=G,
                        q_len=Sq, k_len=Sk, head_dim=D, causal=causal, causal_offset=off, seg=seg,
                        k_lens=k_lens, mask=mask, mask_kind=mk or "b11k", masked_rows=mr, packed=packed)


@pytest.mark.parametrize("i", range(len(EDGE)))
def test_edge_sweep(i):
    run_and_compare(make_edge(i, EDGE[i]))


def test_nan_and_inf_scores_make_nan_rows():
    B, H, Sq, Sk, D = 1, 2, 40, 70, 64
    mask = np.zeros((B, 1, 1, Sk), dtype=np.float32)
    mask[0, 0, 0, 5] = np.nan
    c = wl.make_case(name="nan_score", seed=31, dtype="bf16", batch=B, heads=H, q_len=Sq, k_len=Sk, head_dim=D,
                     causal=True, causal_offset=0, mask=mask)
    st, _ = run_and_compare(c)
    assert st["nan_rows"] == H * (Sq - 5)
    mask[0, 0, 0, 5] = np.inf
    mask[0, 0, 0, :5] = -np.inf
    c = wl.make_case(name="inf_score", seed=31, dtype="bf16", batch=B, heads=H, q_len=Sq, k_len=Sk, head_dim=D,
                     causal=True, causal_offset=0, mask=mask, masked_rows="zero")
    run_and_compare(c)


# ---- structural properties ------------------------------------------------------------------


def test_rerun_is_bit_identical():
    c = wl.long_causal_gqa_bf16(batch=1, seq=700, heads=4, kv_heads=2)
    g = GpuCase(c).run()
    _, l1, o1 = g.outputs()
    g.run()
    _, l2, o2 = g.outputs()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2, equal_nan=True)


def test_single_visible_key_is_exact():
    B, H, S, D = 2, 4, 260, 128
    seg = np.tile(np.arange(S, dtype=np.int32), (B, 1))
    c = wl.make_case(name="single_key", seed=41, dtype="bf16", layout="bhsd", batch=B, heads=H, q_len=S,
                     head_dim=D, causal=True, causal_offset=0, seg=seg)
    g = GpuCase(c).run()
    _, _, raw = g.outputs()
    v = c.v.reshape(B, H, S, D)
    assert np.array_equal(raw, v)


def test_gqa_equals_repeated_heads():
    B, H, G, S, D = 1, 8, 2, 300, 64
    c = wl.make_case(name="gqa", seed=43, dtype="bf16", layout="bhsd", batch=B, heads=H, kv_heads=G, q_len=S,
                     head_dim=D, causal=True)
    c2 = wl.make_case(name="mha", seed=43, dtype="bf16", layout="bhsd", batch=B, heads=H, kv_heads=G, q_len=S,
                      head_dim=D, causal=True)
    c2.k = np.repeat(c.k.reshape(B, G, S, D), H // G, axis=1).copy()
    c2.v = np.repeat(c.v.reshape(B, G, S, D), H // G, axis=1).copy()
    c2.problem = dict(c.problem, kv_heads=H, k_layout=wl.layout_of("bhsd", B, H, S, D)[1],
                      v_layout=wl.layout_of("bhsd", B, H, S, D)[1])
    _, l1, o1 = GpuCase(c).run().outputs()
    _, l2, o2 = GpuCase(c2).run().outputs()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_hidden_keys_filled_with_nan_are_not_read():
    c = wl.long_causal_gqa_bf16(batch=2, seq=384, heads=4, kv_heads=1)
    assert c.k_lens.min() < 384
    st, _ = run_and_compare(c)
    assert st["nan_rows"] == 0


@pytest.mark.parametrize("n,D", [(5, 72), (37, 256), (70, 40), (1, 128)])
def test_combine_matches_oracle(n, D):
    """Range counts below, across and beyond one warp's width; the partial rows
    of empty ranges (lse -inf) hold NaN, which must not reach the sum."""
    torch = torch_mod()
    r = np.random.default_rng(51 + n)
    rows = 37
    po = r.standard_normal((rows, n, D)).astype(np.float32)
    pl = (r.standard_normal((rows, n)) * 3).astype(np.float32)
    pl[r.random((rows, n)) < 0.3] = -np.inf
    pl[3] = -np.inf
    pl[4, n // 2] = np.nan
    pl[5, n - 1] = np.inf
    po[np.isneginf(pl)] = np.nan
    for mr in ("nan", "zero"):
        ref_o, ref_l = oracle.combine(po, pl, masked_rows=mr)
        for dt, tol in ((torch.float32, 1e-6), (torch.bfloat16, 1.5e-2)):
            o, l = attn.combine(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), out_dtype=dt,
                                masked_rows=mr, return_lse=True)
            o = o.float().cpu().numpy().astype(np.float64)
            l = l.cpu().numpy().astype(np.float64)
            assert np.array_equal(np.isnan(o), np.isnan(ref_o))
            f = np.isfinite(ref_o)
            assert np.all(np.abs(o[f] - ref_o[f]) <= tol * (1 + np.abs(ref_o[f])))
            assert np.array_equal(np.isnan(l), np.isnan(ref_l)) and np.array_equal(np.isneginf(l), np.isneginf(ref_l))
            fl = np.isfinite(ref_l)
            assert np.allclose(l[fl], ref_l[fl], atol=1e-5)


def test_key_range_split_then_combine_equals_one_call():
    """Two attn_fwd calls on disjoint key ranges merged by attn_combine equal one call."""
    torch = torch_mod()
    B, H, Sq, Sk, D = 1, 4, 100, 600, 128
    c = wl.make_case(name="split", seed=61, dtype="bf16", layout="bhsd", batch=B, heads=H, q_len=Sq, k_len=Sk,
                     head_dim=D)
    full_o, full_l = oracle_full(c)
    kk = torch.from_numpy(c.k.view(np.int16)).cuda().view(torch.bfloat16).reshape(B, H, Sk, D)
    vv = torch.from_numpy(c.v.view(np.int16)).cuda().view(torch.bfloat16).reshape(B, H, Sk, D)
    qq = torch.from_numpy(c.q.view(np.int16)).cuda().view(torch.bfloat16).reshape(B, H, Sq, D)
    parts = []
    for a, b in ((0, 250), (250, 600)):
        o, l = attn.fwd(qq, kk[:, :, a:b], vv[:, :, a:b], layout="bhsd", scale=float(np.float32(1 / np.sqrt(D))),
                        return_lse=True)
        parts.append((o.float(), l))
    po = torch.stack([p[0] for p in parts], dim=3).reshape(B * H * Sq, 2, D).contiguous()
    pl = torch.stack([p[1] for p in parts], dim=3).reshape(B * H * Sq, 2).contiguous()
    o, l = attn.combine(po, pl, out_dtype=torch.bfloat16, return_lse=True)
    o = o.float().cpu().numpy().reshape(B, H, Sq, D)
    assert np.max(np.abs(o - full_o)) <= 2e-2
    assert np.max(np.abs(l.cpu().numpy().reshape(B, H, Sq) - full_l)) <= 1e-3


def test_prefill_with_a_null_workspace_matches_the_first_call():
    """attn_fwd called again with a null workspace and size 0 (what a caller
    passes when attn_fwd_workspace_size returns 0) gives the same bits as the
    first call and matches the oracle."""
    c = wl.long_causal_gqa_bf16(batch=2, seq=1500, heads=8, kv_heads=2)
    g = GpuCase(c).run()
    _, l1, o1 = g.outputs()
    torch = torch_mod()
    ptr = (lambda t: None if t is None else t.data_ptr())
    rc = attn.attn_fwd(g.prob, ptr(g.q), ptr(g.k), ptr(g.v), ptr(g.o), None, None, ptr(g.k_lens), ptr(g.lse), None, 0,
                       torch.cuda.current_stream().cuda_stream)
    assert rc == attn.ATTN_OK
    o, l2, o2 = g.outputs()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    ref_o, ref_l = oracle_full(c)
    compare(o, l2, ref_o, ref_l, "bf16", "nan", "static schedule")


# ---- decode variants (the tensor-core split pass and the generic one) ---------------------

DECODE = [
    # dtype, B, H, G, cap, D, mask, lse, lens
    ("bf16", 3, 16, 16, 1000, 128, False, True, "rand"),     # one query head per kv head
    ("f16", 2, 10, 5, 777, 128, True, True, "rand"),         # 2 heads per group, mask, f16
    ("bf16", 2, 16, 1, 1300, 128, False, False, "zero_full"),  # 16 heads per group, lengths 0 and cap
    ("bf16", 1, 40, 2, 600, 128, True, True, "rand"),        # 20 heads per group: two head chunks
    ("bf16", 2, 8, 2, 900, 64, False, True, "rand"),         # head_dim 64: generic split pass
    ("f16", 2, 6, 3, 513, 96, True, True, None),             # head_dim 96, no lengths: generic
]


@pytest.mark.parametrize("i", range(len(DECODE)))
def test_decode_variants(i):
    dtype, B, H, G, cap, D, use_mask, lse, lens = DECODE[i]
    r = np.random.default_rng(500 + i)
    k_lens = None
    if lens == "rand":
        k_lens = r.integers(1, cap + 1, size=B).astype(np.int32)
    elif lens == "zero_full":
        k_lens = np.array([0, cap], dtype=np.int32)
    mask = None
    if use_mask:
        mask = r.standard_normal((B, 1, 1, cap)).astype(np.float32)
        mask[r.random(mask.shape) < 0.15] = -np.inf
    c = wl.make_case(name=f"decode{i}", seed=600 + i, dtype=dtype, batch=B, heads=H, kv_heads=G, q_len=1,
                     k_len=cap, head_dim=D, k_lens=k_lens, mask=mask, mask_kind="b11k", decode=True)
    st, _ = run_and_compare(c, lse=lse)
    if lens == "zero_full":
        assert st["nan_rows"] == H      # batch entry 0 has no valid key


# ---- visibility variants: sliding window, right-aligned causal bound, last-index lengths -----------

VIS = [
    # dtype, layout, B, H, G, Sq, Sk, D, offset, window, align, lens, last_index, mask
    ("bf16", "bhsd", 2, 8, 2, 300, 700, 128, None, 100, "klens", True, False, None),    # chunked prefill + window
    ("bf16", "bshd", 2, 6, 3, 260, 260, 64, 0, 31, "fixed", False, False, None),         # sliding window, d64
    ("bf16", "bhsd", 3, 4, 4, 200, 900, 64, None, -1, "klens", True, True, None),        # ONNX seqlens_k as given
    ("f16", "bshd", 2, 4, 2, 150, 400, 256, None, 37, "klens", True, False, "b11k"),     # head_dim 256 + mask
    ("f32", "bshd", 2, 2, 1, 70, 90, 32, 5, 9, "fixed", True, True, None),               # CUDA-core float32
    ("f16", "bhsd", 1, 4, 2, 129, 129, 96, None, 0, "fixed", False, False, None),        # window 0, generic path
]


@pytest.mark.parametrize("i", range(len(VIS)))
def test_visibility_variants(i):
    dtype, layout, B, H, G, Sq, Sk, D, off, w, align, use_lens, last, mk = VIS[i]
    r = np.random.default_rng(700 + i)
    k_lens = None
    if use_lens:
        counts = r.integers(Sq, Sk + 1, size=B).astype(np.int32)
        counts[0] = Sk
        k_lens = counts - 1 if last else counts
    mask = None
    if mk is not None:
        mask = r.standard_normal((B, 1, 1, Sk)).astype(np.float32)
        mask[r.random(mask.shape) < 0.1] = -np.inf
    c = wl.make_case(name=f"vis{i}", seed=800 + i, dtype=dtype, layout=layout, batch=B, heads=H, kv_heads=G,
                     q_len=Sq, k_len=Sk, head_dim=D, causal=True, causal_offset=off, k_lens=k_lens, mask=mask,
                     window_left=None if w < 0 else w, causal_align=align,
                     k_lens_kind="last_index" if last else "count")
    run_and_compare(c)


def test_window_zero_returns_the_diagonal_value_exactly_on_the_tensor_core_path():
    B, H, S, D = 2, 4, 300, 128
    c = wl.make_case(name="win0", seed=91, dtype="bf16", layout="bhsd", batch=B, heads=H, q_len=S, head_dim=D,
                     causal=True, causal_offset=0, window_left=0)
    g = GpuCase(c).run()
    _, _, raw = g.outputs()
    assert np.array_equal(raw, c.v.reshape(B, H, S, D))


@pytest.mark.parametrize("D", [128, 64])
def test_decode_sliding_window_and_last_index_lengths(D):
    B, H, G, cap, w = 4, 16, 4, 3000, 700
    r = np.random.default_rng(41 + D)
    counts = r.integers(1, cap + 1, size=B).astype(np.int32)
    counts[0] = 5
    c = wl.make_case(name=f"decwin{D}", seed=43 + D, dtype="bf16", batch=B, heads=H, kv_heads=G, q_len=1,
                     k_len=cap, head_dim=D, k_lens=counts - 1, decode=True, causal=True, window_left=w,
                     causal_align="klens", k_lens_kind="last_index")
    run_and_compare(c)


# ---- score transforms: soft-capping and the softmax sink ----------------------------------------

TRANSFORMS = [
    # dtype, layout, B, H, G, Sq, Sk, D, causal offset (None: not causal), softcap, sink, mask
    ("bf16", "bhsd", 2, 8, 2, 300, 300, 128, 0, 1.0, "heads", None),        # head_dim 128, cap + sink
    ("bf16", "bshd", 2, 6, 3, 200, 333, 64, None, 2.0, "none", "b11k"),      # head_dim 64, cap + mask
    ("f16", "bshd", 2, 4, 2, 150, 400, 256, -60, 0.0, "smooth", "b11k"),     # head_dim 256, smooth softmax,
                                                                             # first rows see no key
    ("f16", "bshd", 1, 4, 4, 129, 300, 256, None, 1.5, "heads", None),       # head_dim 256, cap + sink
    ("bf16", "bshd", 2, 4, 2, 260, 300, 256, None, 2.0, "none", "b11k"),     # head_dim 256 pairs, cap + mask
    ("f32", "bshd", 2, 2, 1, 70, 90, 32, 3, 2.0, "heads", "bhqk"),           # CUDA-core float32
    ("f16", "bhsd", 1, 4, 2, 129, 129, 96, 0, 0.0, "heads", None),           # CUDA-core half path
]


def transform_case(i, spec, decode=False):
    dtype, layout, B, H, G, Sq, Sk, D, off, cap, sink, mk = spec
    r = np.random.default_rng(900 + i)
    mask = None
    if mk is not None:
        shape = {"b11k": (B, 1, 1, Sk), "bhqk": (B, H, Sq, Sk)}[mk]
        mask = r.standard_normal(shape).astype(np.float32)
        mask[r.random(shape) < 0.1] = -np.inf
    head_sink = (r.standard_normal(H) * 2).astype(np.float32) if sink == "heads" else None
    k_lens = r.integers(1, Sk + 1, size=B).astype(np.int32) if decode else None
    return wl.make_case(name=f"tf{i}", seed=950 + i, dtype=dtype, layout=layout, batch=B, heads=H, kv_heads=G,
                        q_len=Sq, k_len=Sk, head_dim=D, causal=off is not None, causal_offset=off, mask=mask,
                        mask_kind=mk or "b11k", softcap=cap, smooth_softmax=sink == "smooth",
                        head_sink=head_sink, k_lens=k_lens, decode=decode)


@pytest.mark.parametrize("i", range(len(TRANSFORMS)))
def test_softcap_and_sink(i):
    st, _ = run_and_compare(transform_case(i, TRANSFORMS[i]))
    assert st["nan_rows"] == 0      # with a sink a row without keys gives O = 0, not NaN


PAIRED = [
    # dtype, B, H, G, Sq, Sk, D, causal offset (None: not causal), mask kind, sink: q_len <= 128 with two or
    # more query heads a kv head, so a CTA takes two heads of one kv head (one query tile each)
    ("bf16", 2, 6, 2, 100, 700, 128, 600, "bhqk", True),    # three heads a group: the last pair has one
    ("f16", 1, 8, 2, 128, 1000, 64, None, "b11k", False),    # q_len exactly one tile, staged mask
    ("bf16", 3, 4, 2, 1, 300, 128, None, None, True),        # one query row, key lengths below
    ("bf16", 1, 4, 1, 129, 400, 64, 0, None, False),         # q_len 129: two tiles of one head (not paired)
    ("f16", 2, 6, 2, 100, 700, 256, 600, "bhqk", True),     # head_dim 256: the CTA pair takes two heads; odd count
    ("bf16", 1, 4, 2, 128, 300, 256, None, "b11k", False),   # head_dim 256, staged mask
]


@pytest.mark.parametrize("i", range(len(PAIRED)))
def test_paired_query_heads(i):
    dtype, B, H, G, Sq, Sk, D, off, mk, sink = PAIRED[i]
    r = np.random.default_rng(1500 + i)
    mask = None
    if mk is not None:
        shape = {"bhqk": (B, H, Sq, Sk), "b11k": (B, 1, 1, Sk)}[mk]
        mask = r.standard_normal(shape).astype(np.float32)
        mask[r.random(shape) < 0.1] = -np.inf
    k_lens = r.integers(1, Sk + 1, size=B).astype(np.int32)
    head_sink = (r.standard_normal(H) * 2).astype(np.float32) if sink else None
    c = wl.make_case(name=f"pair{i}", seed=1550 + i, dtype=dtype, layout="bshd", batch=B, heads=H, kv_heads=G,
                     q_len=Sq, k_len=Sk, head_dim=D, causal=off is not None, causal_offset=off, mask=mask,
                     mask_kind=mk or "b11k", k_lens=k_lens, head_sink=head_sink)
    run_and_compare(c)


NEG_SCALE = [
    # head_dim, mask, segment starts: the transformed-score instantiations of the
    # tensor-core kernels without a softcap (a scale that is not positive)
    (64, False, False),
    (128, True, False),
    (256, True, False),
    (256, False, True),     # segment starts: the single-CTA head_dim-256 kernel
]


@pytest.mark.parametrize("i", range(len(NEG_SCALE)))
def test_negative_scale_takes_the_transform_path(i):
    D, masked, segs = NEG_SCALE[i]
    B, H, G, Sq, Sk = 2, 4, 2, 200, 260
    r = np.random.default_rng(1300 + i)
    mask = None
    if masked:
        mask = r.standard_normal((B, 1, 1, Sk)).astype(np.float32)
        mask[r.random(mask.shape) < 0.1] = -np.inf
    seg = np.repeat(np.arange(0, Sq, 50), 50).astype(np.int32)[None, :].repeat(B, 0) if segs else None
    c = wl.make_case(name=f"neg{i}", seed=1350 + i, dtype="bf16", layout="bhsd", batch=B, heads=H, kv_heads=G,
                     q_len=Sq, k_len=Sk, head_dim=D, scale=-0.05, causal=True, causal_offset=Sk - Sq, mask=mask,
                     seg=seg)
    run_and_compare(c)


DECODE_TF = [
    # dtype, layout, B, H, G, Sq, Sk (capacity), D, offset, softcap, sink, mask
    ("bf16", "bshd", 3, 16, 4, 1, 2000, 128, None, 1.5, "heads", "b11k"),   # tensor-core split pass
    ("f16", "bshd", 2, 8, 2, 1, 900, 64, None, 0.0, "smooth", None),        # generic split pass
    ("bf16", "bshd", 2, 6, 3, 1, 100, 64, None, 2.0, "heads", None),        # one key range, generic pass
]


@pytest.mark.parametrize("i", range(len(DECODE_TF)))
def test_decode_softcap_and_sink(i):
    run_and_compare(transform_case(100 + i, DECODE_TF[i], decode=True))


@pytest.mark.parametrize("int8", [False, True])
def test_decode_result_does_not_depend_on_what_the_workspace_held(int8):
    """Every partial the merge reads is written by the same call: a workspace
    full of 0xFF bytes (NaN floats), the same workspace reused by the next
    call, and one full of zeros all give the oracle's result, with key
    lengths of 0 and 1 among the rows."""
    torch = torch_mod()
    kw = dict(kv_dtype="i8") if int8 else {}
    c = wl.make_case(name="wsre", seed=1401, dtype="bf16", batch=5, heads=16, kv_heads=4, q_len=1, k_len=3000,
                     head_dim=128, k_lens=np.array([3000, 1, 0, 1777, 2999], dtype=np.int32), decode=True, **kw)
    ref_o, ref_l = oracle_full(c)
    g = GpuCase(c, lse=True)
    need = attn.attn_decode_workspace_size(g.prob)
    g.ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    g.ws_bytes = need
    for fill in (None, None, 0):
        if fill is not None:
            g.ws.fill_(fill)
        g.run()
        o, l, _ = g.outputs()
        g.check_guards()
        compare(o, l, ref_o, ref_l, "bf16", "nan", c.name)
        assert attn.attn_device_status() == attn.ATTN_OK


def test_decode_single_range_generic_pass():
    """A cache of at most 128 keys is one key range; the generic pass writes its
    partial result for the combine like any other range."""
    c = wl.make_case(name="dec1r", seed=977, dtype="f16", batch=3, heads=4, kv_heads=2, q_len=1, k_len=96,
                     head_dim=64, k_lens=np.array([96, 1, 50], dtype=np.int32), decode=True)
    run_and_compare(c)


# ---- int8 key/value caches ------------------------------------------------------------------------

INT8 = [
    # dtype, B, H, G, cap, D, scale kind, mask, extras
    ("bf16", 4, 32, 8, 3000, 128, "channel", False, {}),                                   # tensor-core pass
    ("f16", 3, 16, 16, 1500, 128, "tensor", True, {}),                                     # one head per group
    ("bf16", 2, 40, 2, 2100, 128, "channel", False, dict(softcap=2.0, head_sink="heads",
                                                          window_left=700)),               # with transforms
    ("bf16", 2, 8, 2, 900, 64, "channel", True, {}),                                       # generic pass
    ("bf16", 3, 64, 8, 1200, 128, "channel", True, {}),                                    # 8 heads: one MMA column tile
    ("f16", 2, 64, 4, 2500, 128, "tensor", False, {}),                                     # 16 heads: two column tiles
]


@pytest.mark.parametrize("i", range(len(INT8)))
def test_decode_int8_cache(i):
    dtype, B, H, G, cap, D, kind, use_mask, extra = INT8[i]
    r = np.random.default_rng(1100 + i)
    k_lens = r.integers(1, cap + 1, size=B).astype(np.int32)
    mask = None
    if use_mask:
        mask = r.standard_normal((B, 1, 1, cap)).astype(np.float32)
        mask[r.random(mask.shape) < 0.15] = -np.inf
    extra = dict(extra)
    if extra.get("head_sink") == "heads":
        extra["head_sink"] = (r.standard_normal(H) * 2).astype(np.float32)
    if "window_left" in extra:
        extra.update(causal=True, causal_align="klens")
    c = wl.make_case(name=f"q8_{i}", seed=1200 + i, dtype=dtype, batch=B, heads=H, kv_heads=G, q_len=1, k_len=cap,
                     head_dim=D, k_lens=k_lens, mask=mask, decode=True, kv_dtype="i8", kv_scale=kind, **extra)
    run_and_compare(c)


def test_prefill_int8_cache_generic_path():
    c = wl.make_case(name="q8_prefill", seed=1300, dtype="bf16", layout="bhsd", batch=2, heads=4, kv_heads=2,
                     q_len=70, k_len=150, head_dim=64, causal=True, k_lens=np.array([150, 90], dtype=np.int32),
                     kv_dtype="i8", kv_scale="channel")
    run_and_compare(c)


# ---- decode with the cache append fused in --------------------------------------------------------

APPEND = [
    # dtype, B, H, G, cap, D, kv_dtype, k_lens_kind
    ("bf16", 4, 32, 8, 2500, 128, None, "count"),          # tensor-core pass
    ("f16", 3, 8, 2, 700, 64, None, "last_index"),         # CUDA-core pass
    ("bf16", 3, 16, 4, 2000, 128, "i8", "count"),          # int8 tensor-core pass (quantised append)
    ("f16", 2, 6, 3, 500, 64, "i8", "last_index"),         # int8 CUDA-core pass
]


@pytest.mark.parametrize("i", range(len(APPEND)))
def test_decode_with_cache_append(i):
    """attn_decode_append writes each entry's new K/V row at its last valid
    position (bit-exact against the oracle's append, int8 codes included) and
    attends over the updated cache (parity with the oracle on that cache)."""
    torch = torch_mod()
    dtype, B, H, G, cap, D, kv, kind = APPEND[i]
    r = np.random.default_rng(1400 + i)
    counts = r.integers(1, cap + 1, size=B).astype(np.int32)
    counts[0] = cap
    stored = counts - 1 if kind == "last_index" else counts
    c = wl.make_case(name=f"app{i}", seed=1500 + i, dtype=dtype, batch=B, heads=H, kv_heads=G, q_len=1, k_len=cap,
                     head_dim=D, k_lens=stored, k_lens_kind=kind, decode=True, kv_dtype=kv, kv_scale="channel",
                     nan_fill=False)
    new = wl.to_storage(r.standard_normal((2, B, G, D)).astype(np.float32), dtype)
    kn, vn = new[0], new[1]
    g = GpuCase(c)
    dk_new, dv_new = (torch.from_numpy(x.view(np.int16) if x.dtype == np.uint16 else x).cuda() for x in (kn, vn))
    need = attn.attn_decode_workspace_size(g.prob)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    rc = attn.attn_decode_append(g.prob, g.q.data_ptr(), dk_new.data_ptr(), dv_new.data_ptr(), g.k.data_ptr(),
                                 g.v.data_ptr(), g.o.data_ptr(), None, g.k_lens.data_ptr(), g.lse.data_ptr(),
                                 ws.data_ptr(), need, st)
    assert rc == attn.ATTN_OK, attn.status_string(rc)
    torch.cuda.synchronize()
    k2, v2 = oracle.append_rows(c.problem, c.k, c.v, kn, vn, stored, k_scale=c.k_scale, v_scale=c.v_scale)
    if kv is None:
        gk, gv = host_storage(g.k, dtype), host_storage(g.v, dtype)
    else:
        gk, gv = g.k.cpu().numpy(), g.v.cpu().numpy()
    assert np.array_equal(gk, k2.reshape(gk.shape)) and np.array_equal(gv, v2.reshape(gv.shape))
    o, lse, _ = g.outputs()
    ref_o, ref_l = oracle.attn(c.problem, c.q, k2, v2, k_lens=stored, k_scale=c.k_scale, v_scale=c.v_scale)
    compare(o, lse, ref_o.reshape(o.shape), ref_l.reshape(lse.shape), dtype, "nan", f"append{i}")
    assert attn.attn_device_status() == attn.ATTN_OK


def test_ex2_probe_runs_and_keeps_its_chains_bounded():
    """The exponential-throughput probe: every chain x <- -2^x stays in
    [-1, -0.5], so each CTA's sum of 256 threads x 8 chains lies in
    [-2048, -1024]."""
    torch = torch_mod()
    sink = torch.full((8,), float("nan"), dtype=torch.float32, device="cuda")
    assert attn.attn_probe_ex2(8, 64, sink.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    s = sink.cpu().numpy()
    assert np.all(np.isfinite(s)) and np.all(s >= -2048.0) and np.all(s <= -1024.0)


@pytest.mark.parametrize("per_row", [False, True])
@pytest.mark.parametrize("D,dtype,causal", [(128, "bf16", False), (128, "f16", True), (64, "bf16", True),
                                             (256, "f16", False), (256, "bf16", True)])
def test_scores_rising_far_above_the_reference_maximum(D, dtype, causal, per_row):
    """Scores that jump well above a row's reference maximum after its first
    key tiles: by 43 log2 units (P up to 2^43 in bf16 kept without a rescale; in
    f16, past 2^15, the tile is redone), by 87
    and 88 (the tile is redone with its maximum), and to +inf at one key (a
    NaN row).  All against the oracle; the same values also as a mask with a
    row per query ([B,H,Q,K], read from global memory, reloaded on a redo)."""
    B, H, Sq, Sk = 3, 4, 256, 640
    r = np.random.default_rng(77 + D)
    mask = (r.standard_normal((B, 1, 1, Sk)) * 0.5).astype(np.float32)
    mask[0, 0, 0, 200:] += 30.0
    mask[1, 0, 0, 300:] += 60.0
    mask[1, 0, 0, 500:] += 1.0
    mask[2, 0, 0, 150:] += 20.0
    mask[2, 0, 0, 400] = np.inf
    kind = "b11k"
    if per_row:
        mask = np.ascontiguousarray(np.broadcast_to(mask, (B, H, Sq, Sk)))
        kind = "bhqk"
    c = wl.make_case(name=f"rise{D}", seed=88, dtype=dtype, batch=B, heads=H, q_len=Sq, k_len=Sk, head_dim=D,
                     causal=causal, causal_offset=Sk - Sq if causal else None, mask=mask, mask_kind=kind)
    st, _ = run_and_compare(c)
    assert st["nan_rows"] == H * (Sq if not causal else Sq - (400 - (Sk - Sq)))


MIXED = [
    # dtype, B, H, G, cap, lens kind, extras
    ("bf16", 37, 40, 2, 3000, "mixed", {}),                                   # 20 heads a group: two head blocks
    ("f16", 200, 8, 8, 700, "short", {}),                                      # many short rows
    ("bf16", 5, 32, 8, 9000, "mixed", dict(softcap=30.0, head_sink="heads")),  # transforms, long rows
    ("bf16", 64, 16, 4, 1500, "zeros", {}),                                    # most entries without a key
]


@pytest.mark.parametrize("i", range(len(MIXED)))
def test_decode_mixed_key_lengths(i):
    """The tensor-core decode pass over batches whose entries hold zero, few and
    many keys (empty ranges, ranges cut short, rows over many ranges), with
    one or two blocks of query heads per kv head, against the oracle (O and
    LSE)."""
    dtype, B, H, G, cap, kind, extra = MIXED[i]
    r = np.random.default_rng(1600 + i)
    if kind == "mixed":
        k_lens = r.integers(0, cap + 1, size=B)
        k_lens[: max(1, B // 8)] = 0
        k_lens[-1] = cap
    elif kind == "short":
        k_lens = r.integers(1, 200, size=B)
    else:
        k_lens = np.where(r.random(B) < 0.8, 0, r.integers(1, cap + 1, size=B))
    extra = dict(extra)
    if extra.get("head_sink") == "heads":
        extra["head_sink"] = (r.standard_normal(H) * 2).astype(np.float32)
    c = wl.make_case(name=f"bal{i}", seed=1700 + i, dtype=dtype, batch=B, heads=H, kv_heads=G, q_len=1, k_len=cap,
                     head_dim=128, k_lens=k_lens.astype(np.int32), decode=True, **extra)
    run_and_compare(c)
