"""Structural properties of the CUDA path that hold whatever the values:
bounded waits that run out report a status and leave the context usable;
keys hidden from a whole query block are never read; permuting hidden keys
changes nothing; the staged broadcast-mask path at batch > 1 with special
mask values.  All through the C ABI, against the float64 oracle where a
value is compared.

"Attention" (recursiveai.org OneGPU docs), section "Special values": a hidden
key has weight zero and V is not inspected; section "Long calls" and the
bounded-wait contract of this library: a wait that cannot finish ends with a
status, never a hang.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from attention_attn_fwd_02_gb300 import attn, build
from attention_attn_fwd_02_gb300 import workloads as wl
from gpu_util import GpuCase, compare, oracle_full, torch_mod

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = torch_mod()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    attn.lib()
    yield
    attn.attn_test_inject(attn.ATTN_INJECT_NONE)


# ---- bounded waits ---------------------------------------------------------------------------

TIMEOUT_CASES = {
    "prefill_d128": lambda: wl.long_causal_gqa_bf16(seed=71, batch=1, seq=640, heads=4, kv_heads=2),
    "prefill_d64": lambda: wl.make_case(name="to64", seed=72, dtype="bf16", batch=2, heads=4, kv_heads=2,
                                        q_len=300, head_dim=64, causal=True),
    "prefill_d256": lambda: wl.make_case(name="to256", seed=73, dtype="f16", batch=1, heads=2, q_len=200,
                                         k_len=600, head_dim=256),
    # segment starts route head_dim 256 to the single-CTA kernel
    "prefill_d256_segments": lambda: wl.make_case(
        name="to256s", seed=74, dtype="bf16", batch=1, heads=2, q_len=300, head_dim=256, causal=True,
        causal_offset=0, seg=np.repeat(np.arange(0, 300, 100), 100).astype(np.int32)[None, :]),
    "decode_bf16": lambda: wl.decode_bnsh_bf16(seed=77, batch=2, capacity=1024, heads=8, kv_heads=2, min_len=600),
    "decode_int8": lambda: wl.make_case(name="to_q8", seed=78, dtype="bf16", batch=2, heads=8, kv_heads=2, q_len=1,
                                        k_len=2000, head_dim=128, k_lens=np.array([1500, 2000], dtype=np.int32),
                                        decode=True, kv_dtype="i8", kv_scale="channel"),
}


@pytest.mark.parametrize("name", list(TIMEOUT_CASES))
def test_bounded_wait_reports_timeout_and_context_stays_usable(name):
    """The one-shot test fault makes the first CTA announce its first key copy
    without issuing it: that CTA's waits run out (about 2 s), it records
    ATTN_ERR_DEVICE_TIMEOUT, waits for what it did start, frees its tensor
    memory and exits.  The status word reads the timeout once, then clears;
    the next call on the same context is correct."""
    c = TIMEOUT_CASES[name]()
    assert attn.attn_device_status() == attn.ATTN_OK
    assert attn.attn_test_inject(attn.ATTN_INJECT_DROP_FIRST_COPY) == attn.ATTN_OK
    g = GpuCase(c).run()
    torch_mod().cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_ERR_DEVICE_TIMEOUT
    assert attn.attn_device_status() == attn.ATTN_OK      # read once, then cleared
    g.run()                                                # the fault was one-shot
    o, lse, _ = g.outputs()
    g.check_guards()
    ref_o, ref_l = oracle_full(c)
    compare(o, lse, ref_o, ref_l, c.problem["dtype"], c.problem["masked_rows"], name)
    assert attn.attn_device_status() == attn.ATTN_OK


# ---- keys hidden from a whole query block are never read -------------------------------------


def row_ranges(case):
    """Visible key range [lo, hi) of every (batch, row): the page's rules (key length,
    causal bound with its window, segment start), written out here independently."""
    p = case.problem
    B, Sq, Sk = p["batch"], p["q_len"], p["k_len"]
    off = Sk - Sq if p["causal_offset"] is None else p["causal_offset"]
    lo = np.zeros((B, Sq), dtype=np.int64)
    hi = np.full((B, Sq), Sk, dtype=np.int64)
    for b in range(B):
        if case.k_lens is not None:
            hi[b] = min(max(int(case.k_lens[b]), 0), Sk)
        for q in range(Sq):
            if p["causal"]:
                d = q + off
                hi[b, q] = max(0, min(hi[b, q], d + 1))
                if p.get("window_left") is not None:
                    lo[b, q] = max(lo[b, q], d - p["window_left"])
            if case.seg is not None:
                lo[b, q] = max(lo[b, q], min(max(int(case.seg[b, q]), 0), Sk))
    return lo, np.maximum(hi, lo)


def nan_fill_keys(case, b, keys):
    """Set K and V of batch entry b at the given keys to NaN (position-first storage)."""
    dt = case.problem["dtype"]
    bits = {"f16": 0x7E00, "bf16": 0x7FC0}[dt]
    k = case.k.reshape(case.problem["batch"], case.problem["k_len"], -1).copy()
    v = case.v.reshape(k.shape).copy()
    k[b, keys] = bits
    v[b, keys] = bits
    case.k, case.v = k.reshape(case.k.shape), v.reshape(case.v.shape)


STRUCT = [
    # name, head_dim, rows a query block holds on the tensor-core path, extra problem fields, NaN keys of entry 0
    ("causal_d128", 128, 256, dict(causal=True, causal_offset=0), (600, 768)),
    ("segments_d128", 128, 256, dict(causal=True, causal_offset=0, seg="docs"), (0, 256)),
    ("window_d64", 64, 256, dict(causal=True, causal_offset=0, window_left=64), (0, 384)),
    ("segments_d256", 256, 128, dict(causal=True, causal_offset=0, seg="docs"), (0, 256)),
    ("window_d256", 256, 128, dict(causal=True, causal_offset=0, window_left=100), (0, 300)),
]


@pytest.mark.parametrize("i", range(len(STRUCT)))
def test_keys_hidden_from_a_whole_query_block_are_never_read(i):
    """K/V of keys that every row of a query block hides (by the causal bound,
    a window or a segment start) are NaN: rows of blocks whose visible ranges
    avoid them match the oracle; rows that see them are NaN (the oracle's
    answer too); rows that hide them but share a block with a row that sees
    them are NaN or match the oracle, and are NaN within the same 128-row
    query tile (the documented limit of a tensor-core P V: it multiplies the
    hidden V row by zero, and 0 * NaN = NaN)."""
    name, D, block, extra, (a, b_) = STRUCT[i]
    S, B, H = 768, 2, 4
    extra = dict(extra)
    seg = None
    if extra.pop("seg", None) == "docs":
        seg = np.zeros((B, S), dtype=np.int32)
        seg[:, 300:] = 300          # documents [0, 300) and [300, 768)
    c = wl.make_case(name=name, seed=300 + i, dtype="bf16" if D != 256 else "f16", layout="bshd", batch=B,
                     heads=H, kv_heads=2, q_len=S, head_dim=D, seg=seg, **extra)
    nan_fill_keys(c, 0, slice(a, b_))
    g = GpuCase(c).run()
    o, lse, _ = g.outputs()
    g.check_guards()
    ref_o, ref_l = oracle_full(c)
    lo, hi = row_ranges(c)
    dtype = c.problem["dtype"]
    sees = np.zeros((B, S), dtype=bool)
    sees[0] = (lo[0] < b_) & (hi[0] > a) & (hi[0] > lo[0])
    ok_rows, may_rows, tile_rows = [], [], []
    for bb in range(B):
        for q0 in range(0, S, block):
            rows = np.arange(q0, min(q0 + block, S))
            live = rows[hi[bb, rows] > lo[bb, rows]]
            hit = len(live) > 0 and bb == 0 and lo[bb, live].min() < b_ and hi[bb, live].max() > a
            for q in rows:
                if sees[bb, q]:
                    continue
                if not hit:
                    ok_rows.append((bb, q))
                    continue
                t0 = q0 + (q - q0) // 128 * 128          # the row's 128-row query tile
                (tile_rows if sees[bb, t0:t0 + 128].any() else may_rows).append((bb, q))
    assert ok_rows and sees.any() and tile_rows

    def pick(rows):
        r = np.array(rows, dtype=np.int64).reshape(-1, 2)
        return r[:, 0], r[:, 1]

    bi, qi = pick(ok_rows)
    compare(o[bi, :, qi], lse[bi, :, qi], ref_o[bi, :, qi], ref_l[bi, :, qi], dtype, "nan", f"{name} clean blocks")
    assert np.all(np.isnan(o[0, :, sees[0]])) and np.all(np.isnan(ref_o[0, :, sees[0]]))
    bi, qi = pick(tile_rows)
    assert np.all(np.isnan(o[bi, :, qi])), f"{name}: rows sharing a query tile with a NaN key they hide"
    for bb, q in may_rows:
        got = o[bb, :, q]
        if not np.all(np.isnan(got)):
            compare(got[None], lse[bb, :, q][None], ref_o[bb, :, q][None], ref_l[bb, :, q][None], dtype, "nan",
                    f"{name} row {q}")


def test_hidden_key_permutation_changes_nothing():
    """Permuting K/V among keys beyond each entry's key length, and swapping the
    K/V rows of keys whose broadcast mask is -inf, leaves every output bit the
    same (head_dim 64, 128 and 256 tensor-core kernels)."""
    for D, dt in ((64, "bf16"), (128, "bf16"), (256, "f16")):
        B, H, Sq, Sk = 2, 4, 300, 700
        r = np.random.default_rng(91 + D)
        k_lens = np.array([520, 700], dtype=np.int32)
        mask = r.standard_normal((B, 1, 1, Sk)).astype(np.float32)
        hidden = [np.sort(r.choice(k_lens[b], size=40, replace=False)) for b in range(B)]
        for b in range(B):
            mask[b, 0, 0, hidden[b]] = -np.inf
        c = wl.make_case(name=f"perm{D}", seed=95 + D, dtype=dt, layout="bshd", batch=B, heads=H, kv_heads=2,
                         q_len=Sq, k_len=Sk, head_dim=D, k_lens=k_lens, mask=mask, nan_fill=False)
        _, l1, o1 = GpuCase(c).run().outputs()
        k = c.k.reshape(B, Sk, -1).copy()
        v = c.v.reshape(B, Sk, -1).copy()
        for b in range(B):
            tail = np.arange(k_lens[b], Sk)
            if len(tail) > 1:
                pi = r.permutation(tail)
                k[b, tail], v[b, tail] = k[b, pi], v[b, pi]
            hb = hidden[b]
            k[b, hb], v[b, hb] = k[b, hb[::-1]], v[b, hb[::-1]]
        c.k, c.v = k.reshape(c.k.shape), v.reshape(c.v.shape)
        _, l2, o2 = GpuCase(c).run().outputs()
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2, equal_nan=True), f"head_dim {D}"


# ---- broadcast masks staged in shared memory, batch > 1, special values ----------------------

BCAST = [
    # head_dim, batch, k_len (a multiple of 4, not of 128), key lengths below k_len
    (128, 3, 708, True),
    (64, 2, 516, True),
    (128, 2, 260, False),
]


@pytest.mark.parametrize("i", range(len(BCAST)))
def test_staged_broadcast_mask_batches_and_special_values(i):
    """A [B,1,1,K] mask takes the staged (bulk-copied) path when its rows are
    16-byte aligned and k_len is a multiple of 4: every batch entry reads its
    own row (nonzero batch stride), the last key tile is partial, key lengths
    cut rows short, and NaN / +inf / -inf entries give NaN rows, NaN rows and
    hidden keys."""
    D, B, Sk, lens = BCAST[i]
    H, Sq = 4, 200
    r = np.random.default_rng(1900 + i)
    mask = r.standard_normal((B, 1, 1, Sk)).astype(np.float32)
    mask[r.random(mask.shape) < 0.1] = -np.inf
    mask[1, 0, 0, Sk - 5] = np.nan           # the partial last tile: entry 1's rows that see it are NaN
    mask[0, 0, 0, Sk - 100] = np.inf         # entry 0: rows 100.. see it and are NaN
    mask[B - 1, 0, 0, :Sk // 2] = -np.inf    # the last entry: its first half hidden
    k_lens = None
    if lens:
        k_lens = np.full(B, Sk, dtype=np.int32)
        k_lens[1] = Sk - 7                   # entry 1's NaN entry lies beyond its length: never read
        k_lens[0] = Sk - 60
    c = wl.make_case(name=f"bcast{i}", seed=1950 + i, dtype="bf16", layout="bhsd", batch=B, heads=H, kv_heads=2,
                     q_len=Sq, k_len=Sk, head_dim=D, k_lens=k_lens, mask=mask, mask_kind="b11k",
                     causal=True, causal_offset=Sk - Sq)
    g = GpuCase(c).run()
    o, lse, _ = g.outputs()
    g.check_guards()
    ref_o, ref_l = oracle_full(c)
    st = compare(o, lse, ref_o, ref_l, "bf16", "nan", c.name)
    assert st["nan_rows"] > 0
    assert attn.attn_device_status() == attn.ATTN_OK


@pytest.mark.parametrize("D,causal", [(128, False), (64, True)])
def test_padded_masked_keys_bound_the_key_span(D, causal):
    """A staged [B,1,1,K] mask whose first or last keys are -inf (key padding)
    starts and ends a CTA's key tiles at its first and last keys with another
    value: entry 0 is padded from key 500; entry 1 from key 300 except a NaN at
    key 600 (which keeps its tile: the rows that see it are NaN); entry 2 is
    -inf throughout (fully hidden rows, LSE -inf); entry 3 is padded below key
    400 and from key 650 (under the causal bound its first rows see no key).
    Against the oracle, in both MaskedRows modes."""
    B, H, Sq, Sk = 4, 4, 300, 708
    mask = np.random.default_rng(1950 + D).standard_normal((B, 1, 1, Sk)).astype(np.float32)
    mask[0, 0, 0, 500:] = -np.inf
    mask[1, 0, 0, 300:] = -np.inf
    mask[1, 0, 0, 600] = np.nan
    mask[2] = -np.inf
    mask[3, 0, 0, :400] = -np.inf
    mask[3, 0, 0, 650:] = -np.inf
    for mr in ("nan", "zero"):
        c = wl.make_case(name=f"trim{D}{mr}", seed=1960 + D, dtype="bf16", layout="bhsd", batch=B, heads=H,
                         kv_heads=2, q_len=Sq, k_len=Sk, head_dim=D, mask=mask, mask_kind="b11k", masked_rows=mr,
                         causal=causal, causal_offset=Sk - Sq if causal else None)
        g = GpuCase(c).run()
        o, lse, _ = g.outputs()
        g.check_guards()
        ref_o, ref_l = oracle_full(c)
        st = compare(o, lse, ref_o, ref_l, "bf16", mr, c.name)
        assert st["nan_rows"] > 0
        assert attn.attn_device_status() == attn.ATTN_OK


# ---- key tiles whose broadcast mask is -inf throughout are skipped -------------------------------

DEAD = [
    # head_dim, dtype, batch, q_len, k_len, causal, smooth softmax
    (128, "bf16", 3, 300, 1100, False, False),
    (64, "bf16", 2, 200, 700, True, False),
    (256, "f16", 3, 130, 1000, False, False),
    (256, "f16", 2, 200, 640, False, True),
]


@pytest.mark.parametrize("i", range(len(DEAD)))
def test_fully_masked_key_tiles_match_the_oracle(i):
    """A [B,1,1,K] mask with whole 128-key tiles at -inf (the first, one in the
    middle, the last, partial), a NaN inside an otherwise -inf tile (the tile
    stays: rows that see it are NaN), and one batch entry masked everywhere
    (no tile left: a masked row, or O = 0 with the sink's LSE under smooth
    softmax).  The head_dim-256 kernel skips the tiles of -inf; the result
    matches the oracle on every kernel."""
    D, dt, B, Sq, Sk, causal, smooth = DEAD[i]
    r = np.random.default_rng(2100 + i)
    mask = r.standard_normal((B, 1, 1, Sk)).astype(np.float32)
    mask[r.random(mask.shape) < 0.1] = -np.inf
    mask[0, 0, 0, :128] = -np.inf                # first tile
    mask[0, 0, 0, 384:512] = -np.inf             # a middle tile
    mask[0, 0, 0, (Sk // 128) * 128:] = -np.inf  # the partial last tile
    mask[1, 0, 0, 128:384] = -np.inf             # two tiles ...
    mask[1, 0, 0, 300] = np.nan                  # ... one of which keeps a NaN
    mask[B - 1] = -np.inf                        # the last entry: nothing visible
    c = wl.make_case(name=f"dead{i}", seed=2150 + i, dtype=dt, layout="bshd", batch=B, heads=4, kv_heads=2,
                     q_len=Sq, k_len=Sk, head_dim=D, mask=mask, mask_kind="b11k", causal=causal,
                     causal_offset=Sk - Sq if causal else None, smooth_softmax=smooth)
    g = GpuCase(c).run()
    o, lse, _ = g.outputs()
    g.check_guards()
    ref_o, ref_l = oracle_full(c)
    st = compare(o, lse, ref_o, ref_l, dt, "nan", c.name)
    if not smooth:
        assert st["nan_rows"] >= 4 * Sq        # the last entry at least
    assert attn.attn_device_status() == attn.ATTN_OK


# ---- key ranges merged in range order --------------------------------------------------------------

def _split_mask(seed, B, Sk):
    """N(0,1) mask with 10% of keys -inf and the last batch entry -inf throughout."""
    r = np.random.default_rng(seed)
    m = r.standard_normal((B, 1, 1, Sk)).astype(np.float32)
    m[r.random(m.shape) < 0.1] = -np.inf
    m[B - 1] = -np.inf
    return m


def _with_ranges(case, n):
    case.problem = dict(case.problem, key_splits=n)
    return case


SPLIT = {
    # the causal GQA workload with documents, its keys forced into 4 ranges (many of them empty for a block)
    "gqa_doc_4_ranges": lambda: _with_ranges(wl.gqa_doc_causal_bf16(), 4),
    # 64 queries against 8192 keys: the automatic plan cuts 8 ranges
    "short_query_auto": lambda: wl.short_query_cross_bf16(batch=1, heads=8, kv_heads=2),
    # head_dim 256 with a broadcast mask and a fully masked entry, automatic ranges
    "d256_mask_auto": lambda: wl.make_case(
        name="split256", seed=2201, dtype="f16", layout="bshd", batch=2, heads=4, kv_heads=2, q_len=100, k_len=5000,
        head_dim=256, mask=_split_mask(2202, 2, 5000), mask_kind="b11k", masked_rows="zero"),
    # causal bound right-aligned to per-entry key lengths with a sink, 5 forced ranges
    "causal_klens_sink": lambda: _with_ranges(wl.make_case(
        name="splitks", seed=2204, dtype="bf16", layout="bhsd", batch=3, heads=4, kv_heads=1, q_len=200, k_len=3000,
        head_dim=128, causal=True, causal_align="klens", k_lens=np.array([3000, 1700, 0], dtype=np.int32),
        head_sink=np.array([0.5, -1.0, 2.0, 0.0], dtype=np.float32)), 5),
    # head_dim 64, not causal, key lengths that end some ranges early and leave others empty (their
    # first K and V tiles are copied at kernel entry and must be waited for), a ragged key axis
    "klens_ragged_d64": lambda: wl.make_case(
        name="splitkl", seed=2206, dtype="bf16", layout="bshd", batch=3, heads=4, kv_heads=2, q_len=64, k_len=5000,
        head_dim=64, k_lens=np.array([5000, 2000, 1], dtype=np.int32)),
    # float32 on the CUDA-core path, 3 forced ranges
    "f32_generic": lambda: _with_ranges(wl.make_case(
        name="split32", seed=2205, dtype="f32", batch=1, heads=2, q_len=40, k_len=700, head_dim=32, causal=True), 3),
}


@pytest.mark.parametrize("name", list(SPLIT))
def test_key_ranges_merged_in_range_order_match_the_oracle(name):
    """attn_fwd with its keys cut into ranges: each range's partial (O / l and
    LSE) goes to the workspace and the merge combines them in range order; O
    and LSE match the oracle, NaN / masked rows included."""
    c = SPLIT[name]()
    g = GpuCase(c)
    assert attn.attn_fwd_workspace_size(g.prob) > 0, "the plan should cut this problem into ranges"
    g.run()
    o, lse, _ = g.outputs()
    g.check_guards()
    ref_o, ref_l = oracle_full(c)
    compare(o, lse, ref_o, ref_l, c.problem["dtype"], c.problem["masked_rows"], name)
    assert attn.attn_device_status() == attn.ATTN_OK


def test_key_ranges_with_a_nan_score_make_the_row_nan():
    """A +inf mask entry inside one range makes exactly the rows that see it NaN after the merge."""
    B, H, Sq, Sk = 1, 2, 64, 4096
    mask = np.zeros((B, 1, 1, Sk), dtype=np.float32)
    mask[0, 0, 0, 3000] = np.inf
    c = wl.make_case(name="split_inf", seed=2210, dtype="bf16", layout="bhsd", batch=B, heads=H, q_len=Sq, k_len=Sk,
                     head_dim=64, mask=mask, mask_kind="b11k", causal=True, causal_offset=2990)
    g = GpuCase(c)
    assert attn.attn_fwd_workspace_size(g.prob) > 0
    st, _ = run_split_compare(g, c)
    assert st["nan_rows"] == H * (Sq - 10)


def run_split_compare(g, c):
    g.run()
    o, lse, _ = g.outputs()
    ref_o, ref_l = oracle_full(c)
    return compare(o, lse, ref_o, ref_l, c.problem["dtype"], c.problem["masked_rows"], c.name), g
