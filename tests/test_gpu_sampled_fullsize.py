"""Full-size workloads (the shapes the benchmark times), checked on sampled
rows that the oracle computes one by one, plus properties that hold at any
size (row classes, finite outputs, guard bands untouched)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from attention_attn_fwd_02_gb300 import attn, build
from attention_attn_fwd_02_gb300 import workloads as wl
from gpu_util import GpuCase, compare, torch_mod

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = torch_mod()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    attn.lib()


def sample_rows(case, n=192, seed=7):
    p = case.problem
    B, H, Sq = p["batch"], p["heads"], p["q_len"]
    r = np.random.default_rng(seed)
    rows = [(b, h, i) for b in range(B) for h in (0, H - 1) for i in (0, Sq - 1)]
    if case.k_lens is not None and Sq > 1:
        for b in range(B):
            kl = int(case.k_lens[b])
            for i in (kl - 2, kl - 1, kl, kl + 1):
                if 0 <= i < Sq:
                    rows.append((b, int(r.integers(H)), i))
    while len(rows) < n:
        rows.append((int(r.integers(B)), int(r.integers(H)), int(r.integers(Sq))))
    return np.array(rows, dtype=np.int64)


FULL = {
    "long_causal_gqa_bf16": lambda: wl.long_causal_gqa_bf16(),
    "decode_bnsh_bf16": lambda: wl.decode_bnsh_bf16(),
    "cross_mask_f16_nan": lambda: wl.cross_mask_f16(masked_rows="nan"),
    "cross_mask_f16_zero": lambda: wl.cross_mask_f16(masked_rows="zero"),
    "decode_bnsh_int8": lambda: wl.decode_bnsh_int8(),
    "dense_gqa_bf16": lambda: wl.dense_gqa_bf16(),
    "masked_gqa_bf16": lambda: wl.masked_gqa_bf16(),
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_sampled_rows(name):
    case = FULL[name]()
    g = GpuCase(case).run()
    o, lse, _ = g.outputs()
    g.check_guards()
    assert attn.attn_device_status() == attn.ATTN_OK
    rows = sample_rows(case)
    ref_o, ref_l = oracle.attn(case.problem, case.q, case.k, case.v, mask=case.mask, seg=case.seg,
                               k_lens=case.k_lens, rows=rows, head_sink=case.head_sink,
                               k_scale=case.k_scale, v_scale=case.v_scale)
    got_o = o[rows[:, 0], rows[:, 1], rows[:, 2]]
    got_l = lse[rows[:, 0], rows[:, 1], rows[:, 2]]
    compare(got_o, got_l, ref_o, ref_l, case.problem["dtype"], case.problem["masked_rows"], name)
    # properties over every row: NaN rows exactly where no key is visible (the last batch entry of the
    # masked cross-attention workload), finite everywhere else
    D = o.shape[-1]
    nan_rows = np.all(np.isnan(o.reshape(-1, D)), axis=1)
    if name == "cross_mask_f16_nan":
        B = case.problem["batch"]
        assert np.all(nan_rows.reshape(B, -1)[-1]) and not nan_rows.reshape(B, -1)[:-1].any()
    else:
        assert not nan_rows.any()
        assert np.all(np.isfinite(o))
