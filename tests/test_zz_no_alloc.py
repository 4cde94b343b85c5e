"""attn_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (it keeps its partial results in a fixed device array
of the library instead of a caller workspace).  Checked through the C ABI
against attn_decode with a caller workspace, on two calls in a row.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
from __future__ import annotations

import numpy as np
import pytest

from attention_attn_fwd_02_gb300 import attn, build
from attention_attn_fwd_02_gb300 import workloads as wl
from gpu_util import HALF_ABS, LSE_ABS, GpuCase, torch_mod

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = torch_mod()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    attn.lib()


def run_noalloc(g: GpuCase, o, lse):
    torch = torch_mod()
    ptr = (lambda t: None if t is None else t.data_ptr())
    rc = attn.attn_decode_noalloc(g.prob, ptr(g.q), ptr(g.k), ptr(g.v), o.data_ptr(), ptr(g.mask), ptr(g.seg),
                                  ptr(g.k_lens), lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == attn.ATTN_OK, attn.status_string(rc)
    torch.cuda.synchronize()


def close(a, b, tol):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(a), np.isnan(b))
    f = np.isfinite(b)
    assert np.all(np.abs(a[f] - b[f]) <= tol)


@pytest.mark.parametrize("shape", [dict(batch=4, capacity=1024, heads=32, kv_heads=8, min_len=1),
                                   dict(batch=3, capacity=5000, heads=8, kv_heads=2, min_len=1)])
def test_noalloc_matches_workspace_decode_twice(shape):
    torch = torch_mod()
    case = wl.decode_bnsh_bf16(seed=9, **shape)
    g = GpuCase(case, lse=True).run()          # existing entry point, caller workspace
    torch.cuda.synchronize()
    ref_o, ref_l = g.o.clone(), g.lse.clone()
    for _ in range(2):                          # two calls in a row share the fixed array
        o = torch.full_like(g.o, -4096.0)
        lse = torch.full_like(g.lse, 777.0)
        run_noalloc(g, o, lse)
        close(o, ref_o, HALF_ABS)
        close(lse, ref_l, LSE_ABS)
    assert attn.attn_device_status() == attn.ATTN_OK


def test_noalloc_rejects_problems_beyond_its_array():
    big = attn.make_problem(dict(batch=4096, heads=64, kv_heads=8, q_len=1, k_len=65536, head_dim=128, dtype="bf16",
                                 q_layout=(0, 64 * 128, 128, 64 * 128), k_layout=(0, 8 * 65536 * 128, 65536 * 128, 128),
                                 v_layout=(0, 8 * 65536 * 128, 65536 * 128, 128), o_layout=(0, 64 * 128, 128, 64 * 128)))
    assert attn.attn_decode_workspace_size(big) > attn.attn_decode_noalloc_max_scratch()
    fake = 0x10000  # never dereferenced: the size check rejects the call before any launch
    rc = attn.attn_decode_noalloc(big, fake, fake, fake, fake, None, None, None, None, None)
    assert rc == attn.ATTN_ERR_WORKSPACE
