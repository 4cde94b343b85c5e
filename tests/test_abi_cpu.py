"""The C ABI without a GPU: the library builds and loads, exports every entry
point include/attn.h declares, its struct layout matches the binding's, and
host-side argument checks return their status codes before touching CUDA."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

from attention_attn_fwd_02_gb300 import attn, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return attn.lib()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_the_binding_exports():
    assert sorted(declared_functions()) == sorted(attn.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", attn.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    syms = set(re.findall(r"\bT\s+(attn_\w+)", out))
    for name in declared_functions():
        assert name in syms, name
        assert hasattr(L, name)


def test_struct_layout_matches_c(tmp_path):
    src = tmp_path / "sz.c"
    src.write_text(f'#include "{HEADER}"\n#include <stdio.h>\n#include <stddef.h>\n'
                   'int main(void){printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(attn_problem),'
                   ' offsetof(attn_problem, causal_offset), offsetof(attn_problem, q),'
                   ' offsetof(attn_problem, mask), offsetof(attn_problem, seg_batch_stride),'
                   ' offsetof(attn_problem, lse_head_stride)); printf("%zu %zu %zu\\n",'
                   ' offsetof(attn_problem, window_left), offsetof(attn_problem, causal_align),'
                   ' offsetof(attn_problem, k_lens_kind)); printf("%zu %zu\\n", offsetof(attn_problem, softcap),'
                   ' offsetof(attn_problem, head_sink)); printf("%zu %zu %zu\\n", offsetof(attn_problem, kv_dtype),'
                   ' offsetof(attn_problem, v_scale), offsetof(attn_problem, key_splits)); return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.run(["gcc", str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    P = attn.attn_problem
    want = [ctypes.sizeof(P), P.causal_offset.offset, P.q.offset, P.mask.offset, P.seg_batch_stride.offset,
            P.lse_head_stride.offset, P.window_left.offset, P.causal_align.offset, P.k_lens_kind.offset,
            P.softcap.offset, P.head_sink.offset, P.kv_dtype.offset, P.v_scale.offset, P.key_splits.offset]
    assert got == want


def base_problem(**kw):
    d = dict(batch=2, heads=4, kv_heads=2, q_len=8, k_len=8, head_dim=64, dtype="bf16",
             q_layout=(0, 8 * 4 * 64, 64, 4 * 64), k_layout=(0, 8 * 2 * 64, 64, 2 * 64),
             v_layout=(0, 8 * 2 * 64, 64, 2 * 64), o_layout=(0, 8 * 4 * 64, 64, 4 * 64))
    d.update(kw)
    return attn.make_problem(d)


FAKE = 0x10000  # never dereferenced: every case below fails on the host first


@pytest.mark.parametrize("kw,code", [
    (dict(kv_heads=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(head_dim=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(head_dim=257), attn.ATTN_ERR_INVALID_ARG),
    (dict(head_dim=63), attn.ATTN_ERR_INVALID_ARG),          # half types need an even head_dim
    (dict(dtype=7), attn.ATTN_ERR_INVALID_ARG),
    (dict(q_len=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(heads=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(q_layout=(0, -1, 64, 256)), attn.ATTN_ERR_INVALID_ARG),
    (dict(causal=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(masked_rows=5), attn.ATTN_ERR_INVALID_ARG),
    (dict(window_left=3), attn.ATTN_ERR_INVALID_ARG),             # a window needs the causal bound
    (dict(window_left=-2, causal=True), attn.ATTN_ERR_INVALID_ARG),
    (dict(causal_align=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(k_lens_kind=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(softcap=-1.0), attn.ATTN_ERR_INVALID_ARG),
    (dict(softcap=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(smooth_softmax=2), attn.ATTN_ERR_INVALID_ARG),
    (dict(head_sink_ptr=FAKE + 2), attn.ATTN_ERR_ALIGNMENT),
    (dict(kv_dtype="i8"), attn.ATTN_ERR_INVALID_ARG),              # int8 K/V need their scales
    (dict(kv_dtype="i8", k_scale_ptr=FAKE, v_scale_ptr=FAKE + 1), attn.ATTN_ERR_ALIGNMENT),
    (dict(kv_dtype=5), attn.ATTN_ERR_INVALID_ARG),
])
def test_fwd_rejects_invalid_problems(L, kw, code):
    p = base_problem(**kw)
    if "causal" in kw:
        p.causal = int(kw["causal"])
    if "masked_rows" in kw:
        p.masked_rows = kw["masked_rows"]
    for name in ("causal_align", "k_lens_kind", "smooth_softmax", "kv_dtype"):
        if isinstance(kw.get(name), int):
            setattr(p, name, kw[name])
    assert attn.attn_fwd(p, FAKE, FAKE, FAKE, FAKE, None, None, None, None, None, 0, None) == code


def test_fwd_null_and_misaligned_pointers(L):
    p = base_problem()
    assert attn.attn_fwd(p, None, FAKE, FAKE, FAKE, None, None, None, None, None, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd(p, FAKE, FAKE, FAKE, None, None, None, None, None, None, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd(p, FAKE + 1, FAKE, FAKE, FAKE, None, None, None, None, None, 0, None) == attn.ATTN_ERR_ALIGNMENT
    assert attn.attn_fwd(p, FAKE, FAKE, FAKE, FAKE, FAKE + 2, None, None, None, None, 0, None) == attn.ATTN_ERR_ALIGNMENT


def test_empty_problems_are_noops(L):
    assert attn.attn_fwd(base_problem(batch=0), None, None, None, None, None, None, None, None, None, 0, None) == 0
    assert attn.attn_fwd(base_problem(q_len=0), None, None, None, None, None, None, None, None, None, 0, None) == 0


def test_decode_checks(L):
    p = base_problem(q_len=2)
    assert attn.attn_decode_workspace_size(p) == 0
    assert attn.attn_decode(p, FAKE, FAKE, FAKE, FAKE, None, None, None, None, FAKE, 1 << 20,
                            None) == attn.ATTN_ERR_INVALID_ARG
    p = base_problem(q_len=1, k_len=8192)
    need = attn.attn_decode_workspace_size(p)
    assert need > 0 and need % 256 == 0
    assert attn.attn_decode(p, FAKE, FAKE, FAKE, FAKE, None, None, None, None, None, 0,
                            None) == attn.ATTN_ERR_WORKSPACE
    assert attn.attn_decode(p, FAKE, FAKE, FAKE, FAKE, None, None, None, None, FAKE, need - 1,
                            None) == attn.ATTN_ERR_WORKSPACE
    assert attn.attn_decode(p, FAKE, FAKE, FAKE, FAKE, None, None, None, None, FAKE + 16, need,
                            None) == attn.ATTN_ERR_ALIGNMENT


def _r256(x):
    return (x + 255) // 256 * 256


def _plan(k_len, pairs, int8):
    """The decode key-range plan as the header and its comments state it: at most 8
    ranges a row (multiples of 32 keys, at least 128, no longer than the cache rounded
    up); for int8 caches ~4096 ranges over the (batch, kv head) pairs, at most 16 a
    row, multiples of 64 keys, at least 128."""
    if int8:
        n = min(16, max(1, -(-4096 // pairs)))
        length = max(128, -(-(-(-k_len // n)) // 64) * 64)
        return -(-k_len // length)
    length = -(-k_len // 8)
    length = max(128, -(-length // 32) * 32)
    if length > k_len:
        length = -(-k_len // 32) * 32
    return -(-k_len // length)


@pytest.mark.parametrize("k_len,batch,kv_heads,int8", [
    (8192, 64, 8, False), (3000, 4, 2, False), (100, 2, 2, False), (1, 1, 1, False),
    (8192, 64, 8, True), (3000, 4, 2, True), (700, 200, 8, True), (100, 2, 2, True)])
def test_decode_workspace_follows_the_range_plan(L, k_len, batch, kv_heads, int8):
    """The workspace holds one partial (head_dim floats) and one LSE per (batch,
    head, range); the range count follows the shape-only plan."""
    heads, D = 4 * kv_heads, 128
    kw = dict(batch=batch, heads=heads, kv_heads=kv_heads, q_len=1, k_len=k_len, head_dim=D,
              q_layout=(0, heads * D, D, D), o_layout=(0, heads * D, D, D),
              k_layout=(0, kv_heads * k_len * D, k_len * D, D), v_layout=(0, kv_heads * k_len * D, k_len * D, D))
    if int8:
        kw.update(kv_dtype="i8", kv_scale="channel", k_scale_ptr=FAKE, v_scale_ptr=FAKE)   # scales are required
    n = _plan(k_len, batch * kv_heads, int8)
    rows = batch * heads
    assert attn.attn_decode_workspace_size(base_problem(**kw)) == _r256(rows * n * D * 4) + _r256(rows * n * 4)


def _fwd_ranges(B, H, Sq, Sk, D, key_splits):
    """The prefill key-range plan restated from the header: ranges only with
    fewer than 304 blocks of query rows and a long key axis."""
    if key_splits > 0:
        n = min(key_splits, 16)
    else:
        rows = 256 if D <= 128 else 128
        blocks = -(-Sq // rows) * H * B
        if blocks >= 304:
            return 1
        n = min(-(-304 // blocks), 16, Sk // 1024)
    if n < 2:
        return 1
    length = -(-(-(-Sk // n)) // 128) * 128
    return -(-Sk // length)


@pytest.mark.parametrize("B,H,Sq,Sk,D,ks", [
    (1, 32, 64, 8192, 128, 0), (4, 12, 1024, 1024, 64, 0), (4, 12, 1024, 1024, 64, 4), (2, 32, 4096, 4096, 128, 0),
    (1, 4, 100, 5000, 256, 0), (1, 1, 1, 3000, 128, 0), (2, 2, 16, 1500, 64, 0), (1, 2, 8, 8, 64, 3),
    (1, 8, 300, 20000, 128, 40)])
def test_fwd_workspace_follows_the_range_plan(L, B, H, Sq, Sk, D, ks):
    """attn_fwd's workspace holds one partial row and one LSE per (batch, head,
    query row, key range) when the shape-only plan (or key_splits) cuts the keys."""
    G = H
    kw = dict(batch=B, heads=H, kv_heads=G, q_len=Sq, k_len=Sk, head_dim=D, key_splits=ks,
              q_layout=(0, H * Sq * D, Sq * D, D), o_layout=(0, H * Sq * D, Sq * D, D),
              k_layout=(0, G * Sk * D, Sk * D, D), v_layout=(0, G * Sk * D, Sk * D, D))
    n = _fwd_ranges(B, H, Sq, Sk, D, ks)
    rows = B * H * Sq
    want = 0 if n == 1 else _r256(rows * n * D * 4) + _r256(rows * n * 4)
    assert attn.attn_fwd_workspace_size(base_problem(**kw)) == want


def test_fwd_forced_ranges_need_the_workspace(L):
    """key_splits > 1 with no workspace is refused before any launch; a negative count is invalid."""
    kw = dict(batch=1, heads=2, kv_heads=2, q_len=8, k_len=1000, head_dim=64,
              q_layout=(0, 2 * 8 * 64, 8 * 64, 64), o_layout=(0, 2 * 8 * 64, 8 * 64, 64),
              k_layout=(0, 2 * 1000 * 64, 1000 * 64, 64), v_layout=(0, 2 * 1000 * 64, 1000 * 64, 64))
    p = base_problem(key_splits=4, **kw)
    assert attn.attn_fwd_workspace_size(p) > 0
    assert attn.attn_fwd(p, FAKE, FAKE, FAKE, FAKE, None, None, None, None, None, 0, None) == attn.ATTN_ERR_WORKSPACE
    p = base_problem(key_splits=-1, **kw)
    assert attn.attn_fwd(p, FAKE, FAKE, FAKE, FAKE, None, None, None, None, None, 0, None) == attn.ATTN_ERR_INVALID_ARG


def test_combine_checks(L):
    assert attn.attn_combine(4, 0, 64, None, None, 0, None, 64, None, 0, None) == 0
    assert attn.attn_combine(4, 3, 0, FAKE, FAKE, 0, FAKE, 64, None, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_combine(4, 3, 64, FAKE, FAKE, 9, FAKE, 64, None, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_combine(4, 3, 64, None, FAKE, 0, FAKE, 64, None, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_combine(4, 3, 64, FAKE, FAKE, 1, FAKE + 1, 64, None, 0, None) == attn.ATTN_ERR_ALIGNMENT


def test_probe_checks(L):
    """The exponential probe rejects its bad arguments before any launch."""
    E = attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_probe_ex2(0, 1, FAKE, None) == E
    assert attn.attn_probe_ex2(1, 0, FAKE, None) == E
    assert attn.attn_probe_ex2(1, 1, None, None) == E
    assert attn.attn_probe_ex2(1, 1, FAKE + 2, None) == E


def test_status_strings_and_version(L):
    for code in range(7):
        assert attn.status_string(code) and attn.status_string(code) != "unknown status"
    assert attn.status_string(99) == "unknown status"
    assert attn.attn_version() >= 250


def test_test_inject_checks(L):
    """The one-shot test fault: known codes are accepted (and disarmed again
    here, so no later launch takes it); unknown codes are rejected."""
    assert attn.attn_test_inject(attn.ATTN_INJECT_DROP_FIRST_COPY) == attn.ATTN_OK
    assert attn.attn_test_inject(attn.ATTN_INJECT_NONE) == attn.ATTN_OK
    assert attn.attn_test_inject(7) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_test_inject(-1) == attn.ATTN_ERR_INVALID_ARG
