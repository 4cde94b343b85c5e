"""Pins for the oracle's cache append (CPU, no GPU): the update that precedes a
decode step writes each (batch, kv head)'s new key/value row at cache position
L_b - 1, L_b the batch entry's clamped length including the new token
("com.microsoft.GroupQueryAttention" (webgpu-kernels README): present_key /
present_value sharing the past buffer, seqlens_k, the int8 decode variant that
appends quantised rows).

Checks: for float caches the result equals the cache with numpy's own slice
assignment of the new rows, bit for bit, and nothing else changes; entries of
length 0 are left alone; last-index lengths write one row further back than
counts of the same value.  For int8 caches the codes are fixed by exact cases:
values that are integer multiples of a power-of-two scale give those integers,
exact halves round to the even neighbour, and values beyond the range saturate
to -128 / 127.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from attention_attn_fwd_02_gb300 import workloads as wl


def problem(B, G, cap, D, dtype="bf16", **kw):
    d = dict(batch=B, heads=G, kv_heads=G, q_len=1, k_len=cap, head_dim=D, dtype=dtype,
             k_layout=wl.layout_of("bhsd", B, G, cap, D)[1], v_layout=wl.layout_of("bhsd", B, G, cap, D)[1])
    d.update(kw)
    return d


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_float_append_is_the_slice_assignment(dtype):
    B, G, cap, D = 3, 2, 10, 8
    r = np.random.default_rng(1)
    kc = wl.to_storage(r.standard_normal((B, G, cap, D)).astype(np.float32), dtype)
    vc = wl.to_storage(r.standard_normal((B, G, cap, D)).astype(np.float32), dtype)
    kn = wl.to_storage(r.standard_normal((B, G, D)).astype(np.float32), dtype)
    vn = wl.to_storage(r.standard_normal((B, G, D)).astype(np.float32), dtype)
    k_lens = np.array([10, 0, 4], dtype=np.int32)
    k2, v2 = oracle.append_rows(problem(B, G, cap, D, dtype), kc, vc, kn, vn, k_lens)
    ek, ev = kc.copy(), vc.copy()
    for b, L in enumerate(k_lens):
        if L >= 1:
            ek[b, :, L - 1] = kn[b]
            ev[b, :, L - 1] = vn[b]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)
    assert np.array_equal(k2[1], kc[1])                        # length 0: untouched
    # last-index lengths: the same stored values mean one more key, so one row further
    k3, _ = oracle.append_rows(problem(B, G, cap, D, dtype, k_lens_kind="last_index"), kc, vc, kn, vn,
                               np.array([8, 0, 3], dtype=np.int32))
    assert np.array_equal(k3[0, :, 8], kn[0]) and np.array_equal(k3[2, :, 3], kn[2])
    assert np.array_equal(k3[1, :, 0], kn[1])


def test_int8_codes_exact_multiples_ties_and_saturation():
    B, G, cap, D = 1, 2, 4, 8
    kc = np.zeros((B, G, cap, D), dtype=np.int8)
    ks = np.float32(0.0625)                                      # a power of two: x / s exact
    vals = np.array([[3, -7, 0, 127, -128, 2.5, -2.5, 1.5],        # multiples, ends, halves (ties to even)
                     [3.5, -3.5, 1000, -1000, 126.6, -127.4, 0.49, -0.51]], dtype=np.float32)
    want = np.array([[3, -7, 0, 127, -128, 2, -2, 2],
                     [4, -4, 127, -128, 127, -127, 0, -1]], dtype=np.int8)
    kn = wl.to_storage((vals * ks)[None], "f32")
    p = problem(B, G, cap, D, "f32", kv_dtype="i8", kv_scale="tensor")
    k2, _ = oracle.append_rows(p, kc, kc, kn, kn, np.array([3], dtype=np.int32), k_scale=[ks], v_scale=[ks])
    assert np.array_equal(k2[0, :, 2], want)
    assert np.all(k2[0, :, [0, 1, 3]] == 0)


def test_int8_per_channel_scales_follow_the_channel_index():
    B, G, cap, D = 2, 2, 3, 4
    kc = np.zeros((B, G, cap, D), dtype=np.int8)
    sc = np.exp2(-np.arange(G * D, dtype=np.float32))              # distinct per (g, d)
    ints = np.arange(B * G * D).reshape(B, G, D) % 50 - 25
    kn = wl.to_storage((ints * sc.reshape(G, D)).astype(np.float32), "bf16")
    p = problem(B, G, cap, D, "bf16", kv_dtype="i8", kv_scale="channel")
    k2, _ = oracle.append_rows(p, kc, kc, kn, kn, np.array([3, 1], dtype=np.int32), k_scale=sc, v_scale=sc)
    assert np.array_equal(k2[0, :, 2], ints[0]) and np.array_equal(k2[1, :, 0], ints[1])
