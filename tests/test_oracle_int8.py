"""Pins for the oracle's int8 key/value cache (CPU, no GPU): each cache element
is a signed 8-bit integer times a float32 scale, one scale per cache or one per
(kv head, head-dim channel) ("com.microsoft.GroupQueryAttention"
(webgpu-kernels README), inputs k_scale and v_scale, attributes k_quant_type,
v_quant_type and kv_cache_bit_width).

Checks: with power-of-two scales every dequantised value is exact in bfloat16,
so the int8 problem must equal, bit for bit, the same problem with a bfloat16
cache holding those values (this pins the int8 reading and the channel index
g * head_dim + d: a transposed or per-head index changes the values); a brute
force with arbitrary scales; per-channel scales that are all equal give the
per-tensor result.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from attention_attn_fwd_02_gb300 import workloads as wl
from tutil import brute_force, canonical_problem, representable

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def int8_problem(B, H, G, Sq, Sk, D, per_channel, seed):
    r = np.random.default_rng(seed)
    Q = representable(r.standard_normal((B, H, Sq, D)), "bf16")
    K8 = r.integers(-128, 128, size=(B, G, Sk, D)).astype(np.int8)
    V8 = r.integers(-128, 128, size=(B, G, Sk, D)).astype(np.int8)
    n = G * D if per_channel else 1
    ks = np.exp2(r.integers(-9, -4, size=n)).astype(np.float32)
    vs = np.exp2(r.integers(-9, -4, size=n)).astype(np.float32)
    return Q, K8, V8, ks, vs


def dequant(x8, sc, per_channel, G, D):
    s = sc.reshape(G, 1, D) if per_channel else sc.reshape(1, 1, 1)
    return x8.astype(np.float64) * s.astype(np.float64)


@pytest.mark.parametrize("per_channel", [False, True])
def test_int8_cache_equals_the_dequantised_bf16_cache_bit_for_bit(per_channel):
    B, H, G, Sq, Sk, D = 2, 4, 2, 3, 11, 8
    Q, K8, V8, ks, vs = int8_problem(B, H, G, Sq, Sk, D, per_channel, 3)
    Kd = np.stack([dequant(K8[b], ks, per_channel, G, D) for b in range(B)])
    Vd = np.stack([dequant(V8[b], vs, per_channel, G, D) for b in range(B)])
    prob, qs, ks16, vs16 = canonical_problem(Q, Kd, Vd, "bf16", "bhsd", causal=True, causal_offset=6)
    assert np.array_equal(representable(Kd, "bf16"), Kd)           # the bf16 cache holds them exactly
    k_lens = np.array([11, 7], dtype=np.int32)
    o1, l1 = oracle.attn(prob, qs, ks16, vs16, k_lens=k_lens)
    p8 = dict(prob, kv_dtype="i8", kv_scale="channel" if per_channel else "tensor")
    o2, l2 = oracle.attn(p8, qs, K8, V8, k_lens=k_lens, k_scale=ks, v_scale=vs)
    assert np.array_equal(o1, o2, equal_nan=True) and np.array_equal(l1, l2, equal_nan=True)


def test_int8_brute_force_with_arbitrary_scales():
    B, H, G, Sq, Sk, D = 1, 2, 1, 4, 6, 4
    r = np.random.default_rng(5)
    Q, K8, V8, _, _ = int8_problem(B, H, G, Sq, Sk, D, True, 5)
    ks = r.uniform(0.001, 0.05, size=G * D).astype(np.float32)
    vs = r.uniform(0.001, 0.05, size=G * D).astype(np.float32)
    Kd = np.stack([dequant(K8[b], ks, True, G, D) for b in range(B)])
    Vd = np.stack([dequant(V8[b], vs, True, G, D) for b in range(B)])
    prob, qs, _, _ = canonical_problem(Q, Kd, Vd, "bf16", "bshd", scale=0.5)
    p8 = dict(prob, kv_dtype="i8", kv_scale="channel",
              k_layout=wl.layout_of("bhsd", B, G, Sk, D)[1], v_layout=wl.layout_of("bhsd", B, G, Sk, D)[1])
    o, lse = oracle.attn(p8, qs, K8, V8, k_scale=ks, v_scale=vs)
    ref_o, ref_l = brute_force(Q, Kd, Vd, 0.5, lambda b, q, k: True)
    assert np.allclose(o.reshape(ref_o.shape), ref_o, rtol=1e-12, atol=1e-15)
    assert np.allclose(lse.reshape(ref_l.shape), ref_l, rtol=1e-12, atol=1e-15)


def test_equal_channel_scales_equal_one_tensor_scale():
    B, H, G, Sq, Sk, D = 2, 2, 2, 3, 9, 4
    Q, K8, V8, _, _ = int8_problem(B, H, G, Sq, Sk, D, False, 7)
    prob, qs, _, _ = canonical_problem(Q, np.zeros((B, G, Sk, D)), np.zeros((B, G, Sk, D)), "bf16", "bhsd")
    p8 = dict(prob, kv_dtype="i8")
    o1, l1 = oracle.attn(dict(p8, kv_scale="tensor"), qs, K8, V8, k_scale=np.float32([0.03]),
                         v_scale=np.float32([0.2]))
    o2, l2 = oracle.attn(dict(p8, kv_scale="channel"), qs, K8, V8, k_scale=np.full(G * D, 0.03, np.float32),
                         v_scale=np.full(G * D, 0.2, np.float32))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
