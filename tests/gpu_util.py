"""GPU-side helpers for the parity tests: move a seeded case to the device,
run it through the C ABI, bring the outputs back, and compare them with the
oracle under the tolerances the tests state."""
from __future__ import annotations

import numpy as np

import oracle
from attention_attn_fwd_02_gb300 import attn
from attention_attn_fwd_02_gb300 import workloads as wl
from tutil import widen

# Bars stated for this path: float32 per element |d| <= 2e-6 (1 + |O|); half types
# |d| <= 1.5e-2 absolute; LSE |d| <= 1e-3; row classes (finite / NaN / zero) exact.
F32_REL = 2e-6
HALF_ABS = 1.5e-2
LSE_ABS = 1e-3
# "Attention" (recursiveai.org OneGPU docs), section "Tolerances": scaled error bounds.
SCALED = {"f32": 1e-5, "f16": 2e-3, "bf16": 8e-3}
SENTINEL = -4096.0   # exactly representable in f32, f16 and bf16


def torch_mod():
    import torch
    return torch


def dev(a: np.ndarray | None, dtype: str | None = None):
    """numpy storage -> CUDA tensor (uint16 patterns become f16/bf16 tensors)."""
    if a is None:
        return None
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.cuda()


def host_storage(t, dtype: str) -> np.ndarray:
    torch = torch_mod()
    t = t.detach().cpu().contiguous()
    if dtype == "f32":
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


class GpuCase:
    """Device buffers of a case plus output buffers, run through the C ABI."""

    def __init__(self, case: wl.Case, lse=True, guard=64):
        torch = torch_mod()
        self.case = case
        p = case.problem
        self.dtype = p["dtype"]
        self.q, self.k, self.v = dev(case.q, self.dtype), dev(case.k, self.dtype), dev(case.v, self.dtype)
        self.mask = dev(case.mask)
        self.seg = dev(case.seg)
        self.k_lens = dev(case.k_lens)
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[self.dtype]
        n_o = int(np.prod(case.o_shape))
        # guard bands of a sentinel pattern around every output buffer
        self.guard = guard
        self.o_buf = torch.full((n_o + 2 * guard,), SENTINEL, dtype=tdt,
                                device="cuda")
        self.o = self.o_buf[guard:guard + n_o]
        B, H, Sq = p["batch"], p["heads"], p["q_len"]
        self.lse_buf = torch.full((B * H * Sq + 2 * guard,), 777.0, dtype=torch.float32, device="cuda") if lse else None
        self.lse = self.lse_buf[guard:guard + B * H * Sq] if lse else None
        self.sink = dev(case.head_sink)
        self.k_scale, self.v_scale = dev(case.k_scale), dev(case.v_scale)
        ptr = (lambda t: None if t is None else t.data_ptr())
        self.prob = attn.make_problem(dict(p, head_sink_ptr=ptr(self.sink), k_scale_ptr=ptr(self.k_scale),
                                           v_scale_ptr=ptr(self.v_scale)))
        self.ws = None
        self.ws_bytes = 0

    def run(self, stream=None):
        torch = torch_mod()
        st = torch.cuda.current_stream().cuda_stream if stream is None else stream
        P = attn
        ptr = (lambda t: None if t is None else t.data_ptr())
        if self.case.decode:
            need = P.attn_decode_workspace_size(self.prob)
            if self.ws is None or self.ws_bytes < need:
                self.ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
                self.ws_bytes = need
            rc = P.attn_decode(self.prob, ptr(self.q), ptr(self.k), ptr(self.v), ptr(self.o), ptr(self.mask),
                               ptr(self.seg), ptr(self.k_lens), ptr(self.lse), ptr(self.ws), self.ws_bytes, st)
        else:
            need = P.attn_fwd_workspace_size(self.prob)
            if need and (self.ws is None or self.ws_bytes < need):
                self.ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
                self.ws_bytes = need
            rc = P.attn_fwd(self.prob, ptr(self.q), ptr(self.k), ptr(self.v), ptr(self.o), ptr(self.mask),
                            ptr(self.seg), ptr(self.k_lens), ptr(self.lse), ptr(self.ws) if need else None,
                            self.ws_bytes if need else 0, st)
        if rc != 0:
            raise attn.AttnError(rc, "attn_decode" if self.case.decode else "attn_fwd")
        return self

    def check_guards(self):
        torch = torch_mod()
        torch.cuda.synchronize()
        g = self.guard
        ob = self.o_buf.float().cpu().numpy()
        assert np.all(ob[:g] == SENTINEL) and np.all(ob[-g:] == SENTINEL), "write outside O"
        if self.lse_buf is not None:
            lb = self.lse_buf.cpu().numpy()
            assert np.all(lb[:g] == 777.0) and np.all(lb[-g:] == 777.0), "write outside LSE"

    def outputs(self):
        """(O canonical [B,H,Sq,D] float64, LSE [B,H,Sq] float64 or None, raw O storage)."""
        torch = torch_mod()
        torch.cuda.synchronize()
        p = self.case.problem
        B, H, Sq, D = p["batch"], p["heads"], p["q_len"], p["head_dim"]
        raw = host_storage(self.o, self.dtype).reshape(self.case.o_shape)
        o = widen(raw, self.dtype)
        if p["o_kind"] == "bshd":
            o = o.transpose(0, 2, 1, 3)
        lse = None if self.lse is None else self.lse.cpu().numpy().astype(np.float64).reshape(B, H, Sq)
        return np.ascontiguousarray(o), lse, raw


def oracle_full(case: wl.Case):
    p = case.problem
    o, lse = oracle.attn(p, case.q, case.k, case.v, mask=case.mask, seg=case.seg, k_lens=case.k_lens,
                         head_sink=case.head_sink, k_scale=case.k_scale, v_scale=case.v_scale)
    B, H, Sq, D = p["batch"], p["heads"], p["q_len"], p["head_dim"]
    return o.reshape(B, H, Sq, D), lse.reshape(B, H, Sq)


def compare(o, lse, ref_o, ref_lse, dtype, masked_rows="nan", where=""):
    """Apply the bars; returns a dict of error statistics.  Raises AssertionError on failure."""
    D = o.shape[-1]
    o2 = o.reshape(-1, D)
    r2 = ref_o.reshape(-1, D)
    # row classes: finite / NaN / zero rows must agree exactly
    ref_nan = np.all(np.isnan(r2), axis=1)
    got_nan = np.all(np.isnan(o2), axis=1)
    assert np.array_equal(ref_nan, got_nan), f"{where}: NaN-row classes differ ({np.sum(ref_nan != got_nan)} rows)"
    assert not np.any(np.isnan(o2[~got_nan])), f"{where}: NaN inside a non-NaN row"
    if masked_rows == "zero":
        ref_zero = np.all(r2 == 0, axis=1)
        assert np.all(o2[ref_zero] == 0), f"{where}: masked rows not zero"
    fin = ~ref_nan
    diff = np.abs(o2[fin] - r2[fin])
    stats = {"rows": int(r2.shape[0]), "nan_rows": int(ref_nan.sum())}
    if fin.any():
        if dtype == "f32":
            bound = F32_REL * (1 + np.abs(r2[fin]))
            bad = diff > bound
        else:
            bad = diff > HALF_ABS
        stats["max_abs_err"] = float(diff.max())
        denom = float(np.abs(r2[fin]).max())
        stats["scaled_err"] = float(diff.max() / denom) if denom > 0 else 0.0
        assert not bad.any(), (f"{where}: {int(bad.sum())} elements beyond the bar; worst {diff.max():.3g} at "
                               f"ref {r2[fin][bad][0]:.6g}")
        assert stats["scaled_err"] <= SCALED[dtype], f"{where}: scaled error {stats['scaled_err']:.3g}"
    if lse is not None and ref_lse is not None:
        l1, l2 = lse.reshape(-1), ref_lse.reshape(-1)
        assert np.array_equal(np.isnan(l1), np.isnan(l2)), f"{where}: LSE NaN classes differ"
        assert np.array_equal(np.isneginf(l1), np.isneginf(l2)), f"{where}: LSE -inf classes differ"
        f = np.isfinite(l2)
        if f.any():
            le = np.abs(l1[f] - l2[f])
            stats["lse_max_err"] = float(le.max())
            assert le.max() <= LSE_ABS, f"{where}: LSE error {le.max():.3g}"
    return stats
