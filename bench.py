"""Benchmark of the fused attention forward on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * prefill: attn_fwd on the long causal GQA workload (bf16, batch 2, 32 heads
    over 8 KV heads, 4096 queries and keys, head_dim 128, head-first layout,
    per-batch key lengths in [2048, 4096]);
  * decode: attn_decode on the batched single-query workload (bf16, batch 64,
    32 heads over 8 KV heads, BNSH cache [64, 8, 8192, 128], valid lengths in
    [512, 8192]): split-range pass + range-order combine.
value = prefill TFLOP/s (4 * head_dim * visible query-key pairs / prefill time);
the decode KV GB/s (K and V bytes of the valid cache rows / decode time) is in
the "decode" object.  Inputs are resident in HBM when the timed region starts;
L2 is flushed (a 256 MiB write) between timed steps.  e2e repeats the prefill
through the public Python API with host buffers: pinned-host -> device copies
of Q, K, V and the key lengths, the call, and device -> host copies of O and
LSE, all inside the timed region.

--impl reference times the float64 CPU oracle on the host cores instead (a
bounded sample of the same workload per step), for the driver's reference arm.

Run: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica (the path has no
exchange step); rank 0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from attention_attn_fwd_02_gb300 import workloads as wl  # noqa: E402

METRIC = "prefill TFLOP/s & decode KV GB/s at 1 GB300, as % of BF16/HBM roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
    except (OSError, subprocess.SubprocessError):
        out = ""
    for line in out.splitlines():
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values, world: int, device=None):
    """Element-wise maximum of per-rank timings (seconds) over all ranks.

    The path has no exchange step, so ranks are independent replicas: the
    whole job finishes when the slowest rank does."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def ex2_rate(torch, attn, dev) -> float:
    """Exponentials per second of the whole GPU, from the library's ex2 probe
    (8 CTAs of 256 threads per SM, 8 chains a thread), best of three timed
    launches after one warm-up."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = 8 * sms, 2048
    sink = torch.empty(blocks, dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream(dev)
    best = None
    for rep in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        rc = attn.attn_probe_ex2(blocks, iters, sink.data_ptr(), st.cuda_stream)
        e1.record(st)
        if rc:
            raise attn.AttnError(rc, "attn_probe_ex2")
        e1.synchronize()
        if rep:
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
    return blocks * 256.0 * iters * 8 / (best / 1e3)


def job_throughput(units_per_rank: float, world: int, steps: int, slowest_seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return world * steps * units_per_rank / slowest_seconds


def decode_kv_bytes(case) -> int:
    """K and V bytes of the valid cache rows (2 bytes an element, 1 for an int8 cache)."""
    p = case.problem
    kl = np.clip(case.k_lens.astype(np.int64), 0, p["k_len"])
    es = 1 if p.get("kv_dtype") == "i8" else 2
    return int(kl.sum()) * p["kv_heads"] * p["head_dim"] * 2 * es


def source_digest(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "attention_attn_fwd_02_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, digest: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_digest") != digest:
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- the CPU oracle (reference arm and cpu_baseline leg) --------------------------------


def oracle_prefill_sample(case, seconds: float, nthreads: int, seed: int = 0):
    """Time the oracle on sampled query rows of the prefill workload; returns (TFLOP/s, rows, wall s)."""
    import oracle
    p = case.problem
    B, H, Sq, D = p["batch"], p["heads"], p["q_len"], p["head_dim"]
    rng = np.random.default_rng(seed)

    def rows_flops(rows):
        off = p["k_len"] - p["q_len"] if p["causal_offset"] is None else p["causal_offset"]
        kl = np.minimum(case.k_lens[rows[:, 0]].astype(np.int64), p["k_len"])
        hi = np.minimum(kl, rows[:, 2] + off + 1)
        return 4.0 * D * float(np.maximum(hi, 0).sum())

    n = 512
    while True:
        rows = np.stack([rng.integers(0, B, n), rng.integers(0, H, n), rng.integers(0, Sq, n)], axis=1)
        t0 = time.perf_counter()
        oracle.attn(p, case.q, case.k, case.v, k_lens=case.k_lens, rows=rows, nthreads=nthreads)
        dt = time.perf_counter() - t0
        if dt >= seconds or n >= B * H * Sq:
            return rows_flops(rows) / dt / 1e12, n, dt
        n = int(min(B * H * Sq, n * max(2.0, 1.2 * seconds / max(dt, 1e-3))))


def oracle_decode_sample(case, seconds: float, nthreads: int, seed: int = 0):
    """Time the oracle on sampled (batch, head) rows of the decode workload; returns (GB/s, rows, wall s)."""
    import oracle
    p = case.problem
    B, H, G, D = p["batch"], p["heads"], p["kv_heads"], p["head_dim"]
    rng = np.random.default_rng(seed)
    n = 64
    while True:
        rows = np.stack([rng.integers(0, B, n), rng.integers(0, H, n), np.zeros(n, dtype=np.int64)], axis=1)
        t0 = time.perf_counter()
        oracle.attn(p, case.q, case.k, case.v, k_lens=case.k_lens, rows=rows, nthreads=nthreads)
        dt = time.perf_counter() - t0
        # bytes the sampled rows read (K and V of their valid cache rows, each head row counted once per
        # kv group share: q_per_group query heads read one kv head)
        kl = np.minimum(case.k_lens[rows[:, 0]].astype(np.int64), p["k_len"])
        by = float(kl.sum()) * D * 2 * 2 / (H // G)
        if dt >= seconds or n >= B * H:
            return by / dt / 1e9, n, dt
        n = int(min(B * H, n * max(2.0, 1.2 * seconds / max(dt, 1e-3))))


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = oracle.default_threads()
    case = wl.long_causal_gqa_bf16()
    per_step = max(1.0, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_prefill_sample(case, per_step / 4, cores, seed=1)
    vals, walls, rows = [], [], 0
    for s in range(args.steps):
        v, n, dt = oracle_prefill_sample(case, per_step, cores, seed=100 + s)
        vals.append(v)
        walls.append(dt)
        rows += n
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(walls)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": case.name, "sample": f"{rows} random query rows over {args.steps} steps"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": f"{rows} random query rows of {case.name}, float64 three-pass oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- the GPU arm ----------------------------------------------------------------------------


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from attention_attn_fwd_02_gb300 import attn, build
    build.build()
    L = attn.lib()

    pf = wl.long_causal_gqa_bf16()
    dc = wl.decode_bnsh_bf16(batch=args.decode_batch)
    P = pf.problem
    D = P["head_dim"]
    pairs = wl.visible_pairs(pf)
    flops = 4.0 * D * pairs
    kv_bytes = decode_kv_bytes(dc)

    def to_dev(a, dtype):
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16 if dtype == "bf16" else torch.float16)
        return t.to(dev)

    B, H, Sq = P["batch"], P["heads"], P["q_len"]
    q = to_dev(pf.q, "bf16").reshape(B, H, Sq, D)
    k = to_dev(pf.k, "bf16").reshape(B, P["kv_heads"], P["k_len"], D)
    v = to_dev(pf.v, "bf16").reshape(B, P["kv_heads"], P["k_len"], D)
    kl = torch.from_numpy(pf.k_lens).to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    dP = dc.problem
    dq = to_dev(dc.q, "bf16").reshape(dP["batch"], 1, dP["heads"], dP["head_dim"])
    dk = to_dev(dc.k, "bf16").reshape(dP["batch"], dP["kv_heads"], dP["k_len"], dP["head_dim"])
    dv = to_dev(dc.v, "bf16").reshape(dP["batch"], dP["kv_heads"], dP["k_len"], dP["head_dim"])
    dkl = torch.from_numpy(dc.k_lens).to(dev)
    do = torch.empty_like(dq)
    pprob = attn.make_problem(dict(P, o_layout=P["o_layout"]))
    dprob = attn.make_problem(dP)
    ws_bytes = attn.attn_decode_workspace_size(dprob)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    pws_bytes = attn.attn_fwd_workspace_size(pprob)
    pws = torch.empty(max(pws_bytes, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    st = stream.cuda_stream

    def prefill():
        if args.only == "decode":
            return
        rc = attn.attn_fwd(pprob, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, None, kl.data_ptr(),
                           lse.data_ptr(), pws.data_ptr() if pws_bytes else None, pws_bytes, st)
        if rc:
            raise attn.AttnError(rc, "attn_fwd")

    def decode():
        if args.only == "prefill":
            return
        rc = attn.attn_decode(dprob, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), do.data_ptr(), None, None,
                              dkl.data_ptr(), None, ws.data_ptr(), ws_bytes, st)
        if rc:
            raise attn.AttnError(rc, "attn_decode")

    # correctness spot check on sampled rows before timing (oracle on the host)
    parity = None
    if rank == 0 and not args.no_check and args.only is None:
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        import oracle
        from gpu_util import compare
        prefill()
        decode()
        torch.cuda.synchronize()
        rng = np.random.default_rng(5)
        rows = np.stack([rng.integers(0, B, 64), rng.integers(0, H, 64), rng.integers(0, Sq, 64)], axis=1)
        ro, rl = oracle.attn(P, pf.q, pf.k, pf.v, k_lens=pf.k_lens, rows=rows)
        go = o.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
        gl = lse.cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
        st1 = compare(go, gl, ro, rl, "bf16", "nan", "bench prefill")
        drows = np.stack([rng.integers(0, dP["batch"], 64), rng.integers(0, dP["heads"], 64),
                          np.zeros(64, dtype=np.int64)], axis=1)
        dro, _ = oracle.attn(dP, dc.q, dc.k, dc.v, k_lens=dc.k_lens, rows=drows)
        dgo = do.float().cpu().numpy()[drows[:, 0], 0, drows[:, 1]].astype(np.float64)
        st2 = compare(dgo, None, dro, None, "bf16", "nan", "bench decode")
        parity = {"prefill_max_abs_err": st1.get("max_abs_err"), "prefill_lse_max_err": st1.get("lse_max_err"),
                  "decode_max_abs_err": st2.get("max_abs_err"), "rows_checked": 128, "status": "ok"}

    for _ in range(args.warmup):
        flush.zero_()
        prefill()
        decode()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t_wall0 = time.perf_counter()
        for s in range(args.steps):
            flush.zero_()
            evs[s][0].record(stream)
            prefill()
            evs[s][1].record(stream)
            decode()
            evs[s][2].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t_wall = time.perf_counter() - t_wall0
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    dec_ms = [e[1].elapsed_time(e[2]) for e in evs]
    step_ms = [a + b for a, b in zip(pre_ms, dec_ms)]
    pre_s, dec_s, step_s = max_over_ranks([sum(pre_ms) / 1e3, sum(dec_ms) / 1e3, sum(step_ms) / 1e3], world, dev)
    steps = args.steps
    pre_s = max(pre_s, 1e-12)
    dec_s = max(dec_s, 1e-12)
    value = job_throughput(flops, world, steps, pre_s) / 1e12
    dec_gbs = job_throughput(kv_bytes, world, steps, dec_s) / 1e9

    # e2e through the public API with pinned host buffers: every step copies its
    # inputs host -> device, runs attn_fwd and copies O and LSE back.  Steps are
    # pipelined the way a serving loop would run them: three streams (copies
    # in, compute, copies out) and two device buffer sets, so step s+1's
    # inputs travel while step s computes and step s-1's outputs return.
    e2e = None
    if not args.no_e2e and args.only is None:
        hq = torch.from_numpy(pf.q.view(np.int16)).view(torch.bfloat16).reshape(B, H, Sq, D).pin_memory()
        hk = torch.from_numpy(pf.k.view(np.int16)).view(torch.bfloat16).reshape(k.shape).pin_memory()
        hv = torch.from_numpy(pf.v.view(np.int16)).view(torch.bfloat16).reshape(v.shape).pin_memory()
        hkl = torch.from_numpy(pf.k_lens).pin_memory()
        ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
        hl = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
        bufs = [(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(kl),
                 torch.empty_like(o), torch.empty_like(lse)) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hkl))
        d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
        s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_run(n_steps):
            ev_in = [torch.cuda.Event() for _ in range(n_steps)]
            ev_cmp = [torch.cuda.Event() for _ in range(n_steps)]
            ev_out = [torch.cuda.Event() for _ in range(n_steps)]
            for s in range(n_steps):
                dq2, dk2, dv2, dkl2, do2, dl2 = bufs[s % 2]
                with torch.cuda.stream(s_in):
                    if s >= 2:
                        s_in.wait_event(ev_cmp[s - 2])      # buffer set free: step s-2 has read it
                    dq2.copy_(hq, non_blocking=True)
                    dk2.copy_(hk, non_blocking=True)
                    dv2.copy_(hv, non_blocking=True)
                    dkl2.copy_(hkl, non_blocking=True)
                    ev_in[s].record(s_in)
                s_cmp.wait_event(ev_in[s])
                if s >= 2:
                    s_cmp.wait_event(ev_out[s - 2])         # outputs of step s-2 are home
                rc = attn.attn_fwd(pprob, dq2.data_ptr(), dk2.data_ptr(), dv2.data_ptr(), do2.data_ptr(), None,
                                   None, dkl2.data_ptr(), dl2.data_ptr(), pws.data_ptr() if pws_bytes else None,
                                   pws_bytes, s_cmp.cuda_stream)
                if rc:
                    raise attn.AttnError(rc, "attn_fwd")
                ev_cmp[s].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp[s])
                    ho[s % 2].copy_(do2, non_blocking=True)
                    hl[s % 2].copy_(dl2, non_blocking=True)
                    ev_out[s].record(s_out)
            return ev_out[-1]

        e2e_run(max(2, args.warmup))
        torch.cuda.synchronize()
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_start.record(s_in)
        s_cmp.wait_event(e_start)
        s_out.wait_event(e_start)
        last = e2e_run(steps)
        s_out.wait_event(last)
        e_end.record(s_out)
        torch.cuda.synchronize()
        (e_s,) = max_over_ranks([e_start.elapsed_time(e_end) / 1e3], world, dev)
        # The host link's own rates on the same pinned buffers (best of three
        # single copies of Q in and O out), to read the e2e number against.
        def copy_gbs(dst, src):
            best = 0.0
            for _ in range(3):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                dst.copy_(src, non_blocking=True)
                b.record(stream)
                b.synchronize()
                best = max(best, src.numel() * src.element_size() / (a.elapsed_time(b) / 1e3) / 1e9)
            return best
        h2d_gbs, d2h_gbs = copy_gbs(bufs[0][0], hq), copy_gbs(ho[0], bufs[0][4])
        e2e = {"value": job_throughput(flops, world, steps, e_s) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs,
               "copy_bound_tflops": flops / (h2d / (h2d_gbs * 1e9)) / 1e12,
               "pipelining": "copies in, compute and copies out on three streams, two buffer sets"}

    pk, pk_kind = peaks()
    digest = source_digest("prefill_tc.cu", "tc_ptx.cuh")
    pre_launch_s = pre_s / steps
    roof = {"bound": "tensor", "achieved": flops / pre_launch_s / 1e12, "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s", "frac": flops / pre_launch_s / 1e12 / pk["bf16_tflops"],
            "peak_sustained": pk.get("bf16_tflops_sustained"),
            "frac_sustained": (flops / pre_launch_s / 1e12 / pk["bf16_tflops_sustained"]
                               if pk.get("bf16_tflops_sustained") else None),
            "traffic": ncu_traffic("prefill_tc", digest), "kernel": "attn::tc::prefill_tc_kernel<128,bf16>",
            "peak_kind": f"{pk_kind} bf16 dense, burst", "algorithmic_flops_per_launch": flops}
    dec_roof = {"bound": "hbm", "achieved": kv_bytes / (dec_s / steps) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": kv_bytes / (dec_s / steps) / 1e9 / pk["hbm_gbs"],
                "traffic": ncu_traffic("decode_split", source_digest("decode.cu", "simt.cu")),
                "peak_kind": f"{pk_kind} HBM copy", "frac_of_8tbs_spec": kv_bytes / (dec_s / steps) / 8e12,
                "algorithmic_bytes_per_launch": kv_bytes}
    # Exponential co-roofline: one exponential per visible pair (taken after the timed region).
    exp_roof = None
    if args.only != "decode":
        rate = ex2_rate(torch, attn, dev)
        sm_mhz = (clk.summary() or {}).get("sm_mhz")
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        pps = pairs / pre_launch_s
        exp_roof = {"ex2_per_s": rate, "pairs_per_s": pps, "frac": pps / rate,
                    "ex2_per_clock_per_sm": rate / (sms * sm_mhz * 1e6) if sm_mhz else None,
                    "basis": "one exponential per visible pair; ex2 probe kernel, 8 chains per thread"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.only is None:
        import oracle
        oracle.build()
        cores = oracle.default_threads()
        cv, n, dt = oracle_prefill_sample(pf, 10.0, cores)
        cpu = {"value": cv, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
               "sample": f"{n} random query rows of {pf.name} ({dt:.1f} s wall)",
               "single_thread": oracle_single_thread()}
    cases = None
    if rank == 0 and world == 1 and not args.no_cases and args.only is None:
        cases = extra_cases(pk, pk_kind)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * step_s / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{pf.name} + {dc.name}", "prefill": pf.name, "decode": dc.name,
                   "visible_pairs": pairs, "decode_kv_bytes": kv_bytes, "l2": "flushed (256 MiB write) between steps",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": None if args.only == "decode" else roof,
        "exp_roofline": exp_roof,
        "decode": (None if args.only == "prefill" else
               {"value": dec_gbs, "unit": "GB/s", "ms_per_step": 1e3 * dec_s / steps, "roofline": dec_roof}),
        "prefill_ms_per_step": 1e3 * pre_s / steps,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "extra": {"cases": cases,
                  "note": "per-call device times of the other workloads (median, L2 flushed before each call), "
                          "measured after the timed region; not part of value"},
        "gpu_launches": steps * ((args.only != "decode") + 2 * (args.only != "prefill")),
        "clocks": clk.summary(),
        "wall_s_timed_region": t_wall,
        "parity": parity,
        "library": {"path": attn.LIB_PATH, "version": L.attn_version()},
    }
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


CASES = {
    "tiny_f32_mha": lambda: wl.tiny_f32_mha(),
    "gqa_doc_causal_bf16": lambda: wl.gqa_doc_causal_bf16(),
    "long_causal_gqa_bf16": lambda: wl.long_causal_gqa_bf16(),
    "dense_gqa_bf16": lambda: wl.dense_gqa_bf16(),
    "masked_gqa_bf16": lambda: wl.masked_gqa_bf16(),
    "rowmask_gqa_bf16": lambda: wl.rowmask_gqa_bf16(),
    "short_query_cross_bf16": lambda: wl.short_query_cross_bf16(),
    "decode_bnsh_bf16": lambda: wl.decode_bnsh_bf16(),
    "decode_bnsh_int8": lambda: wl.decode_bnsh_int8(),
    "cross_mask_f16": lambda: wl.cross_mask_f16(),
    "cross_mask_f16_zero": lambda: wl.cross_mask_f16(masked_rows="zero"),
}


def time_case(case, steps: int, warmup: int, flush: bool = True, flush_kind: str = "write", lead_us: int = 0):
    """Median and minimum device time (ms) of one call of `case` through the C ABI,
    inputs resident in HBM, an L2 flush before each timed call: a 256 MiB write
    (which leaves L2 full of dirty lines, written back during the call), or with
    flush_kind "read" a 256 MiB read (L2 left clean and holding no input).
    lead_us > 0 puts a device-side wait of that length before the start event,
    so that the call is enqueued while the GPU is still busy and its host-side
    work stays outside the device-timed region (needed without a flush)."""
    import torch
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from gpu_util import GpuCase
    g = GpuCase(case, lse=True, guard=0)
    fl = torch.empty(256 << 20, dtype=torch.uint8, device="cuda") if flush else None
    for _ in range(warmup):
        g.run()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ms = []
    for _ in range(steps):
        if fl is not None:
            if flush_kind == "read":
                fl.sum(dtype=torch.int64)
            else:
                fl.zero_()
        if lead_us:
            torch.cuda._sleep(int(lead_us * 2000))   # ~lead_us at 2 GHz
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        g.run()
        e1.record(st)
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    return statistics.median(ms), min(ms)


def case_line(case, med_ms: float, pk: dict, pk_kind: str) -> dict:
    """Throughput of one call: decode KV GB/s against the HBM copy peak, prefill TFLOP/s
    against the bf16 peaks (burst and sustained)."""
    p = case.problem
    if case.decode:
        by = decode_kv_bytes(case)
        v = by / (med_ms / 1e3) / 1e9
        return {"unit": "GB/s", "value": v, "algorithmic_bytes": by, "frac": v / pk["hbm_gbs"],
                "peak_kind": f"{pk_kind} HBM copy"}
    fl = 4.0 * p["head_dim"] * wl.visible_pairs(case)
    v = fl / (med_ms / 1e3) / 1e12
    return {"unit": "TFLOP/s", "value": v, "algorithmic_flops": fl, "frac": v / pk["bf16_tflops"],
            "frac_sustained": v / pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
            "peak_kind": f"{pk_kind} bf16 dense (burst; sustained beside it)"}


def run_case(args):
    """Time one call of one named workload (inputs resident in HBM) and print a per-case line.

    Not the benchmark line: used for the per-workload table and for profiling the
    kernel a workload selects.  Each timed call is preceded by a 256 MiB L2 flush
    unless --no-flush is given; the line reports the median call time."""
    import torch
    from attention_attn_fwd_02_gb300 import attn, build
    build.build()
    attn.lib()
    torch.cuda.set_device(0)
    case = CASES[args.case]()
    med, mn = time_case(case, args.steps, args.warmup, flush=not args.no_flush, lead_us=100 if args.no_flush else 0)
    rc = attn.attn_device_status()
    pk, pk_kind = peaks()
    line = {"line": "case", "case": case.name, "steps": args.steps, "warmup": args.warmup, "ms_median": med,
            "ms_min": mn, "l2": ("not flushed (warm; a 100 us device-side wait before each call)" if args.no_flush
                                else "flushed (256 MiB write) before each call"),
            "status": attn.status_string(rc)}
    line.update(case_line(case, med, pk, pk_kind))
    print(json.dumps(line), flush=True)


# Workloads timed per call inside the default benchmark run (after its timed
# region) so their numbers sit in the same record: the tiny float32 MHA, the
# causal GQA with documents, the head_dim-256 masked cross-attention in both
# MaskedRows modes, and the context cases.
EXTRA_CASES = ("tiny_f32_mha", "gqa_doc_causal_bf16", "cross_mask_f16", "cross_mask_f16_zero", "dense_gqa_bf16",
               "masked_gqa_bf16", "rowmask_gqa_bf16", "short_query_cross_bf16", "decode_bnsh_int8")


def extra_cases(pk, pk_kind):
    from attention_attn_fwd_02_gb300 import attn
    out = {}
    for name in EXTRA_CASES:
        case = CASES[name]()
        small = name in ("tiny_f32_mha", "gqa_doc_causal_bf16")
        med, mn = time_case(case, 50 if small else 10, 5 if small else 3)
        d = {"workload": case.name, "ms_median": med, "ms_min": mn}
        d.update(case_line(case, med, pk, pk_kind))
        if small:
            # The small (latency-bound) workloads also as back-to-back calls with
            # L2 left warm (median of 200), beside the flushed figure.
            med_w, _ = time_case(case, 200, 5, flush=False, lead_us=100)
            w = case_line(case, med_w, pk, pk_kind)
            d["warm_l2_back_to_back"] = {"ms_median": med_w, "value": w["value"], "frac": w.get("frac")}
        if case.decode:
            # A decode reads more than L2 holds; beside the write-flushed figure,
            # the same call after a 256 MiB read (no dirty lines to write back).
            med_r, _ = time_case(case, 10, 3, flush_kind="read")
            r = case_line(case, med_r, pk, pk_kind)
            d["after_read_flush"] = {"ms_median": med_r, "value": r["value"], "frac": r["frac"]}
        d["status"] = attn.status_string(attn.attn_device_status())
        out[name] = d
    return out


def oracle_single_thread(names=("tiny_f32_mha", "gqa_doc_causal_bf16")):
    """Wall time of the float64 oracle on ONE host thread over the whole of the small workloads."""
    import oracle
    oracle.build()
    out = {}
    for name in names:
        case = CASES[name]()
        p = case.problem
        t0 = time.perf_counter()
        oracle.attn(p, case.q, case.k, case.v, mask=case.mask, seg=case.seg, k_lens=case.k_lens, nthreads=1)
        dt = time.perf_counter() - t0
        fl = 4.0 * p["head_dim"] * wl.visible_pairs(case)
        out[name] = {"workload": case.name, "seconds": dt, "value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": 1}
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-check", action="store_true")
    ap.add_argument("--no-cases", action="store_true", help="skip the per-call lines of the other workloads")
    ap.add_argument("--decode-batch", type=int, default=64,
                    help="batch of the decode workload (64 = the benchmark workload; smaller only for profiling)")
    ap.add_argument("--only", choices=["prefill", "decode"], default=None,
                    help="run one half of the step only (for profiling); the line is then partial")
    ap.add_argument("--case", choices=sorted(CASES), default=None,
                    help="time one call of one named workload instead of the benchmark step (per-case line)")
    ap.add_argument("--no-flush", action="store_true", help="with --case: keep L2 warm between calls")
    args = ap.parse_args()
    if args.case is not None:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
