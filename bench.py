#!/usr/bin/env python
"""Throughput of the GB300 attention backward pass (dQ + dK + dV).

One step = one full backward pass (attn_bwd: Delta/LSE prep, the fused
tcgen05 tile kernel and, for bf16, the dQ conversion)
over one batch of the chosen workload, with inputs resident in HBM.  The
metric counts 10*D flops per visible (query, key) pair per query head (the
five dense contractions); recomputation is not credited.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own copy of
the workload on its own GPU (weak scaling, no collective on the data path);
the reported value is the work of all ranks over the slowest rank's time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  (default workload: GQA causal + window 1024, B2 Hq32 Hkv8 S4096 D128, fp32 I/O on TF32)
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from attention_backward_pass_gb300 import metrics as MET  # noqa: E402
from attention_backward_pass_gb300 import workloads as W  # noqa: E402

METRIC = "attention-backward TFLOP/s (dQ+dK+dV) and % of GB300 dense tensor peak"
LSE_METRIC = "LSE sweep TFLOP/s (2*D flops per visible pair) and % of GB300 dense tensor peak"
FWD_METRIC = "attention-forward TFLOP/s (4*D flops per visible pair) and % of GB300 dense tensor peak"
L2_BYTES = 129 * 1024 * 1024
# nominal dense ratio TF32 : BF16 on GB300 (1.1 vs 2.25 PFLOP/s)
TF32_OVER_BF16 = 1.1 / 2.25

WORKLOADS = {
    "causal_mha": (W.causal_mha, 1,
                   "causal MHA B4 H16 S1024 D64 fp32 [B,H,S,D]"),
    "gqa_window_f32": (lambda: W.gqa_window(W.DTYPE_F32), 2,
                       "GQA causal+window1024 B2 Hq32 Hkv8 S4096 D128 fp32 [B,S,H,D]"),
    "gqa_window_bf16": (lambda: W.gqa_window(W.DTYPE_BF16), 2,
                        "GQA causal+window1024 B2 Hq32 Hkv8 S4096 D128 bf16 [B,S,H,D]"),
    "masked_dropout": (W.masked_dropout, 3,
                       "masked+dropout B2 H16 Sq512 Sk2048 D64 fp32 causal_offset1536 p0.1"),
    "tiny": (W.tiny, 0, "tiny B1 H2 S64 D64 fp32"),
    "decode": (W.decode, 4, "decode backward: 64 seqs, 8 heads, 1 kv head, D256, history 4096, fp32"),
    "decode_kv": (W.decode, 4, "decode backward pass 2 (d_k_hist, d_v_hist): 64 seqs, 8 heads, "
                               "1 kv head, D256, history 4096, fp32"),
}
DECODE_METRIC = "decode attention-backward GB/s (d_scores+d_q) and % of HBM peak"
DECODE_KV_METRIC = "decode attention-backward pass 2 GB/s (d_k_hist+d_v_hist) and % of HBM peak"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gqa_window_f32", choices=sorted(WORKLOADS),
                    help="default: the GQA causal + sliding-window workload at fp32 I/O (TF32), "
                         "the largest dense configuration")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--recompute-lse", action="store_true",
                    help="dense workloads: the step recomputes the LSE (attn_bwd_lse) first")
    ap.add_argument("--deterministic", action="store_true",
                    help="dense workloads: bit-reproducible dQ (per-key-tile slices, ordered sum)")
    ap.add_argument("--fwd", action="store_true",
                    help="dense workloads: time the fused forward (attn_fwd) instead")
    ap.add_argument("--lse-only", action="store_true",
                    help="dense workloads: time the LSE sweep (attn_bwd_lse) alone")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def measure_matmul_peak(device, dtype_name="tf32", n=8192, reps=10, sustain_s=2.0):
    """Dense tensor-core peak of this GPU for one operand type, measured the
    way the bf16 figures of MEASURED_PEAKS.json are: torch.matmul of n x n x n
    (2 n^3 flops), CUDA events, best of ``reps`` back-to-back products
    (burst) and the mean rate over ``sustain_s`` seconds of back-to-back
    products (sustained).  tf32 = fp32 tensors with TF32 tensor-op math.
    Returns (burst TFLOP/s, sustained TFLOP/s)."""
    import torch
    old = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = dtype_name == "tf32"
    try:
        dt = torch.float32 if dtype_name == "tf32" else torch.bfloat16
        g = torch.Generator(device=device).manual_seed(0)
        a = torch.randn(n, n, device=device, dtype=dt, generator=g)
        b = torch.randn(n, n, device=device, dtype=dt, generator=g)
        c = torch.empty(n, n, device=device, dtype=dt)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        torch.cuda.synchronize()
        flops = 2.0 * n ** 3
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        count = 0
        t0 = time.perf_counter()
        e0.record()
        while time.perf_counter() - t0 < sustain_s:
            for _ in range(10):
                torch.matmul(a, b, out=c)
            count += 10
            e1.record()
            e1.synchronize()
        sustained = flops * count / (e0.elapsed_time(e1) * 1e-3) / 1e12
        del a, b, c
        return flops / (best * 1e-3) / 1e12, sustained
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old


def tensor_peak(p, device, peaks, peak_src):
    """(peak TFLOP/s, description, extra fields) for the tile kernels' operand
    type: bf16 from MEASURED_PEAKS.json (burst), TF32 measured in this run
    with measure_matmul_peak (burst), with the nominal-ratio figure kept
    beside it for comparison."""
    bf16_peak = float(peaks.get("bf16_tflops", 1900.0))
    if p.dtype == W.DTYPE_BF16:
        return bf16_peak, f"bf16 dense, {peak_src} burst (MEASURED_PEAKS.json)", {}
    burst, sustained = measure_matmul_peak(device, "tf32")
    extra = {"tf32_burst_tflops": burst, "tf32_sustained_tflops": sustained,
             "tf32_nominal_ratio_tflops": bf16_peak * TF32_OVER_BF16}
    return burst, ("tf32 dense, measured in this run: torch.matmul fp32 with TF32 math, "
                   "8192^3, best of 10 (burst)"), extra


def max_over_ranks(x: float, device="cpu") -> float:
    """The largest x over all ranks (the slowest rank's time), or x itself when
    no process group is running.  Every rank must call it."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, steps: int, total_ms: float) -> float:
    """Units all ranks processed per second, over the slowest rank's time."""
    return units_per_rank * world * steps / (total_ms * 1e-3)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------- inputs

def synth_forward(p, Q, K, V, mask):
    """O and LSE for the timed backward, from a plain torch forward on the GPU
    (input synthesis, untimed; no dropout).  Fully masked rows get LSE = 3e38
    and O = 0, the WGSL page's convention."""
    import torch
    dev = Q.device
    B, H, Hkv = p.batch, p.num_heads, p.num_kv_heads
    G = H // Hkv
    O = torch.empty_like(Q)
    LSE = torch.empty(p.lse_shape(), dtype=torch.float32, device=dev)
    i = torch.arange(p.seq_q, device=dev)[:, None] + p.causal_offset
    j = torch.arange(p.seq_k, device=dev)[None, :]
    allowed = torch.ones(p.seq_q, p.seq_k, dtype=torch.bool, device=dev)
    if p.causal:
        allowed &= j <= i
    if p.window:
        allowed &= (i - j).abs() < p.window
    for b in range(B):
        for h in range(H):
            kvh = h // G
            if p.layout == W.LAYOUT_BHSD:
                q, k, v = Q[b, h].float(), K[b, kvh].float(), V[b, kvh].float()
            else:
                q, k, v = Q[b, :, h].float(), K[b, :, kvh].float(), V[b, :, kvh].float()
            s = p.scale * (q @ k.T)
            al = allowed
            if mask is not None:
                m = mask[b, 0]
                al = al & (m > -1e30)
                s = s + torch.where(m > -1e30, m, torch.zeros_like(m))
            s = s.masked_fill(~al, float("-inf"))
            lse = torch.logsumexp(s, dim=-1)
            empty = ~torch.isfinite(lse)
            P = torch.exp(s - torch.where(empty, torch.zeros_like(lse), lse)[:, None])
            P = torch.where(al, P, torch.zeros_like(P))
            o = (P @ v).to(Q.dtype)
            o[empty] = 0
            lse = torch.where(empty, torch.full_like(lse, 3.0e38), lse)
            if p.layout == W.LAYOUT_BHSD:
                O[b, h] = o
            else:
                O[b, :, h] = o
            LSE[b, h] = lse
    return O, LSE


def device_inputs(p, seed, device):
    import torch
    Qn, Kn, Vn, dOn, maskn = W.make_inputs(p, seed)
    tdt = torch.bfloat16 if p.dtype == W.DTYPE_BF16 else torch.float32
    to = lambda x: torch.from_numpy(x).to(device).to(tdt)  # noqa: E731
    Q, K, V, dO = to(Qn), to(Kn), to(Vn), to(dOn)
    mask = torch.from_numpy(maskn).to(device) if maskn is not None else None
    O, LSE = synth_forward(p, Q, K, V, mask)
    return dict(Q=Q, K=K, V=V, O=O, dO=dO, LSE=LSE, mask=mask,
                numpy=dict(Q=Qn, K=Kn, V=Vn, dO=dOn, mask=maskn))


# --------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            sel = str(device_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        loaded = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def load_under_clock_sampling(step, seconds=0.8):
    """Untimed steps right before the timed ones, so that the clock sampler
    (200 ms period) sees the GPU under this load; the timed region itself is
    only milliseconds long."""
    import torch
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(20):
            step()
        torch.cuda.synchronize()


# --------------------------------------------------------------- CPU oracle

def oracle_sample_tflops(p, numpy_inputs, O_np, LSE_np, budget_s: float, rng_seed=0):
    """Time the fp64 oracle on seeded (batch, kv-head) groups until the time
    budget is used; returns (TFLOP/s scaled to the metric's flop count, groups
    done, total groups, seconds)."""
    from oracle import attention as OA
    groups_all = [(b, g) for b in range(p.batch) for g in range(p.num_kv_heads)]
    rng = np.random.default_rng(rng_seed)
    order = rng.permutation(len(groups_all))
    per_group = MET.counted_flops(p) / len(groups_all)
    f = lambda x: None if x is None else x.astype(np.float64)  # noqa: E731
    Q, K, V, dO = (f(numpy_inputs[k]) for k in ("Q", "K", "V", "dO"))
    mask = numpy_inputs["mask"]
    done, t_total = 0, 0.0
    for idx in order:
        grp = [groups_all[idx]]
        t0 = time.perf_counter()
        OA.backward(p, Q, K, V, O_np, dO, LSE_np, mask, groups=grp)
        t_total += time.perf_counter() - t0
        done += 1
        if t_total >= budget_s:
            break
    return per_group * done / t_total / 1e12, done, len(groups_all), t_total


# --------------------------------------------------------------- main arms

def run_reference_decode(args):
    """Reference arm for the decode workloads: the oracle on one sequence per
    step (fp64 numpy on the host cores), value in the arm's GB/s unit."""
    make, seed, desc = WORKLOADS[args.workload]
    p = make()
    kv_pass = args.workload == "decode_kv"
    from oracle import decode as OD
    k, v, d_out, logits = W.make_decode_inputs(p, seed)
    e = np.exp(logits - logits.max(axis=-1, keepdims=True))  # input synthesis
    probs = e / e.sum(axis=-1, keepdims=True)
    nbytes = MET.decode_kv_bytes(p) if kv_pass else MET.decode_bytes(p)
    per_seq = nbytes / p.num_seqs
    if kv_pass:
        q = W.make_decode_queries(p, seed)
        d_scores, _ = OD.decode_backward(k, v, probs, d_out)  # untimed inputs
    vals = []
    for step in range(args.warmup + args.steps):
        n = step % p.num_seqs
        t0 = time.perf_counter()
        if kv_pass:
            OD.decode_backward_kv(q, probs, d_out, d_scores, p.n_kv_heads, seqs=[n])
        else:
            OD.decode_backward(k, v, probs, d_out, seqs=[n])
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            vals.append(dt)
    value = per_seq * len(vals) / sum(vals) / 1e9
    sample = (f"one sequence of {p.num_seqs} per step, fp64 numpy; ms_per_step is the time of "
              "that one sequence")
    line = {
        "impl": "reference", "metric": DECODE_KV_METRIC if kv_pass else DECODE_METRIC,
        "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.mean(vals) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": desc, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    if args.workload in ("decode", "decode_kv"):
        return run_reference_decode(args)
    make, seed, desc = WORKLOADS[args.workload]
    p = make()
    from oracle import attention as OA
    Qn, Kn, Vn, dOn, maskn = W.make_inputs(p, seed)
    f = lambda x: x.astype(np.float64)  # noqa: E731
    groups_all = [(b, g) for b in range(p.batch) for g in range(p.num_kv_heads)]
    # the same work as the arm being compared: the LSE sweep, the forward, or
    # the backward (default)
    if args.lse_only:
        metric, flops = LSE_METRIC, MET.lse_flops(p)
    elif args.fwd:
        metric, flops = FWD_METRIC, 2.0 * MET.lse_flops(p)
    else:
        metric, flops = METRIC, MET.counted_flops(p)
    per_group = flops / len(groups_all)
    vals, secs = [], []
    # fp64 copies made once, outside the timed calls; steps cycle over (at
    # most) four seeded groups, whose O / LSE inputs are synthesised once
    Q64, K64, V64, dO64 = f(Qn), f(Kn), f(Vn), f(dOn)
    rng = np.random.default_rng(0)
    picks = [groups_all[int(i)] for i in rng.permutation(len(groups_all))[:4]]
    fwd_cache = {}
    for step in range(args.warmup + args.steps):
        grp = [picks[step % len(picks)]]
        if args.lse_only:
            t0 = time.perf_counter()
            OA.lse(p, Q64, K64, maskn, groups=grp)
        elif args.fwd:
            t0 = time.perf_counter()
            OA.forward(p, Q64, K64, V64, maskn, groups=grp)
        else:
            if grp[0] not in fwd_cache:  # untimed input synthesis
                fwd_cache[grp[0]] = OA.forward(p, Q64, K64, V64, maskn, groups=grp)
            O, LSE = fwd_cache[grp[0]]
            t0 = time.perf_counter()
            OA.backward(p, Q64, K64, V64, O, dO64, LSE, maskn, groups=grp)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            vals.append(per_group / dt / 1e12)
            secs.append(dt)
    # value: the work timed (one group per step) over the time it took
    value = per_group * len(secs) / sum(secs) / 1e12
    cores = os.cpu_count()
    sample = (f"one (batch, kv-head) group of {len(groups_all)} per step "
              f"({per_group / 1e9:.2f} GFLOP counted), fp64 numpy; ms_per_step is the time of "
              "that one group")
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.mean(secs) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": desc, "sample": sample, "groups_per_step": 1,
                   "groups_in_workload": len(groups_all), "flops_per_step": per_group},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    import attention_backward_pass_gb300 as ab

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    ab.load_library()
    make, seed, desc = WORKLOADS[args.workload]
    p = make()
    p.deterministic = 1 if args.deterministic else 0
    x = device_inputs(p, seed, device)
    tdt = x["Q"].dtype
    dQ = torch.empty(p.q_shape(), dtype=tdt, device=device)
    dK = torch.empty(p.kv_shape(), dtype=tdt, device=device)
    dV = torch.empty(p.kv_shape(), dtype=tdt, device=device)
    ws = ab.alloc_workspace(p, device)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    rec = args.recompute_lse
    lse_buf = torch.empty_like(x["LSE"]) if rec else x["LSE"]

    def step():
        if rec:
            ab.attn_bwd_lse(p, x["Q"], x["K"], x["mask"], lse_buf)
        ab.attn_bwd(p, x["Q"], x["K"], x["V"], x["O"], x["dO"], lse_buf, x["mask"], dQ, dK, dV,
                    ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if ab.check_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # the K timed steps: attn_bwd as a caller issues it (inside it the tile
    # kernel may start while the prepare kernel finishes)
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    load_under_clock_sampling(step)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.zero_()  # L2 flush between timed steps (outside the events)
        sevs[k][0].record(stream)
        step()
        sevs[k][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    if ab.check_device_error() != 0:
        raise RuntimeError("device error word set during the timed steps")
    step_ms = [e[0].elapsed_time(e[1]) for e in sevs]
    # the same steps once more through the three staged entry points, with
    # events between the stages: the per-kernel split (not part of the value)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.zero_()
        e = evs[k]
        e[4].record(stream)
        if rec:  # no saved LSE: the sweep is part of the step
            ab.attn_bwd_lse(p, x["Q"], x["K"], x["mask"], lse_buf)
        e[0].record(stream)
        ab.attn_bwd_prepare(p, x["Q"], x["K"], x["O"], x["dO"], lse_buf, dQ, ws)
        e[1].record(stream)
        ab.attn_bwd_tiles(p, x["Q"], x["K"], x["V"], x["dO"], x["mask"], dQ, dK, dV, ws)
        e[2].record(stream)
        ab.attn_bwd_finish(p, dQ, ws)
        e[3].record(stream)
    torch.cuda.synchronize()
    if ab.check_device_error() != 0:
        raise RuntimeError("device error word set during the staged steps")
    lse_ms = [e[4].elapsed_time(e[0]) for e in evs]
    tile_ms = [e[1].elapsed_time(e[2]) for e in evs]
    prep_ms = [e[0].elapsed_time(e[1]) for e in evs]
    fin_ms = [e[2].elapsed_time(e[3]) for e in evs]
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, device)
    flops = MET.counted_flops(p)
    value = whole_job_rate(flops, world, args.steps, total_ms) / 1e12
    ms_per_step = total_ms / args.steps

    # roofline of the dominant kernel (the fused tile kernel)
    peaks, peak_src = load_peaks()
    tile_mean = statistics.mean(tile_ms)
    achieved = flops / (tile_mean * 1e-3) / 1e12
    traffic = read_traffic(args.workload)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(p, x, dQ, dK, dV, ws, args, stream, world)
    # after the timed regions: the reference products heat the GPU
    peak, peak_note, peak_extra = tensor_peak(p, device, peaks, peak_src)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        O_np = x["O"].float().cpu().numpy().astype(np.float64)
        LSE_np = x["LSE"].cpu().numpy().astype(np.float64)
        val, done, tot, secs = oracle_sample_tflops(p, x["numpy"], O_np, LSE_np, budget_s=12.0)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{done} of {tot} (batch, kv-head) groups, {secs:.1f} s, fp64 numpy"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if p.dtype == W.DTYPE_BF16 else "tf32",
            "data": "synthetic",
            "config": {"workload": desc, "l2": "flushed between timed steps (256 MiB write)",
                       "flops_per_step": flops, "parallelism": f"replicas x{world}",
                       "lse": ("recomputed in the step by attn_bwd_lse (its 2*D flops per "
                               "visible pair are not counted)") if rec else "given",
                       "dq": ("deterministic: per-key-tile slices summed in key-tile order"
                              if p.deterministic else "fp32 reduce-add (atomic)")},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                         "kernel": "dkdv_kernel (tcgen05 tile kernel)", "peak_source": peak_note,
                         "kernel_ms": tile_mean, "prep_ms": statistics.mean(prep_ms),
                         "finish_ms": statistics.mean(fin_ms),
                         "lse_ms": statistics.mean(lse_ms) if rec else 0.0,
                         "step_frac": value / peak, **peak_extra},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": ab.kernels_per_call(p, recompute_lse=rec) * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_lse_only(args):
    """The LSE sweep alone (attn_bwd_lse) on a dense workload: tensor-bound,
    value = 2*D flops per visible pair / time."""
    import torch
    import attention_backward_pass_gb300 as ab
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    ab.load_library()
    make, seed, desc = WORKLOADS[args.workload]
    p = make()
    Qn, Kn, _, _, maskn = W.make_inputs(p, seed)
    tdt = torch.bfloat16 if p.dtype == W.DTYPE_BF16 else torch.float32
    Q = torch.from_numpy(Qn).to(device).to(tdt)
    K = torch.from_numpy(Kn).to(device).to(tdt)
    mask = torch.from_numpy(maskn).to(device) if maskn is not None else None
    lse = torch.empty(p.lse_shape(), dtype=torch.float32, device=device)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def step():
        ab.attn_bwd_lse(p, Q, K, mask, lse)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    load_under_clock_sampling(step)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for a, b in evs:
        flush.zero_()  # L2 flush between timed steps (outside the events)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    if ab.check_device_error() != 0:
        raise RuntimeError("device error word set")
    ms = [a.elapsed_time(b) for a, b in evs]
    total = sum(ms)
    total = max_over_ranks(total, device)
    flops = MET.lse_flops(p)
    value = whole_job_rate(flops, world, args.steps, total) / 1e12
    peaks, src = load_peaks()
    peak, note, peak_extra = tensor_peak(p, device, peaks, src)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import attention as OA
        groups_all = [(b, g) for b in range(p.batch) for g in range(p.num_kv_heads)]
        t0 = time.perf_counter()
        done = 0
        for grp in groups_all:
            OA.lse(p, Qn.astype(np.float64), Kn.astype(np.float64), maskn, groups=[grp])
            done += 1
            if time.perf_counter() - t0 > 12.0:
                break
        secs = time.perf_counter() - t0
        cpu = {"value": flops / len(groups_all) * done / secs / 1e12, "unit": "TFLOP/s",
               "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{done} of {len(groups_all)} (batch, kv-head) groups, {secs:.1f} s, "
                         "fp64 numpy"}
    if rank == 0:
        mean_ms = statistics.mean(ms)
        line = {
            "metric": LSE_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if p.dtype == W.DTYPE_BF16 else "tf32", "data": "synthetic",
            "config": {"workload": "LSE sweep of " + desc,
                       "l2": "flushed between timed steps (256 MiB write)",
                       "flops_per_step": flops, "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": flops / (mean_ms * 1e-3) / 1e12,
                         "peak": peak, "unit": "TFLOP/s",
                         "frac": flops / (mean_ms * 1e-3) / 1e12 / peak,
                         "traffic": read_traffic(args.workload, prefix="lse_"),
                         "kernel": "lse_kernel (persistent tcgen05)", "peak_source": note,
                         **peak_extra},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_fwd(args):
    """The fused forward (attn_fwd) on a dense workload: tensor-bound,
    value = 4*D flops per visible pair (S = Q K^T and O = P V) / time."""
    import torch
    import attention_backward_pass_gb300 as ab
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    ab.load_library()
    make, seed, desc = WORKLOADS[args.workload]
    p = make()
    Qn, Kn, Vn, _, maskn = W.make_inputs(p, seed)
    tdt = torch.bfloat16 if p.dtype == W.DTYPE_BF16 else torch.float32
    Q, K, V = (torch.from_numpy(a).to(device).to(tdt) for a in (Qn, Kn, Vn))
    mask = torch.from_numpy(maskn).to(device) if maskn is not None else None
    O = torch.empty(p.q_shape(), dtype=tdt, device=device)
    lse = torch.empty(p.lse_shape(), dtype=torch.float32, device=device)
    ws = torch.empty(ab.fwd_workspace_size(p), dtype=torch.uint8, device=device)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def step():
        ab.attn_fwd(p, Q, K, V, mask, O, lse, ws)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if ab.check_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    load_under_clock_sampling(step)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for a, b in evs:
        flush.zero_()  # L2 flush between timed steps (outside the events)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    if ab.check_device_error() != 0:
        raise RuntimeError("device error word set")
    ms = [a.elapsed_time(b) for a, b in evs]
    total = max_over_ranks(sum(ms), device)
    flops = 2.0 * MET.lse_flops(p)  # 2*D for S, 2*D for P V
    value = whole_job_rate(flops, world, args.steps, total) / 1e12
    peaks, src = load_peaks()
    peak, note, peak_extra = tensor_peak(p, device, peaks, src)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import attention as OA
        groups_all = [(b, g) for b in range(p.batch) for g in range(p.num_kv_heads)]
        f = lambda a: a.astype(np.float64)  # noqa: E731
        t0 = time.perf_counter()
        done = 0
        for grp in groups_all:
            OA.forward(p, f(Qn), f(Kn), f(Vn), maskn, groups=[grp])
            done += 1
            if time.perf_counter() - t0 > 12.0:
                break
        secs = time.perf_counter() - t0
        cpu = {"value": flops / len(groups_all) * done / secs / 1e12, "unit": "TFLOP/s",
               "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{done} of {len(groups_all)} (batch, kv-head) groups, {secs:.1f} s, "
                         "fp64 numpy"}
    if rank == 0:
        mean_ms = statistics.mean(ms)
        line = {
            "metric": FWD_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if p.dtype == W.DTYPE_BF16 else "tf32", "data": "synthetic",
            "config": {"workload": "forward of " + desc,
                       "l2": "flushed between timed steps (256 MiB write)",
                       "flops_per_step": flops, "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "tensor", "achieved": flops / (mean_ms * 1e-3) / 1e12,
                         "peak": peak, "unit": "TFLOP/s",
                         "frac": flops / (mean_ms * 1e-3) / 1e12 / peak,
                         "traffic": read_traffic(args.workload, prefix="fwd_"),
                         "kernel": "fwd_kernel (persistent tcgen05)", "peak_source": note,
                         **peak_extra},
            "cpu_baseline": cpu, "e2e": None,
            "gpu_launches": args.steps,  # fwd_kernel (V is read MN-major: no transpose)
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_e2e(p, x, dQ, dK, dV, ws, args, stream, world):
    """The same metric end to end through the public API with host buffers.

    Every step copies that step's inputs from pinned host memory to the
    device, runs attn_bwd and copies dQ, dK, dV back to pinned host memory.
    The three phases of consecutive steps overlap on three streams (inputs of
    step k+1 and outputs of step k-1 move while step k computes), with two
    device copies of the inputs and outputs so that a step never overwrites
    what another step still reads.  Value = counted flops per step / mean
    step time over the timed steps; the copy rates of each direction are
    reported beside it."""
    import torch
    import attention_backward_pass_gb300 as ab
    names = (["Q", "K", "V", "O", "dO"] + ([] if args.recompute_lse else ["LSE"])
             + (["mask"] if x["mask"] is not None else []))
    n = max(3, min(args.steps, 10))
    steps = n + 2  # the first two are untimed
    host_in = [{k: torch.empty_like(x[k], device="cpu").pin_memory() for k in names}
               for _ in range(2)]
    for hb in host_in:
        for k in names:
            hb[k].copy_(x[k])
    dev_in = [{k: torch.empty_like(x[k]) for k in names} for _ in range(2)]
    dev_out = [[torch.empty_like(t) for t in (dQ, dK, dV)] for _ in range(2)]
    host_out = [[torch.empty_like(t, device="cpu").pin_memory() for t in (dQ, dK, dV)]
                for _ in range(2)]
    h2d = sum(host_in[0][k].numel() * host_in[0][k].element_size() for k in names)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    in_done = [ev() for _ in range(steps)]
    comp_done = [ev() for _ in range(steps)]
    out_done = [ev() for _ in range(steps)]
    in_start = [ev() for _ in range(steps)]
    out_start = [ev() for _ in range(steps)]
    start = ev()

    def issue_in(k):
        s = k % 2
        with torch.cuda.stream(s_in):
            if k >= 2:  # the compute of step k-2 has read this input set
                s_in.wait_event(comp_done[k - 2])
            in_start[k].record(s_in)
            for nm in names:
                dev_in[s][nm].copy_(host_in[s][nm], non_blocking=True)
            in_done[k].record(s_in)

    torch.cuda.synchronize()
    start.record(stream)
    issue_in(0)
    for k in range(steps):
        s = k % 2
        if k + 1 < steps:
            issue_in(k + 1)
        stream.wait_event(in_done[k])
        if k >= 2:  # step k-2's outputs have left this output set
            stream.wait_event(out_done[k - 2])
        d = dev_in[s]
        ab.attn_bwd(p, d["Q"], d["K"], d["V"], d["O"], d["dO"],
                    None if args.recompute_lse else d["LSE"], d.get("mask"), *dev_out[s], ws,
                    stream=stream)
        comp_done[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[k])
            out_start[k].record(s_out)
            for t_h, t_d in zip(host_out[s], dev_out[s]):
                t_h.copy_(t_d, non_blocking=True)
            out_done[k].record(s_out)
    torch.cuda.synchronize()
    if ab.check_device_error() != 0:
        raise RuntimeError("device error word set during the end-to-end steps")
    # step k ends when its outputs are on the host; timed: steps 2 .. steps-1
    ms = out_done[1].elapsed_time(out_done[steps - 1]) / n
    ms = max_over_ranks(ms, dQ.device)
    value = MET.counted_flops(p) * world / (ms * 1e-3) / 1e12
    h2d_ms = statistics.mean(in_start[k].elapsed_time(in_done[k]) for k in range(2, steps))
    d2h_ms = statistics.mean(out_start[k].elapsed_time(out_done[k]) for k in range(2, steps))
    # the last step's outputs match the device-resident run (dQ is summed in
    # whatever order the key tiles finish, so only up to rounding: fp32
    # rounding, or one bf16 unit after the bf16 conversion)
    tol = 1e-2 if p.dtype == W.DTYPE_BF16 else 1e-5
    for t_h, t_d in zip(host_out[(steps - 1) % 2], (dQ, dK, dV)):
        a, b = t_h.to(t_d.device).float(), t_d.float()
        if float((a - b).abs().max()) > tol * max(float(b.abs().max()), 1e-30):
            raise RuntimeError("end-to-end outputs differ from the device-resident run")
    return {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "h2d_gbs": h2d / (h2d_ms * 1e-3) / 1e9, "d2h_gbs": d2h / (d2h_ms * 1e-3) / 1e9,
            "pipelining": "H2D of step k+1 and D2H of step k-1 overlap step k (three streams, "
                          "two buffer sets)"}


def read_traffic(workload, prefix="dkdv_"):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary (profiles/<prefix><workload>.md, line 'traffic_bytes_per_launch: N'),
    or None when there is no summary for this workload."""
    path = os.path.join(ROOT, "profiles", f"{prefix}{workload}.md")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            if line.strip().startswith("traffic_bytes_per_launch:"):
                try:
                    return float(line.split(":", 1)[1].split()[0])
                except ValueError:
                    return None
    return None


def run_decode(args):
    """Decode backward: memory-bound; value = algorithmic bytes / time."""
    import torch
    import attention_backward_pass_gb300 as ab
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl")
    device = torch.device("cuda", torch.cuda.current_device())
    ab.load_library()
    kv_pass = args.workload == "decode_kv"
    make, seed, desc = WORKLOADS[args.workload]
    p = make()
    k, v, d_out, logits = W.make_decode_inputs(p, seed)
    lg = torch.from_numpy(logits).to(device)
    probs = torch.softmax(lg, dim=-1).contiguous()  # input synthesis
    t = {n: torch.from_numpy(a).to(device) for n, a in (("k", k), ("v", v), ("d_out", d_out))}
    d_scores = torch.empty((p.num_seqs, p.n_heads, p.history_len), device=device)
    d_q = torch.empty((p.num_seqs, p.n_heads, p.head_dim), device=device)
    ws = ab.alloc_decode_workspace(p, device)
    stream = torch.cuda.current_stream()

    def step():
        ab.attn_bwd_decode(p, t["k"], t["v"], probs, t["d_out"], d_scores, d_q, ws)

    if kv_pass:
        # pass 2 consumes pass 1's d_scores (computed once, before timing)
        step()
        q_np = W.make_decode_queries(p, seed)
        q_t = torch.from_numpy(q_np).to(device)
        hshape = (p.num_seqs, p.history_len, p.n_kv_heads, p.head_dim)
        d_k = torch.empty(hshape, device=device)
        d_v = torch.empty(hshape, device=device)

        def step():
            ab.attn_bwd_decode_kv(p, q_t, probs, t["d_out"], d_scores, d_k, d_v)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    load_under_clock_sampling(step)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for a, b in evs:  # inputs (537 MB of K/V) are larger than L2
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    if ab.check_device_error() != 0:
        raise RuntimeError("device error word set")
    ms = [a.elapsed_time(b) for a, b in evs]
    total = sum(ms)
    total = max_over_ranks(total, device)
    nbytes = MET.decode_kv_bytes(p) if kv_pass else MET.decode_bytes(p)
    value = whole_job_rate(nbytes, world, args.steps, total) / 1e9
    peaks, src = load_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import decode as OD2
        pr = probs.cpu().numpy()
        ds_np = d_scores.cpu().numpy() if kv_pass else None
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < 10.0 and n < p.num_seqs:
            if kv_pass:
                OD2.decode_backward_kv(q_np, pr, d_out, ds_np, p.n_kv_heads, seqs=[n])
            else:
                OD2.decode_backward(k, v, pr, d_out, seqs=[n])
            n += 1
        secs = time.perf_counter() - t0
        cpu = {"value": nbytes / p.num_seqs * n / secs / 1e9, "unit": "GB/s",
               "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{n} of {p.num_seqs} sequences, {secs:.1f} s, fp64 numpy"}
    if rank == 0:
        mean_ms = statistics.mean(ms)
        line = {
            "metric": DECODE_KV_METRIC if kv_pass else DECODE_METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": desc, "l2": "inputs larger than L2",
                       "bytes_per_step": nbytes, "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": nbytes / (mean_ms * 1e-3) / 1e9,
                         "peak": peak, "unit": "GB/s",
                         "frac": nbytes / (mean_ms * 1e-3) / 1e9 / peak,
                         "traffic": read_traffic("kv" if kv_pass else "passes", prefix="decode_"),
                         "kernel": "decode_kv_kernel" if kv_pass
                         else "decode_dp_kernel + decode_dq_kernel",
                         "peak_source": f"{src} hbm_gbs"},
            "cpu_baseline": cpu, "e2e": None,
            "gpu_launches": (1 if kv_pass else 2) * args.steps, "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.lse_only and args.workload not in ("decode", "decode_kv"):
        return run_lse_only(args)
    if args.fwd and args.workload not in ("decode", "decode_kv"):
        return run_fwd(args)
    if args.workload in ("decode", "decode_kv"):
        return run_decode(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
