#!/usr/bin/env python
"""Throughput of exact attention forward + backward on GB300 through libattn.

One step = one forward (attn_fwd) and one backward (attn_bwd_preprocess,
attn_bwd_dkdv, attn_bwd_dq) over the whole workload, inputs resident in HBM.
Grouped-query and block-sparse workloads run attn_fwd_gqa / attn_bwd_gqa and
attn_fwd_sparse / attn_bwd_sparse (the backward as one call); the e4m3
workloads run attn_quantize_fp8 on Q, K, V and attn_fwd_fp8.  Throughput
counts the algorithmic FLOPs (forward 4*B*H*n^2*d, backward 10*B*H*n^2*d,
both halved for a causal mask; kept entries only for a block pattern).  The
end-to-end leg copies every step's inputs from pinned host memory and its
results back, overlapped with the kernels of neighbouring steps.  A sustained
leg then repeats the step for a few seconds, so that the clocks settle under
the power cap, and reports it against the sustained tensor peak.  Prints one
JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--mode atomic|pass|auto] [--impl ours|reference]
                  [--no-cpu-baseline] [--sustain-s SECONDS]

Under torchrun each rank runs its own copy of the workload on its GPU (every
(b, h) head is independent, so there is no collective on the data path:
weak scaling); the timed region is bracketed by barriers and the maximum
elapsed time over ranks is reported.  --impl reference times the float64 CPU
oracle on the host cores instead (rank 0 only).
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from io_aware_exact_05_gb300.flops import (attention_flops, kept_entries,  # noqa: E402
                                           sparse_attention_flops)
from io_aware_exact_05_gb300.inputs import make_block_mask, make_inputs, workload  # noqa: E402

METRIC = "attention fwd+bwd TFLOP/s (bf16, 1×GB300) and % of dense BF16 tensor peak"
METRIC_FP8 = ("attention fwd TFLOP/s with e4m3 Q/K/V/P (bf16 inputs quantised on device), "
              "1×GB300")
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "b2h16_n8k_d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# end-to-end steps: enough that the pipeline's fill and drain (one step's
# input copy before the first kernel, one result copy after the last) are a
# small share of the region
E2E_MIN_STEPS = 24


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_workload(w, rank):
    """Each rank draws its own batch: the same shapes, the seed offset by the
    rank (weak scaling: every rank processes a full workload)."""
    return w.with_shape(seed=w.seed + 7919 * rank)


def max_over_ranks(x, dist, device):
    """The largest value of x over all ranks (the job's elapsed time is its
    slowest rank's); x itself without a process group."""
    if not dist:
        return x
    import torch.distributed as tdist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step, world, steps, ms):
    """Whole-job throughput: the FLOPs every rank did over the slowest rank's time."""
    return flops_per_step * world * steps / (ms * 1e-3) / 1e12


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags)
                          if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------ reference arm
def block_mask_of(w):
    """The workload's block pattern (uint8 [nb][nb]) or None when dense."""
    return make_block_mask(w.n, *w.sparse, w.seed) if w.sparse else None


def metric_of(w):
    return METRIC_FP8 if w.fp8 else METRIC


def step_flops(w, n=None):
    """Algorithmic FLOPs of one step of w (on its first n tokens): forward +
    backward, or the forward alone for an e4m3 workload."""
    n = w.n if n is None else n
    if w.fp8:
        f = attention_flops(w.B, w.H, n, w.d, w.causal)
        return {"fwd": f["fwd"], "bwd": 0, "total": f["fwd"]}
    if w.sparse:
        nb = (n + 127) // 128
        kept = kept_entries(block_mask_of(w).numpy()[:nb, :nb], n, w.causal)
        return sparse_attention_flops(w.B, w.H, w.d, kept)
    return attention_flops(w.B, w.H, n, w.d, w.causal)


def oracle_step(w, x, heads, n_sub=None):
    """Float64 CPU oracle forward + backward over the given heads, on the
    first n_sub tokens of each (the whole head by default).  For an e4m3
    workload: per-head e4m3 quantisation of q, k, v, then the forward of the
    values the codes stand for."""
    import oracle
    from oracle import fp8

    m = w.n if n_sub is None else n_sub
    bm = block_mask_of(w)
    bm = None if bm is None else bm.numpy().astype(bool)[:(m + 127) // 128, :(m + 127) // 128]
    q = x["q"].reshape(w.B * w.H, w.n, w.d)
    k, v = (x[n].reshape(w.B * w.kv_heads, w.n, w.d) for n in ("k", "v"))
    g = w.H // w.kv_heads
    for h in heads:
        hk = (h // w.H) * w.kv_heads + (h % w.H) // g   # key/value head of query head h
        if w.fp8:
            ops = [fp8.dequantize(*fp8.quantize_per_head(t[:m].double().numpy())[:2])
                   for t in (q[h], k[hk], v[hk])]
            oracle.attention_forward_head(*ops, w.scale, w.causal)
            continue
        oracle.attention_forward_head(q[h][:m], k[hk][:m], v[hk][:m], w.scale, w.causal,
                                      None, bm)
        do = x["do"].reshape(w.B * w.H, w.n, w.d)
        oracle.attention_backward_head(q[h][:m], k[hk][:m], v[hk][:m], do[h][:m], w.scale,
                                       w.causal, bm)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def time_oracle(w, x, budget_s=12.0, max_heads=4):
    """Time the oracle on whole heads until ~budget_s of CPU work."""
    heads, t = [], 0.0
    for h in range(min(max_heads, w.B * w.H)):
        t0 = time.perf_counter()
        oracle_step(w, x, [h])
        t += time.perf_counter() - t0
        heads.append(h)
        if t >= budget_s:
            break
    f = step_flops(w)["total"] * len(heads) // (w.B * w.H)
    return {"value": f / t / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": "float64 numpy oracle, %s of %d of %d whole heads of %s "
                      "(%.1f s)" % ("e4m3 quantisation + forward" if w.fp8
                                    else "forward+backward", len(heads),
                                    w.B * w.H, w.name, t)}


def run_reference(args, w):
    """The float64 oracle on the host cores.  One step = forward + backward of
    the first n_sub tokens of one head, n_sub chosen from a calibration run so
    that warm-up + timed steps take about 90 s in total."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    x = make_inputs(w)
    cal = min(1024, w.n)
    t0 = time.perf_counter()
    oracle_step(w, x, [0], cal)
    t_cal = max(time.perf_counter() - t0, 1e-3)
    target = min(5.0, 90.0 / max(1, args.steps + args.warmup))
    n_sub = int(round(cal * (target / t_cal) ** 0.5 / 128)) * 128
    n_sub = max(128, min(w.n, n_sub))
    per_step = step_flops(w, n_sub)["total"] // (w.B * w.H)
    for i in range(args.warmup):
        oracle_step(w, x, [i % (w.B * w.H)], n_sub)
    t0 = time.perf_counter()
    for s in range(args.steps):
        oracle_step(w, x, [s % (w.B * w.H)], n_sub)
    el = time.perf_counter() - t0
    val = per_step * args.steps / el / 1e12
    sample = ("%s of the first %d of %d tokens of one head (d=%d, %s) per step, "
              "float64 numpy oracle" % ("e4m3 quantisation + forward" if w.fp8
                                        else "forward+backward", n_sub, w.n,
                                        w.d, "causal" if w.causal else "full"))
    line = {"metric": metric_of(w), "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.kv_heads, "n": w.n,
                       "d": w.d, "causal": w.causal},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("bwd_kv.cuh", "bwd_kv128.cu", "sm100.cuh"):
        h.update(open(os.path.join(ROOT, "io_aware_exact_05_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:16]


def dq_mode_used(mode, w):
    """The dQ mode a bf16 backward of workload w runs (the library's own rule
    for "auto"): the reduce-adds from the key-tile kernel for d <= 128; for
    d = 256 the spill mode (dS^T through the workspace, one GEMM) when the
    call is non-causal, dense and one key/value head per query head and the
    n x n buffer is at most 4 GiB, else the separate dQ pass."""
    if mode != "auto":
        return mode
    if w.d <= 128:
        return "atomic"
    ld = (w.n + 7) // 8 * 8
    if (not w.causal and not w.sparse and w.kv_heads == w.H
            and w.B * w.H * w.n * ld * 2 <= 4 << 30):
        return "spill"
    return "pass"


def traffic_per_launch(w):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source and this workload."""
    p = os.path.join(ROOT, "profiles", "bwd_dkdv_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    if not d.get("workload", "").startswith(w.name + ":"):
        return None
    return d.get("dram_bytes_per_launch_full_workload")


def preprocess_roofline(w, mode_used, ms, pk, src):
    """HBM roofline of the D preprocess (delta_kernel): it reads O, dO and LSE,
    writes D and LSE2 (rows padded to 128) and, in atomic dQ mode, zeroes the
    fp32 dQ accumulator."""
    rows = w.B * w.H * w.n
    rows_pad = w.B * w.H * ((w.n + 127) // 128 * 128)
    nbytes = 2 * rows * w.d * 2 + rows * 4 + 2 * rows_pad * 4
    if mode_used == "atomic":
        nbytes += rows * w.d * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak = float(pk["hbm_gbs"])
    return {"kernel": "delta_kernel (attn_bwd_preprocess)", "bound": "hbm",
            "bytes_per_launch": nbytes, "achieved": gbs, "peak": peak, "unit": "GB/s",
            "frac": gbs / peak, "peak_source": "%s hbm_gbs" % src}


def e2e_ms_pipelined(step, bufsets, hx, ho, steps, st):
    """Elapsed ms of `steps` steps through the public API with host buffers:
    every step copies its inputs from pinned host memory (hx) into one of the
    device buffer sets, runs step(bufs) on stream st and copies its results
    (the keys of ho) back to pinned host memory.  Host-to-device and
    device-to-host copies run on their own streams, so the copies of one step
    overlap the kernels of its neighbours; events keep each buffer set from
    being refilled before its step has read it, or reused before its results
    have been copied out."""
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    nb = len(bufsets)
    ready = [torch.cuda.Event() for _ in range(nb)]
    done = [torch.cuda.Event() for _ in range(nb)]
    drained = [torch.cuda.Event() for _ in range(nb)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(st)
    cin.wait_event(t0)
    cout.wait_event(t0)
    for i in range(steps):
        j = i % nb
        bufs = bufsets[j]
        if i >= nb:
            cin.wait_event(done[j])          # step i - nb has read these inputs
        with torch.cuda.stream(cin):
            for name, h in hx.items():
                bufs[name].copy_(h, non_blocking=True)
        ready[j].record(cin)
        st.wait_event(ready[j])
        if i >= nb:
            st.wait_event(drained[j])        # results of step i - nb are out
        step(bufs)
        done[j].record(st)
        cout.wait_event(done[j])
        with torch.cuda.stream(cout):
            for name, h in ho.items():
                h.copy_(bufs[name], non_blocking=True)
        drained[j].record(cout)
    st.wait_stream(cout)
    t1.record(st)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


def sustained_leg(step, bufs, ev, kernel_stage, seconds, st, gpu_index):
    """Repeat the step back to back for at least `seconds` of wall time after
    the timed region (the clocks settle under the power cap over seconds).
    Steps run in chunks of len(ev), each step with its stage events; returns
    the mean step time, the mean time of stage `kernel_stage` and the clocks
    sampled over the leg."""
    clocks = ClockSampler(gpu_index)
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    steps, total_ms, kern_ms = 0, 0.0, 0.0
    wall0 = time.perf_counter()
    while time.perf_counter() - wall0 < seconds:
        t0.record(st)
        for e in ev:
            step(bufs, e)
        t1.record(st)
        torch.cuda.synchronize()
        total_ms += t0.elapsed_time(t1)
        kern_ms += sum(e[kernel_stage].elapsed_time(e[kernel_stage + 1]) for e in ev)
        steps += len(ev)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    return {"steps": steps, "wall_s": wall, "ms_per_step": total_ms / steps,
            "kernel_ms": kern_ms / steps, "clocks": clk}


def run_ours(args, w):
    from io_aware_exact_05_gb300 import attn

    ws_n, rank, local = dist_env()
    dist = ws_n > 1
    if dist:
        import torch.distributed as tdist

        tdist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mode = {"atomic": attn.ATTN_DQ_ATOMIC, "pass": attn.ATTN_DQ_PASS,
            "spill": attn.ATTN_DQ_SPILL, "auto": attn.ATTN_DQ_AUTO}[args.mode]
    mode_used = dq_mode_used(args.mode, w)
    wr = rank_workload(w, rank)
    x = make_inputs(wr)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.n, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    buf0 = {"q": q, "k": k, "v": v, "do": do, "o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    wsb = attn.attn_bwd_gqa_workspace_size(w.B, w.H, w.kv_heads, w.n, w.d, attn.ATTN_BF16,
                                           w.causal, mode)
    work = torch.empty(wsb, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream()
    sc = w.scale
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]

    grouped = w.kv_heads != w.H
    bmask = block_mask_of(w)
    if bmask is not None:   # block-sparse: the pattern on the device, list workspaces
        bmask = bmask.to(dev)
        fws = torch.empty(attn.attn_fwd_sparse_workspace_size(w.n, w.d), dtype=torch.uint8,
                          device=dev)
        work = torch.empty(attn.attn_bwd_sparse_workspace_size(w.B, w.H, w.n, w.d,
                                                               attn.ATTN_BF16, w.causal, mode),
                           dtype=torch.uint8, device=dev)

    def step(b=buf0, e=None):
        q, k, v, do, o, lse, dq, dk, dv = (b[n] for n in ("q", "k", "v", "do", "o", "lse",
                                                           "dq", "dk", "dv"))
        if e: e[0].record(st)
        if bmask is not None:   # the sparse backward is one call: timed as the dK/dV stage
            attn.attn_fwd_sparse(q, k, v, o, lse, sc, w.causal, bmask, fws, st)
            if e: e[1].record(st); e[2].record(st)
            attn.attn_bwd_sparse(q, k, v, o, do, lse, dq, dk, dv, sc, w.causal, bmask, mode,
                                 work, st)
            if e: e[3].record(st); e[4].record(st)
            return
        if grouped:   # the grouped backward is one call: timed as the dK/dV stage
            attn.attn_fwd_gqa(q, k, v, o, lse, sc, w.causal, st)
            if e: e[1].record(st); e[2].record(st)
            attn.attn_bwd_gqa(q, k, v, o, do, lse, dq, dk, dv, sc, w.causal, mode, work, st)
            if e: e[3].record(st); e[4].record(st)
            return
        attn.attn_fwd(q, k, v, o, lse, sc, w.causal, st)
        if e: e[1].record(st)
        attn.attn_bwd_preprocess(o, do, lse, w.causal, mode, work, st)
        if e: e[2].record(st)
        attn.attn_bwd_dkdv(q, k, v, do, dk, dv, sc, w.causal, mode, work, st)
        if e: e[3].record(st)
        attn.attn_bwd_dq(q, k, v, do, dq, sc, w.causal, mode, work, st)
        if e: e[4].record(st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    rc = attn.attn_status()
    if rc:
        raise RuntimeError("device status after warm-up: " + attn.attn_strerror(rc))

    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        tdist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    n_launch0 = attn.attn_launch_count()
    t0.record(st)
    for i in range(args.steps):
        step(buf0, ev[i])
    t1.record(st)
    launches = attn.attn_launch_count() - n_launch0
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()
    clk = clocks.stop()
    el_ms = t0.elapsed_time(t1)
    el_ms = max_over_ranks(el_ms, dist, dev)
    rc = attn.attn_status()
    if rc:
        raise RuntimeError("device status after timing: " + attn.attn_strerror(rc))
    stage_ms = [sum(ev[i][s].elapsed_time(ev[i][s + 1]) for i in range(args.steps)) / args.steps
                for s in range(4)]

    fl = step_flops(w)
    per_step = fl["total"]
    value = whole_job_tflops(per_step, ws_n, args.steps, el_ms)
    pk, src = peaks()

    # ---- end to end through the public API with host buffers
    hx = {n: x[n].pin_memory() for n in ("q", "k", "v", "do")}
    ho = {n: torch.empty(buf0[n].shape, dtype=buf0[n].dtype, pin_memory=True)
          for n in ("o", "lse", "dq", "dk", "dv")}
    h2d = sum(t.numel() * t.element_size() for t in hx.values())
    d2h = sum(t.numel() * t.element_size() for t in ho.values())
    e2e_steps = args.e2e_steps or max(E2E_MIN_STEPS, args.steps)
    buf1 = {n: torch.empty_like(t) for n, t in buf0.items()}
    e2e_ms_pipelined(step, [buf0, buf1], hx, ho, 2, st)     # warm-up
    if dist:
        tdist.barrier()
    e2e_ms = e2e_ms_pipelined(step, [buf0, buf1], hx, ho, e2e_steps, st)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_val = whole_job_tflops(per_step, ws_n, e2e_steps, e2e_ms)
    rc = attn.attn_status()
    if rc:
        raise RuntimeError("device status after the end-to-end run: " + attn.attn_strerror(rc))

    # ---- sustained: the same step back to back for seconds, after the timed region
    sus = None
    if args.sustain_s > 0:
        sus = sustained_leg(step, buf0, ev, 2, args.sustain_s, st, local)
        rc = attn.attn_status()
        if rc:
            raise RuntimeError("device status after the sustained run: " + attn.attn_strerror(rc))

    if rank == 0:
        kv_ms = stage_ms[2]
        # the key-tile kernel does all five backward products when it also
        # forms dQ (atomic mode), four of them (S, dP, dV, dK) in the pass and
        # spill modes (dQ by the query-tile pass or by a GEMM over dS)
        kv_flops = fl["bwd"] if mode_used == "atomic" else fl["bwd"] * 8 // 10
        achieved = kv_flops / (kv_ms * 1e-3) / 1e12
        peak = float(pk["bf16_tflops"])
        tr = traffic_per_launch(w)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "pct_of_peak": 100.0 * value / ws_n / peak,
            "config": {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.kv_heads, "n": w.n,
                       "d": w.d, "causal": w.causal, "dq_mode": mode_used,
                       "block_pattern": ({"window": w.sparse[0], "global": w.sparse[1],
                                          "random": w.sparse[2], "block": 128}
                                         if w.sparse else None),
                       "parallelism": "replicas x%d (heads independent)" % ws_n,
                       "l2": "inputs larger than L2: Q,K,V,dO = %.0f MB per GPU vs 126 MB L2"
                             % (h2d / 1e6)},
            "stage_ms": {"fwd": stage_ms[0], "bwd_preprocess": stage_ms[1],
                         "bwd_dkdv": stage_ms[2], "bwd_dq": stage_ms[3]},
            "tflops": {"fwd": fl["fwd"] / (stage_ms[0] * 1e-3) / 1e12,
                       "bwd": fl["bwd"] / (sum(stage_ms[1:]) * 1e-3) / 1e12},
            "preprocess": preprocess_roofline(w, mode_used, stage_ms[1], pk, src)
                          if not (grouped or bmask is not None) else None,
            "roofline": {"kernel": "%s (attn_bwd_dkdv)" % (
                             "bwd_kv128_kernel" if w.d == 128 else "bwd_kv_kernel"),
                         "bound": "tensor", "flops_per_launch": kv_flops,
                         "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": tr,
                         "peak_source": "%s bf16_tflops (burst); sustained %s" % (
                             src, pk.get("bf16_tflops_sustained"))},
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "overlap": "two buffer sets; H2D, kernels and D2H on three streams"},
            "gpu_launches": launches,
            "clocks": clk,
        }
        if sus is not None:
            speak = float(pk.get("bf16_tflops_sustained", peak))
            k_ach = kv_flops / (sus["kernel_ms"] * 1e-3) / 1e12
            line["sustained"] = {
                "what": "the step repeated back to back for %.1f s after the timed region "
                        "(%d steps), CUDA events per step" % (sus["wall_s"], sus["steps"]),
                "value": per_step / (sus["ms_per_step"] * 1e-3) / 1e12, "unit": UNIT,
                "ms_per_step": sus["ms_per_step"],
                "kernel": line["roofline"]["kernel"], "kernel_ms": sus["kernel_ms"],
                "achieved": k_ach, "peak": speak, "frac": k_ach / speak,
                "peak_source": "%s bf16_tflops_sustained" % src,
                "clocks": sus["clocks"]}
        if not args.no_cpu_baseline and ws_n == 1:
            line["cpu_baseline"] = time_oracle(w, x)
        print(json.dumps(line), flush=True)
    if dist:
        tdist.barrier()
        tdist.destroy_process_group()


def run_fp8(args, w):
    """One step = per-head e4m3 quantisation of the bf16 Q, K, V on the device
    (attn_quantize_fp8, V transposed) and one FP8 forward (attn_fwd_fp8)."""
    from io_aware_exact_05_gb300 import attn

    ws_n, rank, local = dist_env()
    dist = ws_n > 1
    if dist:
        import torch.distributed as tdist

        tdist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wr = rank_workload(w, rank)
    x = make_inputs(wr)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    BH = w.B * w.H
    q8 = torch.empty(w.B, w.H, w.n, w.d, dtype=torch.float8_e4m3fn, device=dev)
    k8 = torch.empty_like(q8)
    vt8 = torch.empty(w.B, w.H, w.d, w.n, dtype=torch.float8_e4m3fn, device=dev)
    ds = [torch.empty(w.B, w.H, dtype=torch.float32, device=dev) for _ in range(3)]
    buf0 = {"q": q, "k": k, "v": v, "o": None, "lse": None}
    qws = torch.empty(max(4, attn.attn_quantize_fp8_workspace_size(BH, w.n, w.d)),
                      dtype=torch.uint8, device=dev)
    o = torch.empty(w.B, w.H, w.n, w.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.H, w.n, dtype=torch.float32, device=dev)
    buf0["o"], buf0["lse"] = o, lse
    st = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]

    def step(b=buf0, e=None):
        if e: e[0].record(st)
        attn.attn_quantize_fp8(b["q"], q8, ds[0], False, None, qws, st)
        attn.attn_quantize_fp8(b["k"], k8, ds[1], False, None, qws, st)
        attn.attn_quantize_fp8(b["v"], vt8, ds[2], True, None, qws, st)
        if e: e[1].record(st)
        attn.attn_fwd_fp8(q8, k8, vt8, b["o"], b["lse"], w.scale, w.causal, *ds, stream=st)
        if e: e[2].record(st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    rc = attn.attn_status()
    if rc:
        raise RuntimeError("device status after warm-up: " + attn.attn_strerror(rc))
    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        tdist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    n_launch0 = attn.attn_launch_count()
    t0.record(st)
    for i in range(args.steps):
        step(buf0, ev[i])
    t1.record(st)
    launches = attn.attn_launch_count() - n_launch0
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()
    clk = clocks.stop()
    el_ms = t0.elapsed_time(t1)
    el_ms = max_over_ranks(el_ms, dist, dev)
    rc = attn.attn_status()
    if rc:
        raise RuntimeError("device status after timing: " + attn.attn_strerror(rc))
    stage_ms = [sum(ev[i][s].elapsed_time(ev[i][s + 1]) for i in range(args.steps)) / args.steps
                for s in range(2)]
    per_step = step_flops(w)["total"]
    value = whole_job_tflops(per_step, ws_n, args.steps, el_ms)

    # ---- end to end: bf16 inputs from pinned host memory, O and LSE back
    hx = {n: x[n].pin_memory() for n in ("q", "k", "v")}
    ho = {n: torch.empty(buf0[n].shape, dtype=buf0[n].dtype, pin_memory=True)
          for n in ("o", "lse")}
    h2d = sum(t.numel() * t.element_size() for t in hx.values())
    d2h = sum(t.numel() * t.element_size() for t in ho.values())
    e2e_steps = args.e2e_steps or max(E2E_MIN_STEPS, args.steps)
    buf1 = {n: torch.empty_like(t) for n, t in buf0.items()}
    e2e_ms_pipelined(step, [buf0, buf1], hx, ho, 2, st)     # warm-up
    if dist:
        tdist.barrier()
    e2e_ms = e2e_ms_pipelined(step, [buf0, buf1], hx, ho, e2e_steps, st)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_val = whole_job_tflops(per_step, ws_n, e2e_steps, e2e_ms)
    rc = attn.attn_status()
    if rc:
        raise RuntimeError("device status after the end-to-end run: " + attn.attn_strerror(rc))

    if rank == 0:
        pk, src = peaks()
        # dense e4m3 peak: the measured bf16 peak x the nominal e4m3 / bf16
        # ratio (4.5 / 2.25 PFLOP/s)
        peak = 2.0 * float(pk["bf16_tflops"])
        achieved = per_step / (stage_ms[1] * 1e-3) / 1e12
        # quantiser: 2 bytes read + 1 byte written per element of Q, K, V
        q_bytes = 3 * BH * w.n * w.d * 3
        q_gbs = q_bytes / (stage_ms[0] * 1e-3) / 1e9
        line = {
            "metric": METRIC_FP8, "value": value, "unit": UNIT, "n_gpus": ws_n,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3", "data": "synthetic",
            "pct_of_peak": 100.0 * value / ws_n / peak,
            "config": {"workload": w.name, "B": w.B, "H": w.H, "n": w.n, "d": w.d,
                       "causal": w.causal,
                       "quantisation": "per-head amax/448 on device, V as [d][n], no rotation",
                       "parallelism": "replicas x%d (heads independent)" % ws_n,
                       "l2": "inputs larger than L2: Q,K,V bf16 = %.0f MB per GPU vs 126 MB L2"
                             % (h2d / 1e6)},
            "stage_ms": {"quantize_qkv": stage_ms[0], "fwd_fp8": stage_ms[1]},
            "tflops": {"fwd_fp8_kernel": achieved},
            "roofline": {"kernel": "fwd_fp8_kernel (attn_fwd_fp8)", "bound": "tensor",
                         "flops_per_launch": per_step, "achieved": achieved, "peak": peak,
                         "unit": UNIT, "frac": achieved / peak, "traffic": None,
                         "peak_source": "%s bf16_tflops (burst) x 2 (nominal e4m3/bf16)" % src},
            "quantize_roofline": {"bound": "hbm", "bytes_per_step": q_bytes, "achieved": q_gbs,
                                  "peak": float(pk["hbm_gbs"]), "unit": "GB/s",
                                  "frac": q_gbs / float(pk["hbm_gbs"])},
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "overlap": "two buffer sets; H2D, kernels and D2H on three streams"},
            "gpu_launches": launches,
            "clocks": clk,
        }
        if not args.no_cpu_baseline and ws_n == 1:
            line["cpu_baseline"] = time_oracle(w, x)
        print(json.dumps(line), flush=True)
    if dist:
        tdist.barrier()
        tdist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--mode", default="auto", choices=["atomic", "pass", "spill", "auto"],
                    help="dQ mode; auto: atomic for d <= 128, the dQ pass above; spill: "
                         "d = 256 non-causal only, dS through the workspace and a GEMM")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0,
                    help="steps of the end-to-end leg (default: max(%d, --steps))"
                         % E2E_MIN_STEPS)
    ap.add_argument("--sustain-s", type=float, default=3.0,
                    help="seconds of back-to-back steps after the timed region, reported "
                         "against the sustained peak (0: skip)")
    args = ap.parse_args()
    w = workload(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
    elif w.fp8:
        run_fp8(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
