"""Benchmark of the QAT attention hot path (forward + straight-through backward).

One step = qat_attn_fwd + qat_attn_bwd over the video-DiT workload
B=1, H=40, Nq=Nkv=32768, D=128, non-causal, P fake-quantized to FP8 E4M3 per
query row x 64-key tile, on seeded synthetic N(0, 1) bf16 inputs resident in HBM.
Each input tensor (335 MB) is larger than L2 (129 MB), so no L2 flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Metric: TFLOP/s counting the algorithmic flops of the
method, 16 * pairs * D per step (forward 3 GEMMs = 6 pairs D: QK^T, quant(P) V, P V;
backward 5 GEMMs = 10 pairs D: QK^T, dO V^T, P^T dO, dS^T Q, dS K).
``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload (the host-core reference arm).  Under torchrun each rank runs its own copy of
the workload (weak scaling; no data-path collective).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "QAT attention fwd+bwd TFLOPS (% of GB300 bf16 tensor peak) at seq 32K, d=128"
UNIT = "TFLOP/s"
WORKLOAD = "c4"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def pairs_of(w) -> int:
    return w.pairs


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The maximum of a per-rank time over all ranks (the job's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as tdist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step_per_rank: float, steps: int, world: int,
                     max_ms: float) -> float:
    """Weak scaling: every rank runs its own workload; the job's throughput is all the
    ranks' work divided by the slowest rank's time."""
    return world * flops_per_step_per_rank * steps / (max_ms * 1e-3) / 1e12


def kernel_traffic(*kernels: str):
    """DRAM bytes per launch of `kernels` together at the benchmarked workload, from the
    committed ncu summary, or None when any kernel's source has changed since the capture."""
    import hashlib
    total = 0
    try:
        with open(os.path.join(ROOT, "profiles", "roofline_traffic.json")) as f:
            recs = json.load(f)
        for kernel in kernels:
            rec = recs[kernel]
            with open(os.path.join(ROOT, rec["source"]), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != rec["sha256"]:
                    return None
            total += rec["dram_bytes_per_launch"]
        return total
    except (OSError, KeyError, ValueError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def l2_note(w) -> str:
    mb = w.B * w.H * w.Nq * w.D * 2 / 1e6
    if mb > 129:
        return f"inputs larger than L2 ({mb:.1f} MB per query-side tensor vs 129 MB L2); no flush"
    return (f"inputs of {mb:.1f} MB per query-side tensor fit in the 129 MB L2 and are not "
            "flushed: a profiling case, not a measurement under the timing rules")


def workload_config(w):
    if w.name == "c4":
        what = f"video-DiT self-attention B={w.B} H={w.H} Nq=Nkv={w.Nq} D={w.D} non-causal"
    else:
        what = (f"attention B={w.B} H={w.H} Nq={w.Nq} Nkv={w.Nkv} D={w.D} "
                f"{'causal' if w.causal else 'non-causal'}")
    return {
        "workload": f"{w.name}: {what}, P fake-quant FP8 E4M3 per row x 64-key tile",
        "B": w.B, "H": w.H, "Nq": w.Nq, "Nkv": w.Nkv, "D": w.D, "causal": w.causal,
        "sm_scale": "1/sqrt(D)", "quant_mode": "fp8e4m3_row_tile64",
        "l2": l2_note(w),
        "flops_per_step": "16*pairs*D (fwd 6, bwd 10)",
    }


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()  # let nvidia-smi start up before the timed region begins
        while not self.lines and time.time() - t0 < 10.0:
            time.sleep(0.05)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle arm

def oracle_sample_tflops(w, rows: int, seed: int = 0):
    """Times the fp64 oracle on one head of the workload: ``rows`` query rows against all
    keys, forward (with quantization) and backward.  Returns (tflops, seconds, pairs)."""
    import numpy as np

    from oracle import qat_oracle as orc
    rng = np.random.default_rng(1000 * w.idx + 7 + seed)

    def bf16(shape):
        x = rng.standard_normal(size=shape, dtype=np.float32)
        u = x.view(np.uint32).astype(np.uint64)
        return orc.bf16_bits_to_f64(((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16))

    q, do = bf16((rows, w.D)), bf16((rows, w.D))
    k, v = bf16((w.Nkv, w.D)), bf16((w.Nkv, w.D))
    t0 = time.perf_counter()
    orc.head_forward(q, k, v, w.sm_scale, False, quant=True)
    orc.head_backward(q, k, v, do, w.sm_scale, False)
    dt = time.perf_counter() - t0
    pairs = rows * w.Nkv
    return 16.0 * pairs * w.D / dt / 1e12, dt, pairs


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    rows = 256
    for _ in range(args.warmup):
        oracle_sample_tflops(w, rows)
    vals, secs = [], 0.0
    for s in range(args.steps):
        tf, dt, _ = oracle_sample_tflops(w, rows, seed=s)
        vals.append(tf)
        secs += dt
    value = statistics.median(vals)
    sample = (f"one head of {w.name}: {rows} query rows x {w.Nkv} keys, D={w.D}, fp64 forward "
              f"(with FP8 quantization) + backward per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 inputs widened to fp64)",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

OTHER_WORKLOADS = ("c2", "c3", "c5a", "c5b")


def time_workload(name, dev, stream, peaks, reps: int = 20, warmup: int = 3):
    """qat_attn_fwd and qat_attn_bwd of one more workload, each timed alone with CUDA
    events on the launching stream over `reps` warm repeats (median), inputs resident."""
    import numpy as np
    import torch

    from quantization_aware_attention_gb300 import capi
    from quantization_aware_attention_gb300.inputs import WORKLOADS, make_inputs

    w = WORKLOADS[name]
    B, H, Nq, Nkv, D = w.B, w.H, w.Nq, w.Nkv, w.D
    x = {n: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
         for n, a in make_inputs(w).items()}
    o_q, o_hp, dq = (torch.empty_like(x["q"]) for _ in range(3))
    dk, dv = torch.empty_like(x["k"]), torch.empty_like(x["v"])
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    ws_bytes = capi.qat_attn_bwd_workspace_bytes(B, H, Nq, Nkv, D)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    quant = capi.QUANT_P_FP8E4M3_ROW_TILE64

    def fwd():
        st = capi.qat_attn_fwd(x["q"], x["k"], x["v"], o_q, o_hp, lse, B, H, Nq, Nkv, D,
                               w.sm_scale, int(w.causal), quant, stream)
        if st != capi.Status.OK:
            raise capi.QatError(st, "qat_attn_fwd")

    def bwd():
        st = capi.qat_attn_bwd(x["q"], x["k"], x["v"], o_hp, lse, x["do"], dq, dk, dv, B, H, Nq,
                               Nkv, D, w.sm_scale, int(w.causal), quant, ws, ws_bytes, stream)
        if st != capi.Status.OK:
            raise capi.QatError(st, "qat_attn_bwd")

    def timed(fn):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    for _ in range(warmup):
        fwd()
        bwd()
    fwd_ms = timed(fwd)
    bwd_ms = timed(bwd)
    if capi.qat_attn_device_status(stream) != capi.Status.OK:
        raise RuntimeError("a kernel reported an expired bounded wait")
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    fwd_tf = 6.0 * w.pairs * D / (fwd_ms * 1e-3) / 1e12
    bwd_tf = 10.0 * w.pairs * D / (bwd_ms * 1e-3) / 1e12
    step_tf = 16.0 * w.pairs * D / ((fwd_ms + bwd_ms) * 1e-3) / 1e12
    return {"shape": workload_config(w)["workload"], "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf, "step_tflops": step_tf,
            "fwd_frac_of_burst_peak": fwd_tf / burst, "bwd_frac_of_burst_peak": bwd_tf / burst,
            "tokens_per_s": B * Nq / ((fwd_ms + bwd_ms) * 1e-3), "reps": reps,
            "l2": l2_note(w)}


def run_ours(args, w):
    import numpy as np
    import torch
    import torch.distributed as tdist

    from quantization_aware_attention_gb300 import build as qbuild
    from quantization_aware_attention_gb300 import capi
    from quantization_aware_attention_gb300.inputs import make_inputs

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU; the library has no CPU path")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        tdist.init_process_group("nccl", device_id=dev)
    qbuild.build() if rank == 0 else None
    if world > 1:
        tdist.barrier()
    capi.lib()

    B, H, Nq, Nkv, D = w.B, w.H, w.Nq, w.Nkv, w.D
    if w.name == "custom":
        from quantization_aware_attention_gb300.inputs import custom_inputs
        inp = custom_inputs(9000, B, H, Nq, Nkv, D)
    else:
        inp = make_inputs(w)
    host = {n: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
            for n, a in inp.items()}
    del inp
    x = {n: t.to(dev) for n, t in host.items()}
    o_q = torch.empty_like(x["q"])
    o_hp = torch.empty_like(x["q"])
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    dq = torch.empty_like(x["q"])
    dk = torch.empty_like(x["k"])
    dv = torch.empty_like(x["v"])
    ws_bytes = capi.qat_attn_bwd_workspace_bytes(B, H, Nq, Nkv, D)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sm = w.sm_scale
    # fwd kernel; bwd prep, dK/dV and dQ kernels, plus the kernel that adds the dK/dV
    # segment sums when the backward runs stream-K (non-causal only; the workspace then
    # ends with the segments' partial sums, past the 72 bytes per padded query row and
    # the 4 KB ones tile of the unsplit layout)
    rows_pad = B * H * ((Nq + 127) // 128 * 128)
    up256 = lambda n: (n + 255) // 256 * 256
    base_ws = 2 * up256(rows_pad * 4) + 2 * up256(rows_pad * 32) + up256(128 * 32)
    launches_per_step = 4 + (1 if (not w.causal and ws_bytes > base_ws) else 0)

    def fwd():
        st = capi.qat_attn_fwd(x["q"], x["k"], x["v"], o_q, o_hp, lse, B, H, Nq, Nkv, D, sm,
                               int(w.causal), capi.QUANT_P_FP8E4M3_ROW_TILE64, stream)
        if st != capi.Status.OK:
            raise capi.QatError(st, "qat_attn_fwd")

    def bwd():
        st = capi.qat_attn_bwd(x["q"], x["k"], x["v"], o_hp, lse, x["do"], dq, dk, dv, B, H, Nq,
                               Nkv, D, sm, int(w.causal), capi.QUANT_P_FP8E4M3_ROW_TILE64, ws,
                               ws_bytes, stream)
        if st != capi.Status.OK:
            raise capi.QatError(st, "qat_attn_bwd")

    def barrier():
        if world > 1:
            tdist.barrier()
        torch.cuda.synchronize(dev)

    # ---- device-resident timing
    for _ in range(args.warmup):
        fwd()
        bwd()
    clocks = ClockSampler(local)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks.start()
    barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for e0, e1, e2 in ev:
        e0.record(stream)
        fwd()
        e1.record(stream)
        bwd()
        e2.record(stream)
    t_end.record(stream)
    barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    fwd_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1, _ in ev)
    bwd_ms = statistics.mean(e1.elapsed_time(e2) for _, e1, e2 in ev)
    if capi.qat_attn_device_status(stream) != capi.Status.OK:
        raise RuntimeError("a kernel reported an expired bounded wait")

    pairs = w.pairs
    flops_step = 16.0 * pairs * D
    ms_step = total_ms / args.steps
    value = whole_job_tflops(flops_step, args.steps, world, total_ms)

    # ---- end to end: host buffers, every step's copies inside the timed region.  Steps
    # are pipelined over two device buffer sets: the host-to-device copy of step i + 1 and
    # the device-to-host read of step i - 1 run on their own streams while step i computes.
    hout = {}
    if not args.no_e2e:
        hout = {n: torch.empty(host["q"].shape, dtype=torch.bfloat16).pin_memory()
                for n in ("o_q", "dq")}
        hout.update({n: torch.empty(host["k"].shape, dtype=torch.bfloat16).pin_memory()
                     for n in ("dk", "dv")})
    h2d = sum(t.numel() * t.element_size() for t in host.values()) if hout else 0
    d2h = sum(t.numel() * t.element_size() for t in hout.values())
    e2e_steps = 0 if args.no_e2e else max(3, min(args.steps, 10))
    e2e_ms = 0.0
    if e2e_steps:
        xs = [x, {n: torch.empty_like(t) for n, t in x.items()}]
        outs = [dict(o_q=o_q, o_hp=o_hp, lse=lse, dq=dq, dk=dk, dv=dv)]
        outs.append({n: torch.empty_like(t) for n, t in outs[0].items()})
        s_in = torch.cuda.Stream(dev)
        s_out = torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_cmp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def run_e2e(n_steps):
            for i in range(n_steps):
                b = i & 1
                xb, ob = xs[b], outs[b]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_cmp[b])        # step i - 2 is done with xb
                    for n, t in host.items():
                        xb[n].copy_(t, non_blocking=True)
                    ev_in[b].record(s_in)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])          # ob has been read back
                for name, st in (("qat_attn_fwd", capi.qat_attn_fwd(
                        xb["q"], xb["k"], xb["v"], ob["o_q"], ob["o_hp"], ob["lse"], B, H, Nq,
                        Nkv, D, sm, int(w.causal), capi.QUANT_P_FP8E4M3_ROW_TILE64, stream)),
                                 ("qat_attn_bwd", capi.qat_attn_bwd(
                        xb["q"], xb["k"], xb["v"], ob["o_hp"], ob["lse"], xb["do"], ob["dq"],
                        ob["dk"], ob["dv"], B, H, Nq, Nkv, D, sm, int(w.causal),
                        capi.QUANT_P_FP8E4M3_ROW_TILE64, ws, ws_bytes, stream))):
                    if st != capi.Status.OK:
                        raise capi.QatError(st, name)
                ev_cmp[b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp[b])
                    for n in ("o_q", "dq", "dk", "dv"):
                        hout[n].copy_(ob[n], non_blocking=True)
                    ev_out[b].record(s_out)
            stream.wait_event(ev_out[(n_steps - 1) & 1])
            if n_steps >= 2:
                stream.wait_event(ev_out[(n_steps - 2) & 1])

        run_e2e(2)
        barrier()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        s_in.wait_event(s0)
        run_e2e(e2e_steps)
        s1.record(stream)
        barrier()
        e2e_ms = max_over_ranks(s0.elapsed_time(s1), world, dev)
        del xs[1], outs[1]
    e2e_value = whole_job_tflops(flops_step, e2e_steps, world, e2e_ms) if e2e_steps else None

    # ---- the Q/K/V fake-quantization row (HBM-bound): channel mean of K + 3 passes
    qkv = None
    if w.name == WORKLOAD:
        fq = [torch.empty_like(x[n]) for n in ("q", "k", "v")]
        kmean = torch.empty(D, dtype=torch.float32, device=dev)

        def qkv_pass():
            capi.qat_channel_mean(x["k"], kmean, B, H, Nkv, D, stream)
            capi.qat_fake_quant_tokens(x["q"], None, fq[0], None, B, H, Nq, D, stream)
            capi.qat_fake_quant_tokens(x["k"], kmean, fq[1], None, B, H, Nkv, D, stream)
            capi.qat_fake_quant_tokens(x["v"], None, fq[2], None, B, H, Nkv, D, stream)

        for _ in range(3):
            qkv_pass()
        q0 = torch.cuda.Event(enable_timing=True)
        q1 = torch.cuda.Event(enable_timing=True)
        barrier()
        q0.record(stream)
        for _ in range(10):
            qkv_pass()
        q1.record(stream)
        barrier()
        qkv_ms = q0.elapsed_time(q1) / 10
        elem = 2  # bf16
        qkv_bytes = elem * (B * H * Nkv * D                       # K read for the mean
                            + 2 * (B * H * Nq * D + 2 * B * H * Nkv * D))  # 3 x (read + write)
        qkv = {"ms": qkv_ms, "bytes": qkv_bytes, "gbs": qkv_bytes / (qkv_ms * 1e-3) / 1e9,
               "what": "qat_channel_mean(K) + qat_fake_quant_tokens(Q, K - mean, V) at c4"}
        del fq

    # ---- the key-chunk forward + merge row: c4 as 4 chunks of Nkv / 4 keys
    chunked = None
    if w.name == WORKLOAD:
        nch = 4
        clen = Nkv // nch
        acc = [torch.empty(B, H, Nq, D, device=dev), torch.empty(B, H, Nq, D, device=dev),
               torch.empty(B, H, Nq, device=dev)]
        part = [torch.empty_like(acc[0]), torch.empty_like(acc[1]), torch.empty_like(acc[2])]
        quant = capi.QUANT_P_FP8E4M3_ROW_TILE64
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

        def chunked_pass():
            capi.qat_attn_fwd_chunk(x["q"], x["k"], x["v"], *acc, B, H, Nq, Nkv, 0, clen, D, sm,
                                    quant, stream)
            for c in range(1, nch):
                capi.qat_attn_fwd_chunk(x["q"], x["k"], x["v"], *part, B, H, Nq, Nkv, c * clen,
                                        clen, D, sm, quant, stream)
                capi.qat_attn_merge(*acc, *part, o_q if c == nch - 1 else None,
                                    o_hp if c == nch - 1 else None, B, H, Nq, D, stream)

        chunked_pass()
        barrier()
        ev[0].record(stream)
        chunked_pass()
        ev[1].record(stream)
        for c in range(1, nch):
            capi.qat_attn_merge(*acc, *part, None, None, B, H, Nq, D, stream)
        ev[2].record(stream)
        barrier()
        ch_ms = ev[0].elapsed_time(ev[1])
        merge_ms = ev[1].elapsed_time(ev[2]) / (nch - 1)
        # read acc and part, write acc: 3 x (O_q, O_hp, lse) = 3 (2D + 1) fp32 per row
        merge_bytes = 4 * B * H * Nq * 3 * (2 * D + 1)
        chunked = {"chunks": nch, "ms": ch_ms, "tflops": 6.0 * pairs_of(w) * D / (ch_ms * 1e-3) / 1e12,
                   "one_pass_fwd_ms": None, "merge_ms": merge_ms,
                   "merge_gbs": merge_bytes / (merge_ms * 1e-3) / 1e9,
                   "what": "c4 forward as 4 key chunks (fp32 partials) + 3 lse merges"}
        del acc, part

    # ---- the other workloads of the method (parity-test shapes, timed here too)
    others = None
    if w.name == WORKLOAD and not args.no_configs and world == 1:
        others = {n: time_workload(n, dev, stream, load_peaks()[0]) for n in OTHER_WORKLOADS}

    # ---- roofline of the dominant kernel work (the backward call)
    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    bwd_tf = 10.0 * pairs * D / (bwd_ms * 1e-3) / 1e12
    fwd_tf = 6.0 * pairs * D / (fwd_ms * 1e-3) / 1e12
    bwd_exec_flops = 14.0 * pairs * D + 2 * 2.0 * pairs * 16

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, see quantization_aware_attention_gb300/inputs.py)",
        "config": workload_config(w),
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
        "fwd_frac_of_burst_peak": fwd_tf / peak_burst,
        "bwd_frac_of_burst_peak": bwd_tf / peak_burst,
        "tflops_flash_convention": world * 14.0 * pairs * D * args.steps / (total_ms * 1e-3) / 1e12,
        "tokens_per_s": world * B * Nq * args.steps / (total_ms * 1e-3),
        "roofline": {
            "kernel": "qat_attn_bwd call (prep + attn_bwd_dkdv_kernel + attn_bwd_dq_kernel)",
            "bound": "tensor", "achieved": bwd_tf, "peak": peak_sus, "unit": "TFLOP/s",
            "frac": bwd_tf / peak_sus,
            "traffic": (kernel_traffic("bwd_prep_kernel", "attn_bwd_dkdv_kernel",
                                       "attn_bwd_dq_kernel")
                        if w.name == WORKLOAD else None),
            "traffic_unit": "bytes per qat_attn_bwd call: its prep, dK/dV and dQ kernels (DRAM read + write)",
            "peak_kind": f"bf16_tflops_sustained ({peak_src})",
            "algorithmic_flops_per_launch": 10.0 * pairs * D,
            # what the tensor cores execute: S and dP in both kernels (7 products) and the
            # two K=16 lse / Delta steps of the dK/dV kernel
            "executed_flops_per_launch": bwd_exec_flops,
            "executed_achieved": bwd_exec_flops / (bwd_ms * 1e-3) / 1e12,
            "executed_frac": bwd_exec_flops / (bwd_ms * 1e-3) / 1e12 / peak_sus,
        },
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "how": "pinned-host inputs copied in and O_q, dQ, dK, dV copied out every "
                       "step through the C ABI; copies on their own streams overlap the "
                       "neighbouring steps' compute (two device buffer sets)"},
        "gpu_launches": launches_per_step * args.steps,
        "next_rows": {
            "qkv_fake_quant": dict(qkv, frac_of_hbm=qkv["gbs"] / float(
                peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))) if qkv else None,
            "kv_chunk_merge": dict(chunked, one_pass_fwd_ms=fwd_ms) if chunked else None},
        "clocks": clk,
        "configs": others,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows, chunks = 2048, 4
        secs, flops = 0.0, 0.0
        for c in range(chunks):
            _, dt, pairs = oracle_sample_tflops(w, rows, seed=c)
            secs += dt
            flops += 16.0 * pairs * w.D
        line["cpu_baseline"] = {
            "value": flops / secs / 1e12, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": (f"one head of {w.name}: {chunks} x {rows} query rows x {w.Nkv} keys, fp64 "
                       f"forward (with FP8 quantization) + backward, {secs:.1f} s; numpy BLAS "
                       f"matmuls, elementwise steps single-threaded")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        tdist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end run")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other workloads (c2, c3, c5a, c5b)")
    ap.add_argument("--shape", default=None,
                    help="B,H,Nq,Nkv,D[,causal]: a smaller case for profiling instead of the "
                         "benchmarked workload")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    from quantization_aware_attention_gb300.inputs import WORKLOADS, Workload
    w = WORKLOADS[WORKLOAD]
    if args.shape:
        v = [int(x) for x in args.shape.split(",")]
        w = Workload("custom", 9, v[0], v[1], v[2], v[3], v[4], causal=bool(v[5]) if len(v) > 5 else False)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
