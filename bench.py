"""Benchmark of the rotation-based W4A4 hot path on GB300.

One step = one pass of the whole online path over one batch of synthetic input:
  1. rq_fwht_quant      X (tokens x hidden, bf16) -> INT4 codes + scales (the codes
                        stored as the product's E4M3 operand bytes; --a-form packed
                        writes them two per byte instead)
  2. rq_w4a4_gemm       codes x folded INT4 weights -> Y (tokens x out, fp16)
  3. rq_kv_rotate_quant K, V ([tokens][heads][head_dim] bf16) -> packed INT4 cache
The weights are folded and quantized once, before timing (the offline step).

Default workload: "large" -- X 4096 x 8192 bf16 (0.1% outlier channels x100),
GEMM 4096 x 8192 -> 28672, plus the KV write of 8192 tokens x 32 heads x 128 (the
largest configuration that runs on one GPU).  "prefill" (2048 x 4096 -> 14336),
"decode" and "tiny" are also available.

Output: one JSON line.  `value` is the W4A4 layer's integer-op throughput over
the whole step (2*M*N*K per step / step time, TOPS); the per-kernel figures
(GB/s of the rotation kernels, TOPS of the GEMM, roofline fractions) are in
`kernels`.  L2 is flushed (a 2x-L2 buffer is written) between timed steps,
outside the timed events.  Before the timed steps the same step runs back to back
for about a second (a clock soak) while nvidia-smi samples the clocks, so that the
clock record covers the GPU under this load; the timed steps are sampled too.

`parity` reports, on a sample of the step's rows, the codes that differ from the
oracle's (all inside the half-integer tie window, or the run fails) and the worst
per-row relative error of the rotated rows.

`--impl reference` times the CPU oracle instead (on a bounded sample of each
step's work, scaled to the same unit); it is the reference arm of this repo.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own batch (the path
shards by rows with no exchange), timing is the max over ranks and `value` the
sum of the ranks' work over that time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from rotational_w4a4_quantization_gb300 import synth  # noqa: E402

METRIC = "FWHT+INT4-quant GB/s; W4A4 GEMM TOPS; % of HBM / dense-INT8 roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 4.5 / 2.25   # nominal dense ratio (fp8 / bf16) on GB300
SLEEP_CYCLES = 400_000       # ~0.2 ms GPU-side pause between timed steps

# dram__bytes_read.sum + dram__bytes_write.sum of one launch, from the ncu captures
# summarized under profiles/ (kernel, workload, activation-code form); None where no
# capture of the current kernel exists.  Writes still in L2 when a kernel ends are
# not counted by the capture.
NCU_TRAFFIC = {
    ("w4a4_gemm", "large", "e4m3"): 161_607_168 + 202_691_584,
    ("fwht_quant", "large", "e4m3"): 67_176_960 + 3_142_912,
    ("kv_rotate_quant", "kv", None): 134_277_120 + 13_850_112,
}
PROBE_MMAS_PER_SM = 200_000   # FP8 tensor-pipe probe: ~0.1 s of back-to-back MMAs


def host_info():
    """Host cores and CPU model (the oracle's baseline is quoted with them)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        usable = len(os.sched_getaffinity(0))
    except AttributeError:
        usable = os.cpu_count()
    return {"host_cores": os.cpu_count(), "host_cores_usable": usable, "host_cpu": model}


# --------------------------------------------------------------------------
# work accounting (algorithmic bytes / ops)
# --------------------------------------------------------------------------

def fwht_bytes(rows, n, in_bytes=2, code_bytes_per_elem=0.5):
    """Read the row once, write its codes (packed: n/2 bytes; operand form: n)
    and its scale (operand form: the scale and the row's code sum)."""
    return rows * (n * in_bytes + int(n * code_bytes_per_elem) + (8 if code_bytes_per_elem == 1.0 else 4))


def gemm_ops(M, N, K):
    return 2 * M * N * K


def gemm_bytes(M, N, K, out_bytes=2):
    return M * K // 2 + N * K // 2 + 4 * M + 4 * N + out_bytes * M * N


def kv_bytes(T, H, D, in_bytes=2):
    return 2 * T * H * (D * in_bytes + D // 2 + 4)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# --------------------------------------------------------------------------
# distributed helpers (weak scaling, no data-path collective)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_units: float, local_seconds: float, group=None):
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time.  Returns (total_units, max_seconds)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_units, local_seconds
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(u.item()), float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

def gpu_selector(dev, local):
    """nvidia-smi -i argument for this device (its UUID when torch exposes it)."""
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    if uuid:
        u = str(uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    return str(local)


class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="rq_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, timed=None):
        """Median SM clock, max clock and throttle reasons over every sample; with
        `timed` = (t0, t1) wall-clock seconds, also how many samples fell inside."""
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        import datetime
        sm, mx, reasons, stamps = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm.append(float(parts[2]))
                    mx.append(float(parts[3]))
                except ValueError:
                    continue
                try:
                    stamps.append(datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp())
                except ValueError:
                    stamps.append(None)
                for name, val in zip(names, parts[6:10]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
               "samples": len(sm)}
        if timed is not None:
            inside = [c for c, t in zip(sm, stamps) if t is not None and timed[0] <= t <= timed[1]]
            out["samples_in_timed_steps"] = len(inside)
            if inside:
                out["sm_mhz_timed_steps"] = statistics.median(inside)
        return out


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------

def make_inputs(work, kvw, dev):
    x = synth.activations(work.rows, work.n, work.x_dtype, work.data_seed, work.n_outliers,
                          work.outlier_factor)
    wt = synth.weights_t(work.gemm_n, work.n, work.weight_seed, work.w_std)
    k, v = synth.kv_pair(kvw.kv_tokens, kvw.kv_heads, kvw.kv_head_dim, kvw.data_seed,
                         kvw.kv_outliers_per_head, kvw.kv_outlier_factor)
    return x, wt, k, v


def run_gpu(args, work, kvw):
    import rotational_w4a4_quantization_gb300 as rq
    import __graft_entry__

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        __graft_entry__.build()
    barrier()
    rq.load_library()

    seed, flags = synth.SIGN_SEED, rq.RQ_SIGNS_FIRST
    M, K, N = work.rows, work.n, work.gemm_n
    e4 = args.a_form == "e4m3"                      # activation codes as the product's operand bytes
    aflags = flags | (rq.RQ_E4M3_CODES if e4 else 0)
    T, H, D = kvw.kv_tokens, kvw.kv_heads, kvw.kv_head_dim
    x_cpu, wt_cpu, k_cpu, v_cpu = make_inputs(work, kvw, dev)
    x, k, v = x_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev)

    # offline fold + weight quantization (not timed)
    wq, ws = rq.fwht_quant(wt_cpu.to(dev), seed, flags)
    del wt_cpu

    # preallocated outputs
    aq = torch.empty(M, K if e4 else K // 2, dtype=torch.uint8, device=dev)
    as_ = torch.empty((M, 2) if e4 else (M,), dtype=torch.float32, device=dev)   # e4m3: (scale, code sum) per row
    y = torch.empty(M, N, dtype=torch.float16, device=dev)
    kv_out = {"kq": torch.empty(T, H, D // 2, dtype=torch.uint8, device=dev),
              "ks": torch.empty(T, H, dtype=torch.float32, device=dev),
              "vq": torch.empty(T, H, D // 2, dtype=torch.uint8, device=dev),
              "vs": torch.empty(T, H, dtype=torch.float32, device=dev)}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        rq.fwht_quant(x, seed, aflags, q=aq, scales=as_)
        if ev:
            ev[1].record(stream)
        rq.w4a4_gemm(aq, as_, wq, ws, out=y)
        if ev:
            ev[2].record(stream)
        rq.kv_rotate_quant(k, v, seed, flags, out=kv_out)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    assert rq.sync_status() == 0

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_selector(dev, local)) as clk:
        # clock soak: the same step back to back for about args.soak seconds, so
        # that the clocks are sampled under this load (untimed)
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < args.soak:
            for _ in range(8):
                step()
            torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        w0 = time.time()
        for i in range(args.steps):
            flush.fill_(float(i))
            # keep the GPU busy while the host enqueues the step, so the step's
            # events measure kernels, not host launch latency (outside the events)
            torch.cuda._sleep(SLEEP_CYCLES)
            step(events[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        w1 = time.time()
        time.sleep(0.15)                     # let the sampler write its last sample
    barrier()
    clocks = clk.summary(timed=(w0, w1))

    per = {"fwht": [], "gemm": [], "kv": [], "step": []}
    for ev in events:
        per["fwht"].append(ev[0].elapsed_time(ev[1]) / 1e3)
        per["gemm"].append(ev[1].elapsed_time(ev[2]) / 1e3)
        per["kv"].append(ev[2].elapsed_time(ev[3]) / 1e3)
        per["step"].append(ev[0].elapsed_time(ev[3]) / 1e3)
    step_s = sum(per["step"])
    ops_step = gemm_ops(M, N, K)
    total_ops, max_s = aggregate(ops_step * args.steps, step_s)

    # end to end through the public API: host inputs in, host results out.  Two
    # device buffer sets and three streams (copies in, kernels, copies out): step
    # i's kernels overlap step i+1's input copies and step i-1's output copies.
    # Every step's copies stay inside the timed region.
    x_h = x_cpu.pin_memory()
    k_h, v_h = k_cpu.pin_memory(), v_cpu.pin_memory()
    y_h = torch.empty(M, N, dtype=torch.float16).pin_memory()
    kvh = {key: torch.empty(t.shape, dtype=t.dtype).pin_memory() for key, t in kv_out.items()}
    h2d = x_h.numel() * x_h.element_size() + 2 * k_h.numel() * k_h.element_size()
    d2h = y_h.numel() * 2 + sum(t.numel() * t.element_size() for t in kvh.values())
    bufs = [{"x": x, "k": k, "v": v, "aq": aq, "as": as_, "y": y, "kv": kv_out}]
    bufs.append({"x": torch.empty_like(x), "k": torch.empty_like(k), "v": torch.empty_like(v),
                 "aq": torch.empty_like(aq), "as": torch.empty_like(as_), "y": torch.empty_like(y),
                 "kv": {key: torch.empty_like(t) for key, t in kv_out.items()}})
    s_in, s_run, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        j = i % 2
        b = bufs[j]
        if i >= 2:
            s_in.wait_event(ev_run[j])      # step i-2's kernels have read these inputs
        with torch.cuda.stream(s_in):
            b["x"].copy_(x_h, non_blocking=True)
            b["k"].copy_(k_h, non_blocking=True)
            b["v"].copy_(v_h, non_blocking=True)
        ev_in[j].record(s_in)
        s_run.wait_event(ev_in[j])
        if i >= 2:
            s_run.wait_event(ev_out[j])     # step i-2's outputs have been copied out
        rq.fwht_quant(b["x"], seed, aflags, q=b["aq"], scales=b["as"], stream=s_run)
        rq.w4a4_gemm(b["aq"], b["as"], wq, ws, out=b["y"], stream=s_run)
        rq.kv_rotate_quant(b["k"], b["v"], seed, flags, out=b["kv"], stream=s_run)
        ev_run[j].record(s_run)
        s_out.wait_event(ev_run[j])
        with torch.cuda.stream(s_out):
            y_h.copy_(b["y"], non_blocking=True)
            for key in kvh:
                kvh[key].copy_(b["kv"][key], non_blocking=True)
        ev_out[j].record(s_out)

    for i in range(max(2, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(s_in)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(s_out)                         # after the last step's output copies
    torch.cuda.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3
    e2e_ops, e2e_max = aggregate(ops_step * args.steps, e2e_s)
    assert rq.sync_status() == 0

    # the FP8 tensor pipe alone, at this run's clocks (after the timed steps)
    probe = probe_f8_pipe(stream)
    parity = parity_sample(work, kvw, x_cpu, k_cpu, v_cpu, x, k, v, aq, as_, kv_out, e4) if rank == 0 else None

    if rank != 0:
        return None

    peaks = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    avg = {key: sum(vals) / len(vals) for key, vals in per.items()}
    fb = fwht_bytes(M, K, code_bytes_per_elem=1.0 if e4 else 0.5)
    gb_ops = gemm_ops(M, N, K)
    kb = kv_bytes(T, H, D)
    kernels = {
        "fwht_quant": {"us": avg["fwht"] * 1e6, "GB/s": fb / avg["fwht"] / 1e9,
                       "frac_hbm": fb / avg["fwht"] / 1e9 / peaks["hbm_gbs"], "bytes": fb},
        "w4a4_gemm": {"us": avg["gemm"] * 1e6, "TOPS": gb_ops / avg["gemm"] / 1e12,
                      "frac_fp8_tensor": gb_ops / avg["gemm"] / 1e12 / fp8_peak, "ops": gb_ops,
                      "GB/s": gemm_bytes(M, N, K) / avg["gemm"] / 1e9},
        "kv_rotate_quant": {"us": avg["kv"] * 1e6, "GB/s": kb / avg["kv"] / 1e9,
                            "frac_hbm": kb / avg["kv"] / 1e9 / peaks["hbm_gbs"], "bytes": kb},
    }
    # dominant kernel by time
    dom = max(("fwht", "gemm", "kv"), key=lambda key: avg[key])
    kernels["w4a4_gemm"]["frac_fp8_pipe_probe"] = (gb_ops / avg["gemm"] / 1e12 / probe["tflops"]
                                                   if probe else None)
    if dom == "gemm":
        ach = gb_ops / avg["gemm"] / 1e12
        roof = {"kernel": "w4a4_gemm", "bound": "tensor", "achieved": ach, "peak": fp8_peak,
                "unit": "TFLOP/s", "frac": ach / fp8_peak,
                "traffic": NCU_TRAFFIC.get(("w4a4_gemm", work.name, args.a_form)),
                "peak_source": f"{peaks['source']} bf16 burst x {FP8_OVER_BF16} (fp8 dense ratio)",
                "fp8_pipe_probe": probe,
                "frac_fp8_pipe_probe": ach / probe["tflops"] if probe else None}
    else:
        key = "fwht_quant" if dom == "fwht" else "kv_rotate_quant"
        b = fb if dom == "fwht" else kb
        ach = b / avg[dom] / 1e9
        roof = {"kernel": key, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                "traffic": NCU_TRAFFIC.get((key, work.name, args.a_form) if key == "fwht_quant" else (key, "kv", None)),
                "peak_source": f"{peaks['source']} hbm copy"}

    line = {
        "metric": METRIC,
        "value": total_ops / max_s / 1e12,
        "unit": "TOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": max_s / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int4",
        "data": "synthetic",
        "config": bench_config(work, kvw, world, args.a_form),
        "kernels": kernels,
        "parity": parity,
        "roofline": roof,
        "e2e": {"value": e2e_ops / e2e_max / 1e12, "unit": "TOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "wall_s_timed_loop": wall,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(work, kvw, budget_s=args.cpu_budget)
    return line


def probe_f8_pipe(stream):
    """Rate of the FP8 tensor pipe alone (M128 N256 K32 MMAs back to back on every
    SM), timed with events on `stream`: the ceiling of the pipe the GEMM runs on,
    at this run's clocks.  Median of 3 after one warm-up."""
    import rotational_w4a4_quantization_gb300 as rq
    ctas = rq.probe_f8_mma(1000, stream=stream)
    times = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ctas = rq.probe_f8_mma(PROBE_MMAS_PER_SM, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    if rq.sync_status() != 0:
        return None
    t = statistics.median(times)
    flops = 2 * 128 * 256 * 32 * PROBE_MMAS_PER_SM * ctas
    return {"tflops": flops / t / 1e12, "mmas_per_sm": PROBE_MMAS_PER_SM, "ctas": ctas,
            "shape": "M128 N256 K32 kind::f8f6f4 (e4m3), zeros in shared memory"}


def parity_sample(work, kvw, x_cpu, k_cpu, v_cpu, x, k, v, aq, as_, kv_out, e4, rows=64, kv_tokens=64):
    """Codes of a sample of the step's rows against the oracle's (first and last
    `rows` activation rows, first and last `kv_tokens` tokens of K and V): the
    number of codes that differ (each must lie in the half-integer tie window and
    differ by one, else this raises), and the worst per-row relative error of the
    rotated rows, read back through the fp32 output of a separate call."""
    import oracle
    import rotational_w4a4_quantization_gb300 as rq

    def decode(packed):
        b = packed.astype(np.int16)
        nib = np.stack([b & 15, b >> 4], axis=-1).reshape(packed.shape[0], -1)
        return np.where(nib >= 8, nib - 16, nib)

    def decode_operand(ob):
        # operand bytes: sign in bit 7, |q| in bits 0..3; codes 0,2,4,6,1,3,5,7 of each group of 8
        b = ob.astype(np.int16).reshape(ob.shape[0], -1, 8)
        q = np.where(b & 0x80, -(b & 0x7F), b & 0x7F)
        out = np.empty_like(q)
        out[..., 0::2] = q[..., :4]
        out[..., 1::2] = q[..., 4:]
        return out.reshape(ob.shape[0], -1)

    def diff_count(gq, ref, operand=False):
        g, r = (decode_operand(gq) if operand else decode(gq)), decode(ref["q"])
        d = g != r
        tie = oracle.tie_mask(ref["ratio"])
        bad = d & ~(tie & (np.abs(g - r) == 1))
        if bad.any():
            raise AssertionError(f"{int(bad.sum())} sampled codes differ outside the tie window")
        return int(d.sum()), int(tie.sum())

    oracle.build()
    seed, flags = synth.SIGN_SEED, 1
    M, n = x_cpu.shape
    sel = np.unique(np.r_[np.arange(min(rows, M)), np.arange(max(0, M - rows), M)])
    ref = oracle.fwht_quant(x_cpu[sel].double().numpy(), seed, flags, want_y=True, want_ratio=True)
    gq = aq[torch.from_numpy(sel).to(aq.device)].cpu().numpy()
    a_diff, a_tie = diff_count(gq, ref, operand=e4)
    if e4:
        # the code sum beside each scale, exact for the codes written
        sums = as_[torch.from_numpy(sel).to(as_.device), 1].cpu().numpy()
        if not np.array_equal(sums, decode_operand(gq).astype(np.int64).sum(axis=1).astype(np.float32)):
            raise AssertionError("sampled row code sums differ from the codes written")
    _, _, ygpu = rq.fwht_quant(x[torch.from_numpy(sel).to(x.device)].contiguous(), seed, flags, want_y=True)
    yg = ygpu.cpu().double().numpy()
    err = (np.abs(yg - ref["y"]).max(axis=1) / np.abs(ref["y"]).max(axis=1)).max()
    T, H, D = k_cpu.shape
    tsel = np.unique(np.r_[np.arange(min(kv_tokens, T)), np.arange(max(0, T - kv_tokens), T)])
    kv_diff, kv_tie = 0, 0
    for src, qk in ((k_cpu, "kq"), (v_cpu, "vq")):
        rr = oracle.fwht_quant(src[tsel].reshape(-1, D).double().numpy(), seed, flags, want_ratio=True)
        dd, tt = diff_count(kv_out[qk][torch.from_numpy(tsel).to(k.device)].reshape(-1, D // 2).cpu().numpy(), rr)
        kv_diff += dd
        kv_tie += tt
    return {"activation_rows": int(sel.size), "activation_codes": int(sel.size) * n,
            "activation_codes_differing": a_diff, "activation_codes_in_tie_window": a_tie,
            "fwht_max_row_rel_err": float(err), "fwht_tolerance": 1e-5,
            "kv_vectors": int(tsel.size) * H * 2, "kv_codes_differing": kv_diff, "kv_codes_in_tie_window": kv_tie,
            "tie_window": 1e-4,
            "gemm": "bit-exact int32 on the full output of every workload: GPU tests (oracle over row blocks)"}


def bench_config(work, kvw, world, a_form="e4m3"):
    """The `config` object, the same for both arms."""
    return {"workload": workload_desc(work, kvw),
            "activation_codes": ("INT4 codes stored as the product's E4M3 operand bytes (1 byte per code)"
                                 if a_form == "e4m3" else "INT4 codes packed two per byte"),
            "l2": "flushed between timed steps (2x L2 write, outside timed events)",
            "parallelism": f"replicas x{world}" if world > 1 else "none (one process)"}


# --------------------------------------------------------------------------
# the CPU oracle as baseline / reference arm
# --------------------------------------------------------------------------

def _oracle_sample(work, kvw, gemm_rows, fwht_rows, kv_tokens):
    """Time the oracle on a bounded sample of one step; return seconds for the
    whole step extrapolated by rows (every part is linear in rows)."""
    import oracle
    oracle.build()
    seed, flags = synth.SIGN_SEED, 1
    M, K, N = work.rows, work.n, work.gemm_n
    x = synth.activations(fwht_rows, K, work.x_dtype, work.data_seed, work.n_outliers,
                          work.outlier_factor).double().numpy()
    t0 = time.perf_counter()
    oracle.fwht_quant(x, seed, flags)
    t_fwht = (time.perf_counter() - t0) * (M / fwht_rows)
    aq, sa = synth.random_codes(gemm_rows, K, 1)
    wq, sw = synth.random_codes(N, K, 2)
    t0 = time.perf_counter()
    oracle.w4a4_gemm(aq.numpy(), sa.numpy(), wq.numpy(), sw.numpy(), gemm_rows, N, K)
    t_gemm = (time.perf_counter() - t0) * (M / gemm_rows)
    kk, vv = synth.kv_pair(kv_tokens, kvw.kv_heads, kvw.kv_head_dim, kvw.data_seed)
    kk, vv = kk.double().numpy(), vv.double().numpy()
    t0 = time.perf_counter()
    oracle.kv_rotate_quant(kk, vv, seed, flags)
    t_kv = (time.perf_counter() - t0) * (kvw.kv_tokens / kv_tokens)
    return t_fwht + t_gemm + t_kv, {"fwht_s": t_fwht, "gemm_s": t_gemm, "kv_s": t_kv}


def cpu_baseline(work, kvw, budget_s=15.0):
    # sample sizes: about budget_s of single-core work in total
    gemm_rows = max(1, int(budget_s * 0.5e9 / (work.gemm_n * work.n)))
    step_s, parts = _oracle_sample(work, kvw, gemm_rows=gemm_rows, fwht_rows=64, kv_tokens=256)
    ops = gemm_ops(work.rows, work.gemm_n, work.n)
    return {"value": ops / step_s / 1e12, "unit": "TOPS", "cores": 1, "kind": "oracle",
            "sample": f"oracle (fp64 C, 1 thread) on {gemm_rows} GEMM rows, 64 rotation rows, "
                      f"256 KV tokens; scaled by rows to one full step",
            "step_seconds_extrapolated": step_s, "parts_s": parts, **host_info()}


def workload_desc(work, kvw):
    """The step's workload, named the same way by both arms."""
    return (f"{work.name}: X {work.rows}x{work.n} bf16 -> fwht+int4 -> W4A4 GEMM "
            f"{work.rows}x{work.n}x{work.gemm_n} fp16; kv {kvw.kv_tokens}x{kvw.kv_heads}x{kvw.kv_head_dim} bf16 K,V")


def run_reference(args, work, kvw):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    gemm_rows = 2 if args.steps <= 50 else 1     # keeps a long run within a few minutes
    for _ in range(args.warmup):
        _oracle_sample(work, kvw, gemm_rows, 16, 64)
    total = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s, _parts = _oracle_sample(work, kvw, gemm_rows, 16, 64)
        total += s
    wall = time.perf_counter() - t0
    ops = gemm_ops(work.rows, work.gemm_n, work.n)
    value = ops * args.steps / total / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wall / args.steps * 1e3,          # measured: one sampled step
        "full_step_ms_extrapolated": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int4",
        "data": "synthetic",
        "config": bench_config(work, kvw, world, args.a_form),
        "cpu_baseline": {"value": value, "unit": "TOPS", "cores": 1, "kind": "oracle",
                         "sample": f"each step: {gemm_rows} GEMM rows, 16 rotation rows, 64 KV tokens, "
                                   "scaled by rows to one full step; one host core",
                         **host_info()},
        "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200,
                    help="timed steps (200 large steps span ~0.15 s: several clock samples fall inside)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["rq", "reference"], default="rq")
    ap.add_argument("--workload", choices=["prefill", "large", "decode", "tiny"], default="large")
    ap.add_argument("--soak", type=float, default=1.5, help="seconds of untimed steps while clocks are sampled")
    ap.add_argument("--a-form", choices=["e4m3", "packed"], default="e4m3",
                    help="activation codes between the rotation and the product: the product's E4M3 operand "
                         "bytes (default) or packed INT4 nibbles")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    work = synth.WORKLOADS[args.workload]
    kvw = synth.KV
    line = run_reference(args, work, kvw) if args.impl == "reference" else run_gpu(args, work, kvw)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
