"""Benchmark of the FP8 scaled GEMM + amax hot path on GB300.

Default workload (one "step"): the per-tensor E4M3 GEMM at LLM linear-layer
size, M = N = K = 4096, NT, bf16 out + amax, run once with fast accumulation
and once with slow accumulation (128-K chunks).  Other workloads with
--workload (tiny, blockwise, mx_e4m3, mx_e5m2, skinny_<M>[_adv]).

Prints ONE JSON line (rank 0).  `value` is whole-job TFLOP/s with inputs
resident in HBM; `e2e` is the same metric through the public API with the
operands copied from pinned host memory and C read back every step.
`--impl reference` times the CPU oracle instead (a bounded sample of the
workload on the host cores).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 scaled-GEMM TFLOP/s (+GB/s) at 1 GB300 and % of FP8/HBM roofline"
KERNEL_SOURCES = ["precision_matmul_gb300/csrc/fp8mm_kernel.cuh", "precision_matmul_gb300/csrc/ptx.cuh"]
FP8_PER_BF16 = 2.0  # nominal dense FP8 : BF16 tensor rate (4.5 : 2.25 PFLOP/s)
L2_BYTES = 129 * 10 ** 6


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def problems(name: str):
    from precision_matmul_gb300 import synth
    if name == "llm_4096":
        return [synth.llm_per_tensor(fast_accum=True), synth.llm_per_tensor(fast_accum=False)]
    if name == "llm_4096_fast":
        return [synth.llm_per_tensor(fast_accum=True)]
    if name == "llm_4096_slow":
        return [synth.llm_per_tensor(fast_accum=False)]
    if name == "tiny":
        return [synth.tiny_per_tensor()]
    if name == "blockwise":
        return [synth.blockwise()]
    if name == "mx_e4m3":
        return [synth.mx_batched(fmt=synth.E4M3)]
    if name == "mx_e5m2":
        return [synth.mx_batched(fmt=synth.E5M2)]
    if name.startswith("skinny_"):
        parts = name.split("_")
        M = int(parts[1])
        data = "adversarial" if len(parts) > 2 and parts[2] == "adv" else "gauss40"
        return [synth.skinny(M=M, data=data, fast_accum=True), synth.skinny(M=M, data=data, fast_accum=False)]
    raise SystemExit(f"unknown workload {name}")


WORKLOAD_DESC = {
    "llm_4096": "per-tensor E4M3 GEMM M=N=K=4096 NT, bf16 out + amax, fast then slow accumulation",
    "tiny": "per-tensor E4M3 GEMM M=N=K=256, fp32 out + amax, fast accumulation",
    "blockwise": "E4M3 GEMM M=8192 N=7168 K=2048, A 1x128 / B 128x128 fp32 scales, slow, bf16 out + amax",
    "mx_e4m3": "MX block-scaled batched GEMM L=4 x 4096^3 E4M3, UE8M0 per 32 along K, fp32 out + amax",
    "mx_e5m2": "MX block-scaled batched GEMM L=4 x 4096^3 E5M2, UE8M0 per 32 along K, fp32 out + amax",
}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def read_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    only if it was captured on the current kernel sources and this workload."""
    path = os.path.join(ROOT, "profiles", "fp8mm_kernel_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("kernel_sources_sha256_16") == kernel_hash():
            return t
    except Exception:
        pass
    return None


class ClockSampler:
    """SM clock and clock-event reasons sampled every 10 ms (NVML through ctypes,
    read-only queries) for the duration of the timed region."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []
        self.max_mhz = None
        self.error = None
        self._stop = None
        self._thread = None

    def _handle(self, nvml):
        import ctypes
        import torch
        count = ctypes.c_uint()
        nvml.nvmlDeviceGetCount_v2(ctypes.byref(count))
        want = None
        try:
            want = str(torch.cuda.get_device_properties(self.cuda_index).uuid)
        except Exception:
            pass
        h = ctypes.c_void_p()
        for i in range(count.value):
            if nvml.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(h)) != 0:
                continue
            buf = ctypes.create_string_buffer(96)
            if want and nvml.nvmlDeviceGetUUID(h, buf, 96) == 0 and want in buf.value.decode():
                return h
            if count.value == 1:
                return h
        nvml.nvmlDeviceGetHandleByIndex_v2(self.cuda_index, ctypes.byref(h))
        return h

    def __enter__(self):
        import ctypes
        import threading
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            h = self._handle(nvml)
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            get_reasons = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            self._stop = threading.Event()

            def loop():
                clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
                while not self._stop.is_set():
                    if nvml.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                        r = rs.value if get_reasons(h, ctypes.byref(rs)) == 0 else 0
                        self.samples.append((float(clk.value), int(r)))
                    self._stop.wait(0.01)

            self._thread = threading.Thread(target=loop, daemon=True)
            self._thread.start()
        except Exception as e:  # no NVML: report that instead of guessing
            self.error = str(e)
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [self.error or "no samples"]}
        sm = [s for s, _ in self.samples]
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.max_mhz or max(sm),
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_sample(probs, target_s=8.0, max_rows=None):
    """Time the CPU oracle on a bounded row sample of each problem; TFLOP/s."""
    import oracle
    threads = os.cpu_count() or 1
    total_flops, total_t, descr = 0.0, 0.0, []
    for p in probs:
        a, b, sa, sb = p.a.numpy(), p.b.numpy(), p.scale_a.numpy(), p.scale_b.numpy()
        rows = 8
        while True:
            t0 = time.perf_counter()
            oracle.scaled_gemm(a[:1], b[:1], sa, sb, a_fmt=p.a_fmt, b_fmt=p.b_fmt,
                               scale_mode=p.scale_mode, out_dtype=p.out_dtype, rows=(0, rows), nthreads=threads)
            dt = time.perf_counter() - t0
            if dt > 0.5 or rows >= p.M:
                break
            rows = min(p.M, rows * 4)
        per_row = dt / rows
        want = max(1, min(p.M, int(target_s / len(probs) / per_row)))
        if max_rows:
            want = min(want, max_rows)
        t0 = time.perf_counter()
        oracle.scaled_gemm(a[:1], b[:1], sa, sb, a_fmt=p.a_fmt, b_fmt=p.b_fmt, scale_mode=p.scale_mode,
                           out_dtype=p.out_dtype, rows=(0, want), nthreads=threads)
        dt = time.perf_counter() - t0
        total_t += dt
        total_flops += 2.0 * want * p.N * p.K
        descr.append(f"{p.name}: rows 0..{want} of M={p.M} (all N={p.N}, K={p.K}, batch 0)")
    return total_flops / total_t / 1e12, threads, "; ".join(descr)


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (every rank gets it); x itself on one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank: float, step_s: float, world: int) -> float:
    """Replicas: every rank does the same work per step; the job's rate is
    all ranks' work over the slowest rank's step time."""
    return world * flops_per_rank / step_s / 1e12


def run_reference(args, rank, world):
    if rank != 0:
        return
    probs = problems(args.workload)
    vals = []
    for _ in range(args.warmup):
        oracle_sample(probs, target_s=2.0)
    sample = ""
    for _ in range(args.steps):
        v, cores, sample = oracle_sample(probs, target_s=max(2.0, 60.0 / max(1, args.steps)))
        vals.append(v)
    value = statistics.median(vals)
    flops = sum(p.flops for p in probs)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": flops / (value * 1e12) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD_DESC.get(args.workload, args.workload)},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch
    import precision_matmul_gb300 as pm
    from precision_matmul_gb300 import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device(f"cuda:{local_rank}")
    probs = problems(args.workload)
    ins = []
    for p in probs:
        a, b = p.a.to(dev), p.b.to(dev)
        sa, sb = p.scale_a.to(dev), p.scale_b.to(dev)
        squeeze = p.L == 1
        if squeeze:
            a, b = a[0], b[0]
        shape = (p.M, p.N) if squeeze else (p.L, p.M, p.N)
        c = torch.empty(shape, dtype=synth.OUT_TORCH[p.out_dtype], device=dev)
        amax = torch.empty(1, dtype=torch.float32, device=dev)
        ins.append((p, a, b, sa, sb, c, amax))
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    sink = torch.empty(1, dtype=torch.int64, device=dev)

    def flush_l2():
        # Write 256 MiB (twice the L2), then read it back so that the dirty
        # lines are written back here rather than during the timed GEMM.
        flush.fill_(1)
        torch.sum(flush.view(torch.int64), dim=0, keepdim=True, out=sink)

    stream = torch.cuda.current_stream(dev)

    def call(item):
        p, a, b, sa, sb, c, amax = item
        pm.scaled_mm(a, b, sa, sb, out_dtype=synth.OUT_TORCH[p.out_dtype], use_fast_accum=p.fast_accum,
                     a_fmt=p.a_fmt, b_fmt=p.b_fmt, scale_mode=p.scale_mode, out=c, amax=amax)

    for _ in range(args.warmup):
        for it in ins:
            flush_l2()
            call(it)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    per_call = [[] for _ in ins]
    with ClockSampler(local_rank) as clk:
        t_wall = time.perf_counter()
        evs = []
        for _ in range(args.steps):
            for i, it in enumerate(ins):
                flush_l2()  # L2 flush between timed GEMMs (not timed)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call(it)
                e1.record(stream)
                evs.append((i, e0, e1))
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    for i, e0, e1 in evs:
        per_call[i].append(e0.elapsed_time(e1) / 1e3)
    step_s = max_over_ranks(sum(sum(x) for x in per_call) / args.steps, world, dev)
    flops = sum(p.flops for p in probs)
    value = whole_job_tflops(flops, step_s, world)
    err = pm.fp8mm_device_error(local_rank)
    if err:
        raise SystemExit(f"device abort recorded: {err:#x}")

    # ---- e2e through the public API: pinned host operands in, C and amax out
    host = []
    for p, a, b, sa, sb, c, amax in ins:
        ha = a.cpu().pin_memory()
        hb = b.cpu().pin_memory()
        hsa, hsb = sa.cpu().pin_memory(), sb.cpu().pin_memory()
        hc = torch.empty(c.shape, dtype=c.dtype).pin_memory()
        hm = torch.empty(1, dtype=torch.float32).pin_memory()
        host.append((p, ha, hb, hsa, hsb, hc, hm))
    h2d = sum(x[1].numel() * x[1].element_size() + x[2].numel() * x[2].element_size() +
              x[3].numel() * 4 + x[4].numel() * 4 for x in host)
    d2h = sum(x[5].numel() * x[5].element_size() + 4 for x in host)

    def e2e_step():
        for (p, ha, hb, hsa, hsb, hc, hm), (_, a, b, sa, sb, c, amax) in zip(host, ins):
            a.copy_(ha, non_blocking=True)
            b.copy_(hb, non_blocking=True)
            sa.copy_(hsa, non_blocking=True)
            sb.copy_(hsb, non_blocking=True)
            call((p, a, b, sa, sb, c, amax))
            hc.copy_(c, non_blocking=True)
            hm.copy_(amax, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3 / args.steps
    e2e_value = world * flops / e2e_s / 1e12

    if rank != 0:
        return
    # ---- roofline of the dominant kernel: the call with the largest share of the step
    hbm, bf16, bf16_sus, peak_src = read_peaks()
    fp8_peak = bf16 * FP8_PER_BF16
    plans = [pm.plan_for((p.M, p.N, p.K, p.L, p.a_fmt, p.b_fmt, p.scale_mode, p.out_dtype,
                          1 if p.fast_accum else 0, 0, 0, 0, local_rank, 0)) for p in probs]
    launches = sum(pl.kernel_launches() for pl in plans)
    call_s = [sum(x) / len(x) for x in per_call]
    dom = max(range(len(probs)), key=lambda i: call_s[i])
    algo_flops, algo_bytes = plans[dom].roofline()
    dom_s = call_s[dom]
    t_roof = max(algo_flops / (fp8_peak * 1e12), algo_bytes / (hbm * 1e9))
    bound = "tensor" if algo_flops / (fp8_peak * 1e12) >= algo_bytes / (hbm * 1e9) else "hbm"
    traffic = read_traffic()
    tr_key = f"{args.workload}:{dom}"
    if bound == "tensor":
        roof = {"bound": "tensor", "achieved": algo_flops / dom_s / 1e12, "peak": fp8_peak,
                "unit": "TFLOP/s", "frac": (algo_flops / dom_s / 1e12) / fp8_peak,
                "traffic": (traffic or {}).get(tr_key),
                "peak_source": f"{peak_src} bf16 burst {bf16:.1f} TFLOP/s x nominal FP8:BF16 ratio 2"}
    else:
        roof = {"bound": "hbm", "achieved": algo_bytes / dom_s / 1e9, "peak": hbm, "unit": "GB/s",
                "frac": (algo_bytes / dom_s / 1e9) / hbm, "traffic": (traffic or {}).get(tr_key),
                "peak_source": f"{peak_src} HBM copy bandwidth"}
    roof["kernel"] = (f"fp8mm_kernel<BN={plans[dom].info()['block_n']}, "
                      f"{'slow' if plans[dom].info()['slow'] else 'fast'}> ({probs[dom].name}, "
                      f"{'fast' if probs[dom].fast_accum else 'slow'} accumulation)")
    roof["roofline_time_us"] = t_roof * 1e6
    roof["gbs"] = algo_bytes / dom_s / 1e9
    roof["algorithmic_flops_per_launch"] = algo_flops
    roof["algorithmic_bytes_per_launch"] = algo_bytes
    per_call_ms = [1e3 * statistics.median(x) for x in per_call]
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, sample = oracle_sample(probs, target_s=args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}
    p0 = probs[0]
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8_e4m3" if p0.a_fmt == 0 else "fp8_e5m2", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC.get(args.workload, args.workload), "M": p0.M, "N": p0.N,
                       "K": p0.K, "L": p0.L, "calls_per_step": len(probs),
                       "per_call_ms": per_call_ms, "plans": [pl.info() for pl in plans],
                       "l2": "L2 flushed before every timed GEMM: 256 MiB written, then read back (not timed)",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches * args.steps, "clocks": clk.summary(), "wall_s": t_wall,
            "kernel_sources_sha256_16": kernel_hash()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llm_4096")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
