"""Benchmark of the FP8 scaled GEMM + amax hot path on GB300.

One "step" (the default workload, ``all``) is one call of every workload the
metric is quoted on, each with its own synthetic inputs resident in HBM:

  c1    per-tensor E4M3 256^3, fp32 out, fast accumulation
  c2    per-tensor E4M3 4096^3 NT, bf16 out, fast and slow accumulation
  c3    E4M3 8192 x 7168 x 2048, A 1x128 / B 128x128 fp32 scales, slow, bf16 out
  c4    MX batch 4 x 4096^3 (UE8M0 per 32 along K), fp32 out, E4M3 and E5M2
  c5    skinny N = 28672, K = 8192, M in {16, 64, 256, 1024, 2048, 8192},
        per-tensor E4M3 gauss40, bf16 out, fast and slow accumulation

every call with the fused amax.  ``value`` is the whole step's TFLOP/s (all
calls' flops over the sum of their device times); ``per_config`` reports every
call against its own roofline (tensor-bound: of the FP8 peak; HBM-bound: of
the copy bandwidth); ``roofline`` is the dominant call of the step.
``next_rows`` times, apart from the step, the forms beyond the five
configurations: an FP8 output, a bias, the NN layout, NVFP4 / MXFP4 operands
and a batched GEMM with b given K-outermost.  ``e2e``
is the same metric through the public API with the step's operands copied
from pinned host memory (once per operand set: the fast and slow calls of one
draw share theirs) and every call's C and amax read back, inside the timed
region (copies on their own streams, overlapping the GEMMs as a user's
pipeline would).
``--impl reference`` times the CPU oracle instead (a bounded sample of every
call on the host cores).  Subsets with ``--workload`` (comma-separated names
or groups: c1 .. c5, mx, skinny, or a single call name).

Prints ONE JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import dataclasses
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
# the kernels and the planner (tile shapes and raster decide the DRAM traffic a capture records)
KERNEL_SOURCES = ["precision_matmul_gb300/csrc/fp8mm_kernel.cuh", "precision_matmul_gb300/csrc/ptx.cuh",
                  "precision_matmul_gb300/csrc/fp8mm_host.cu", "precision_matmul_gb300/csrc/fp8mm_aux.cu"]
FP8_PER_BF16 = 2.0  # nominal dense FP8 : BF16 tensor rate (4.5 : 2.25 PFLOP/s)
FP8_NOMINAL_TFLOPS = 4500.0
FP4_PER_BF16 = 6.0  # nominal dense FP4 : BF16 tensor rate on GB300 (13.5 : 2.25 PFLOP/s)
L2_BYTES = 129 * 10 ** 6
SKINNY_M = (16, 64, 256, 1024, 2048, 8192)


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# name -> (description, factory); factories sharing a key in `_SHARED` reuse one input draw
def _catalogue():
    from precision_matmul_gb300 import synth
    cat = {
        "c1_tiny_256": ("per-tensor E4M3 256^3, fp32 out, fast", lambda: synth.tiny_per_tensor()),
        "c2_llm4096_fast": ("per-tensor E4M3 4096^3 NT, bf16 out, fast",
                            lambda: synth.llm_per_tensor(fast_accum=True)),
        "c2_llm4096_slow": ("per-tensor E4M3 4096^3 NT, bf16 out, slow (128-K chunks)",
                            lambda: synth.llm_per_tensor(fast_accum=False)),
        "c3_blockwise": ("E4M3 8192x7168x2048, A 1x128 / B 128x128 fp32 scales, slow, bf16 out",
                         lambda: synth.blockwise()),
        "c4_mx_e4m3": ("MX 4 x 4096^3 E4M3, UE8M0 per 32 along K, fp32 out",
                       lambda: synth.mx_batched(fmt=synth.E4M3)),
        "c4_mx_e5m2": ("MX 4 x 4096^3 E5M2, UE8M0 per 32 along K, fp32 out",
                       lambda: synth.mx_batched(fmt=synth.E5M2)),
        # rows beyond the five configurations (timed apart from the metric's step)
        "n1_fp8out_e4m3_4096": ("per-tensor E4M3 4096^3, E4M3 out with scale_result, fast",
                                lambda: _fp8out_4096()),
        "n2_bias_bf16_4096": ("per-tensor E4M3 4096^3, bf16 out + bias [N], fast",
                              lambda: synth.llm_per_tensor(fast_accum=True)),
        "n2_layout_nn_4096": ("per-tensor E4M3 4096^3 NN (b stored [K][N]: K-major copy first), bf16, fast",
                              lambda: synth.llm_per_tensor(fast_accum=True)),
        "n3_nvfp4_4x4096": ("NVFP4 4 x 4096^3 (E2M1, E4M3 factors per 16), fp32 out",
                            lambda: synth.fp4_batched(form="nv16")),
        "n3_mxfp4_4x4096": ("MXFP4 4 x 4096^3 (E2M1, UE8M0 factors per 32), fp32 out",
                            lambda: synth.fp4_batched(form="mx32")),
        "n4_bmm_bkn_4x4096": ("batched per-tensor E4M3 4 x 4096^3 with b as [B][K][N] (BmmFP8FwdOp), bf16",
                              lambda: synth.llm_per_tensor(L=4, fast_accum=True)),
    }
    for M in SKINNY_M:
        for fast in (True, False):
            mode = "fast" if fast else "slow"
            cat[f"c5_skinny_M{M}_{mode}"] = (f"per-tensor E4M3 M={M} N=28672 K=8192 gauss40, bf16 out, {mode}",
                                             (M, "gauss40", fast))
            cat[f"c5_skinny_M{M}_adv_{mode}"] = (
                f"per-tensor E4M3 M={M} N=28672 K=8192 adversarial, bf16 out, {mode}", (M, "adversarial", fast))
    return cat


# extra arguments of the next-row calls
EXTRA = {"n1_fp8out_e4m3_4096": {"scale_result": 1.0}, "n2_bias_bf16_4096": {"bias": True},
         "n2_layout_nn_4096": {"b_major": True}, "n4_bmm_bkn_4x4096": {"b_major": True}}
NEXT = ["n1_fp8out_e4m3_4096", "n2_bias_bf16_4096", "n2_layout_nn_4096", "n3_nvfp4_4x4096", "n3_mxfp4_4x4096",
        "n4_bmm_bkn_4x4096"]


def _fp8out_4096():
    from precision_matmul_gb300 import synth
    p = synth.llm_per_tensor(fast_accum=True, out_dtype=synth.OUT_E4M3)
    p.scale_a.fill_(2.0 ** -8)
    p.scale_b.fill_(2.0 ** -7)
    return p


DEFAULT = (["c1_tiny_256", "c2_llm4096_fast", "c2_llm4096_slow", "c3_blockwise", "c4_mx_e4m3", "c4_mx_e5m2"] +
           [f"c5_skinny_M{M}_{m}" for M in SKINNY_M for m in ("fast", "slow")])
GROUPS = {
    "all": DEFAULT,
    "c1": ["c1_tiny_256"], "tiny": ["c1_tiny_256"],
    "c2": ["c2_llm4096_fast", "c2_llm4096_slow"], "llm_4096": ["c2_llm4096_fast", "c2_llm4096_slow"],
    "llm_4096_fast": ["c2_llm4096_fast"], "llm_4096_slow": ["c2_llm4096_slow"],
    "c3": ["c3_blockwise"], "blockwise": ["c3_blockwise"],
    "c4": ["c4_mx_e4m3", "c4_mx_e5m2"], "mx": ["c4_mx_e4m3", "c4_mx_e5m2"],
    "mx_e4m3": ["c4_mx_e4m3"], "mx_e5m2": ["c4_mx_e5m2"],
    "c5": [f"c5_skinny_M{M}_{m}" for M in SKINNY_M for m in ("fast", "slow")],
    "next": NEXT,
}
for _M in SKINNY_M:
    GROUPS[f"skinny_{_M}"] = [f"c5_skinny_M{_M}_fast", f"c5_skinny_M{_M}_slow"]
    GROUPS[f"skinny_{_M}_adv"] = [f"c5_skinny_M{_M}_adv_fast", f"c5_skinny_M{_M}_adv_slow"]


def workload_names(spec: str) -> list:
    names = []
    cat = _catalogue()
    for part in spec.split(","):
        part = part.strip()
        got = GROUPS.get(part, [part] if part in cat else None)
        if got is None:
            raise SystemExit(f"unknown workload {part}")
        names += [n for n in got if n not in names]
    return names


def problems(spec: str):
    """(name, description, Problem) per call; fast/slow pairs of one skinny draw share inputs."""
    from precision_matmul_gb300 import synth
    cat = _catalogue()
    shared = {}
    out = []
    for name in workload_names(spec):
        desc, f = cat[name]
        if callable(f):
            p = f()
        else:
            M, data, fast = f
            if (M, data) not in shared:
                shared[(M, data)] = synth.skinny(M=M, data=data)
            p = dataclasses.replace(shared[(M, data)], fast_accum=fast)
        out.append((name, desc, p))
    return out


def config_of(spec: str, probs) -> dict:
    """The `config` object both arms print."""
    return {"workload": spec if spec != "all" else "every metric configuration: " + ", ".join(n for n, _, _ in probs),
            "calls_per_step": len(probs),
            "calls": [{"name": n, "M": p.M, "N": p.N, "K": p.K, "L": p.L} for n, _, p in probs]}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def read_traffic():
    """DRAM bytes per launch from the committed ncu summary, keyed by call
    name, only if it was captured on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "fp8mm_kernel_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("kernel_sources_sha256_16") == kernel_hash():
            return t.get("traffic_bytes_per_launch", {})
    except Exception:
        pass
    return {}


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
    """Time the CPU oracle on a bounded row sample of each problem (batch 0,
    all N); returns (TFLOP/s, threads, description)."""
    import oracle
    threads = os.cpu_count() or 1
    total_flops, total_t, descr = 0.0, 0.0, []
    for name, _, p in probs:
        a, b, sa, sb = p.a.numpy(), p.b.numpy(), p.scale_a.numpy(), p.scale_b.numpy()
        rows = 4
        while True:
            t0 = time.perf_counter()
            oracle.scaled_gemm(a[:1], b[:1], sa, sb, a_fmt=p.a_fmt, b_fmt=p.b_fmt,
                               scale_mode=p.scale_mode, out_dtype=p.out_dtype, rows=(0, rows), nthreads=threads)
            dt = time.perf_counter() - t0
            if dt > 0.2 or rows >= p.M:
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
        descr.append(f"{name}: rows 0..{want} of M={p.M}")
    return total_flops / total_t / 1e12, threads, ("oracle on the first rows of batch 0 of every call (all N, all K), "
                                                   "rate extrapolated by flops: " + "; ".join(descr))


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
        oracle_sample(probs, target_s=1.0)
    sample = ""
    cores = os.cpu_count()
    for _ in range(args.steps):
        v, cores, sample = oracle_sample(probs, target_s=max(2.0, 60.0 / max(1, args.steps)))
        vals.append(v)
    value = statistics.median(vals)
    flops = sum(p.flops for _, _, p in probs)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": flops / (value * 1e12) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(args.workload, probs),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cublas_fp8_peak(dev):
    """torch._scaled_mm (cuBLAS) on a per-tensor E4M3 8192^3 GEMM, bf16 out,
    fast accumulation: best of 10 back-to-back calls (a reference point for
    the FP8 tensor peak, not the roofline denominator)."""
    import torch
    try:
        n = 8192
        a = torch.randn(n, n, device=dev).clamp(-448, 448).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).clamp(-448, 448).to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b.t(), one, one, out_dtype=torch.bfloat16, use_fast_accum=True)
        best = 1e9
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b.t(), one, one, out_dtype=torch.bfloat16, use_fast_accum=True)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3)
        del a, b
        return 2.0 * n ** 3 / best / 1e12
    except Exception as e:  # not fatal: it is context only
        return f"unavailable: {type(e).__name__}: {e}"


def run_ours(args, rank, world, local_rank):
    import torch
    import precision_matmul_gb300 as pm
    from precision_matmul_gb300 import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device(f"cuda:{local_rank}")
    probs = problems(args.workload)
    next_probs = problems("next") if (args.next_rows and args.workload == "all") else []

    def prepare(plist):
        items = []
        dev_inputs = {}
        for name, _, p in plist:
            key = id(p.a)
            if key not in dev_inputs:  # fast/slow calls of one draw share their device operands
                dev_inputs[key] = (p.a.to(dev), p.b.to(dev), p.scale_a.to(dev), p.scale_b.to(dev))
            a, b, sa, sb = dev_inputs[key]
            squeeze = p.L == 1
            if squeeze:
                a, b = a[0], b[0]
            ex = EXTRA.get(name, {})
            kw = {}
            if ex.get("b_major"):  # b stored [.., K, N]: the library copies it K-major first
                b = b.transpose(-1, -2).contiguous().transpose(-1, -2)
            if ex.get("bias"):
                g = torch.Generator().manual_seed(11)
                kw["bias"] = (torch.randn(p.N, generator=g) * 100).to(synth.OUT_TORCH[p.out_dtype]).to(dev)
            if "scale_result" in ex:
                kw["scale_result"] = torch.tensor([ex["scale_result"]], dtype=torch.float32, device=dev)
            shape = (p.M, p.N) if squeeze else (p.L, p.M, p.N)
            c = torch.empty(shape, dtype=synth.OUT_TORCH[p.out_dtype], device=dev)
            amax = torch.empty(1, dtype=torch.float32, device=dev)
            items.append((p, a, b, sa, sb, c, amax, kw))
        return items

    ins = prepare(probs)
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    sink = torch.empty(1, dtype=torch.int64, device=dev)

    def flush_l2():
        # Write 256 MiB (twice the L2), then read it back so that the dirty
        # lines are written back here rather than during the timed GEMM.
        flush.fill_(1)
        torch.sum(flush.view(torch.int64), dim=0, keepdim=True, out=sink)

    stream = torch.cuda.current_stream(dev)

    def call(item):
        p, a, b, sa, sb, c, amax, kw = item
        pm.scaled_mm(a, b, sa, sb, out_dtype=synth.OUT_TORCH[p.out_dtype], use_fast_accum=p.fast_accum,
                     a_fmt=p.a_fmt, b_fmt=p.b_fmt, scale_mode=p.scale_mode, out=c, amax=amax, **kw)

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
    flops = sum(p.flops for _, _, p in probs)
    value = whole_job_tflops(flops, step_s, world)
    err = pm.fp8mm_device_error(local_rank)
    if err:
        raise SystemExit(f"device abort recorded: {err:#x}")

    # ---- the next rows (not part of the metric's step): same timing, own loop
    next_call = []
    if next_probs:
        nxt = prepare(next_probs)
        next_call = [[] for _ in nxt]
        for _ in range(3):
            for it in nxt:
                call(it)
        nev = []
        for _ in range(args.next_steps):
            for i, it in enumerate(nxt):
                flush_l2()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call(it)
                e1.record(stream)
                nev.append((i, e0, e1))
        torch.cuda.synchronize()
        for i, e0, e1 in nev:
            next_call[i].append(e0.elapsed_time(e1) / 1e3)
        del nxt
        if pm.fp8mm_device_error(local_rank):
            raise SystemExit("device abort recorded in the next-row calls")

    # ---- sustained: the dominant call back to back for >= sustain_s under the clock sampler
    call_s = [sum(x) / len(x) for x in per_call]
    dom = max(range(len(probs)), key=lambda i: call_s[i])
    sus_idx = next((i for i, (n, _, _) in enumerate(probs) if n == "c2_llm4096_slow"), dom)
    sustained = None
    if args.sustain_s > 0:
        n_calls = max(10, int(args.sustain_s / max(call_s[sus_idx], 1e-6)))
        for _ in range(5):
            call(ins[sus_idx])
        torch.cuda.synchronize()
        with ClockSampler(local_rank) as sclk:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n_calls):
                call(ins[sus_idx])
            e1.record(stream)
            torch.cuda.synchronize()
        s_s = e0.elapsed_time(e1) / 1e3
        sustained = {"call": probs[sus_idx][0], "calls": n_calls, "seconds": s_s,
                     "tflops": probs[sus_idx][2].flops * n_calls / s_s / 1e12, "clocks": sclk.summary(),
                     "note": "back to back, no L2 flush (the operands stay in L2)"}

    # ---- e2e through the public API: pinned host operands in, C and amax out.
    # As a user of the library would pipeline it: each call's operands are
    # copied in on a copy stream (ahead of the compute), the GEMM runs on the
    # current stream, and C and amax are read back on a third stream.  The
    # fast and slow calls of one skinny draw take the same operands, as they
    # do in the device-timed step, so those are copied in once per step.
    # Every operand set has its own device buffers, so no copy overwrites
    # operands a GEMM may still read; a call's C is rewritten only after its
    # previous read-back has finished.
    group_of, host_in, dev_in, users = [], {}, {}, {}
    host_out = []
    for i, (p, a, b, sa, sb, c, amax, _) in enumerate(ins):
        key = (a.data_ptr(), b.data_ptr(), sa.data_ptr(), sb.data_ptr())
        group_of.append(key)
        users.setdefault(key, []).append(i)
        if key not in host_in:
            host_in[key] = tuple(t.cpu().pin_memory() for t in (a, b, sa, sb))
            dev_in[key] = tuple(torch.empty_like(t) if t.is_contiguous() else
                                torch.empty_like(t.transpose(-1, -2).contiguous()).transpose(-1, -2)
                                for t in (a, b, sa, sb))
        host_out.append((torch.empty(c.shape, dtype=c.dtype).pin_memory(),
                         torch.empty(1, dtype=torch.float32).pin_memory()))
    h2d = sum(sum(t.numel() * t.element_size() for t in x) for x in host_in.values())
    d2h = sum(x[0].numel() * x[0].element_size() + 4 for x in host_out)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n_calls = len(ins)
    comp_done = [None] * n_calls
    out_done = [None] * n_calls

    def e2e_step():
        ready = {}
        for i, (p, _, _, _, _, c, amax, kw) in enumerate(ins):
            key = group_of[i]
            a, b, sa, sb = dev_in[key]
            if key not in ready:
                with torch.cuda.stream(s_in):
                    for j in users[key]:
                        if comp_done[j] is not None:
                            s_in.wait_event(comp_done[j])   # the previous step's GEMMs have read these operands
                    for d, h in zip(dev_in[key], host_in[key]):
                        d.copy_(h, non_blocking=True)
                    ready[key] = torch.cuda.Event()
                    ready[key].record(s_in)
            stream.wait_event(ready[key])
            if out_done[i] is not None:
                stream.wait_event(out_done[i])       # C of the previous step has been read back
            call((p, a, b, sa, sb, c, amax, kw))
            comp_done[i] = torch.cuda.Event()
            comp_done[i].record(stream)
            hc, hm = host_out[i]
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                hc.copy_(c, non_blocking=True)
                hm.copy_(amax, non_blocking=True)
                out_done[i] = torch.cuda.Event()
                out_done[i].record(s_out)

    for _ in range(max(1, min(args.warmup, 3))):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for _ in range(args.steps):
        e2e_step()
    for ev in out_done:
        stream.wait_event(ev)                      # every read-back is inside the timed region
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3 / args.steps, world, dev)
    e2e_value = world * flops / e2e_s / 1e12

    if rank != 0:
        return
    # ---- per-call rooflines and the dominant call's
    hbm, bf16, bf16_sus, peak_src = read_peaks()
    fp8_peak = bf16 * FP8_PER_BF16
    cublas = cublas_fp8_peak(dev) if args.cublas_peak else None
    traffic = read_traffic()
    def plan_of(name, p):
        ex = EXTRA.get(name, {})
        return pm.plan_for((p.M, p.N, p.K, p.L, p.a_fmt, p.b_fmt, p.scale_mode, p.out_dtype,
                            1 if p.fast_accum else 0, 0, 0, 0, local_rank, 0, 0, 0, 1 if ex.get("bias") else 0, 0,
                            1 if ex.get("b_major") else 0))

    def entries(plist, times):
        out = []
        for (name, desc, p), ts in zip(plist, times):
            pl = plan_of(name, p)
            f, by = pl.roofline()
            med = statistics.median(ts)
            # FP4 operands run on the FP4 tensor rate (nominal 13.5 : 2.25 against bf16)
            peak = bf16 * (FP4_PER_BF16 if p.a_fmt == synth.E2M1 else FP8_PER_BF16)
            tensor_bound = f / (peak * 1e12) >= by / (hbm * 1e9)
            tf, gbs = f / med / 1e12, by / med / 1e9
            entry = {"name": name, "what": desc, "us": med * 1e6, "tflops": tf, "gbs": gbs,
                     "bound": "tensor" if tensor_bound else "hbm", "peak": peak if tensor_bound else hbm,
                     "frac": tf / peak if tensor_bound else gbs / hbm,
                     "roofline_us": max(f / (peak * 1e12), by / (hbm * 1e9)) * 1e6,
                     "plan": pl.info(), "kernel_launches": pl.kernel_launches(), "traffic": traffic.get(name)}
            if isinstance(cublas, float) and tensor_bound and p.a_fmt != synth.E2M1:
                entry["frac_of_cublas_fp8"] = tf / cublas
                entry["frac_of_nominal_fp8"] = tf / FP8_NOMINAL_TFLOPS
            out.append(entry)
        return out

    plans = [plan_of(n, p) for n, _, p in probs]
    launches = sum(pl.kernel_launches() for pl in plans)
    per_config = entries(probs, per_call)
    next_rows = entries(next_probs, next_call) if next_probs else None
    d = per_config[dom]
    roof = {"bound": d["bound"], "achieved": d["tflops"] if d["bound"] == "tensor" else d["gbs"],
            "peak": fp8_peak if d["bound"] == "tensor" else hbm,
            "unit": "TFLOP/s" if d["bound"] == "tensor" else "GB/s", "frac": d["frac"], "traffic": d["traffic"],
            "peak_source": (f"{peak_src} bf16 burst {bf16:.1f} TFLOP/s x nominal FP8:BF16 ratio 2"
                            if d["bound"] == "tensor" else f"{peak_src} HBM copy bandwidth"),
            "kernel": f"fp8mm_kernel ({d['name']}: BN={d['plan']['block_n']}, "
                      f"{'CTA pair' if d['plan']['cta_pair'] else 'one CTA'}, "
                      f"{'slow' if d['plan']['slow'] else 'fast'} accumulation)",
            "algorithmic_flops_per_launch": plans[dom].roofline()[0],
            "algorithmic_bytes_per_launch": plans[dom].roofline()[1],
            "us_per_launch": d["us"], "roofline_time_us": d["roofline_us"]}
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, sample = oracle_sample(probs, target_s=args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}
    fmts = sorted({{0: "fp8_e4m3", 1: "fp8_e5m2", 2: "fp4_e2m1"}[p.a_fmt] for _, _, p in probs})
    cfg = config_of(args.workload, probs)
    cfg.update({"l2": "L2 flushed before every timed GEMM: 256 MiB written, then read back (not timed)",
                "parallelism": f"replicas x{world}"})
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "/".join(fmts) + " operands, fp32 accumulation", "data": "synthetic",
            "config": cfg, "per_config": per_config, "roofline": roof,
            "next_rows": next_rows,
            "peaks": {"fp8_tflops_used": fp8_peak, "hbm_gbs_used": hbm, "source": peak_src,
                      "fp8_nominal_dense_tflops": FP8_NOMINAL_TFLOPS, "cublas_fp8_8192cubed_tflops": cublas,
                      "fp8_sustained_from_bf16_tflops": bf16_sus * FP8_PER_BF16},
            "sustained": sustained, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches * args.steps, "clocks": clk.summary(), "wall_s": t_wall,
            "kernel_sources_sha256_16": kernel_hash()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--sustain-s", type=float, default=2.0)
    ap.add_argument("--no-cublas-peak", dest="cublas_peak", action="store_false")
    ap.add_argument("--no-next-rows", dest="next_rows", action="store_false")
    ap.add_argument("--next-steps", type=int, default=10)
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
