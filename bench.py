#!/usr/bin/env python3
"""Throughput of the MXFP8 grouped expert-MLP forward on one GB300 (or N replicas).

One step = one grouped_mlp_fwd call over the whole Mixtral-8x7B-shaped expert layer
(E=8, top-2, T=16384 tokens -> R=32768 routed rows, H=4096, F=14336): activation quantize,
device tile schedule, GroupedLinear 1 with the fused ScaledSwiGLU + MXFP8 requant epilogue, and
GroupedLinear 2 to bf16.  Inputs are synthetic (seeded, shapes of the pages' workload) and
resident in HBM when the timed region starts; weights are quantized once beforehand (the
"quantized init" setting), timed separately.

Printed: one JSON line (rank 0).  `value` = 6*R*H*F / step time in TFLOP/s summed over ranks.
Extra keys: roofline (dominant kernel = GroupedLinear 1), quantize (stand-alone MXFP8 quantize
of a 16384 x 14336 bf16 matrix, row- and column-wise, GB/s against HBM), e2e (same step with
host buffers, copies inside the timed region), cpu_baseline (the oracle on a bounded sample),
clocks, gpu_launches.

--impl reference times the CPU oracle instead (bounded row samples of the same workload).
Multi-GPU (torchrun): every rank runs an independent replica of the step ("replicas only": the
path has no exchange), timing is max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GroupedMLP MXFP8 fwd TFLOP/s & % of MXFP8 peak; quantize GB/s & % of HBM"
WORKLOAD = "mixtral"
QUANT_SHAPE = (16384, 14336)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0          # nominal dense ratio (4.5 vs 2.25 PFLOP/s per GPU)
FP4_OVER_BF16 = 6.0          # nominal dense ratio (13.5 vs 2.25 PFLOP/s per GPU)
KERNEL_SOURCES = ["mxfp8_block_scaled_03_gb300/csrc/grouped_gemm.cu", "mxfp8_block_scaled_03_gb300/csrc/mx_device.cuh",
                  "mxfp8_block_scaled_03_gb300/csrc/quantize.cu"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash() -> str:
    """Hash of the kernel sources' code: comments and blank lines are left out, so that a
    comment-only edit keeps the stored DRAM counters valid."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def load_traffic():
    """Per-launch DRAM bytes of the dominant kernels from the committed ncu summary, or None
    when the kernel sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return {}
    if d.get("kernel_hash") != kernel_hash():
        return {}
    return d


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while active."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons, power = [], [], set(), []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# CPU oracle leg (cpu_baseline and --impl reference)
# ------------------------------------------------------------------------------------------------
class OracleSample:
    """The oracle on `nrows` rows of one expert of the workload (a sub-problem with E=1 holding
    that expert's rows and weights: the per-row arithmetic is identical)."""

    def __init__(self, w, expert: int = 0, nrows: int = 64):
        import numpy as np
        import oracle
        self.oracle = oracle
        off = np.concatenate([[0], np.cumsum(w.split_sizes)])
        n = int(w.split_sizes[expert])
        self.x = np.ascontiguousarray(w.x_sorted[off[expert]:off[expert] + n])
        self.gates = None if w.gates is None else np.ascontiguousarray(w.gates[off[expert]:off[expert] + n])
        F, H = w.F, w.H
        self.w1q, self.w1s = oracle.quantize_rowwise(w.w1[expert * 2 * F:(expert + 1) * 2 * F])
        self.w2q, self.w2s = oracle.quantize_rowwise(w.w2[expert * H:(expert + 1) * H])
        self.split = np.array([n], dtype=np.int32)
        self.nrows = min(nrows, n)
        self.flops_per_row = 6.0 * H * F
        self.threads = oracle.default_threads()
        self._step = 0
        self.n_avail = n
        self.name = w.name

    def run(self) -> float:
        import numpy as np
        start = (self._step * self.nrows) % max(1, self.n_avail - self.nrows + 1)
        rows = np.arange(start, start + self.nrows)
        self._step += 1
        t0 = time.perf_counter()
        self.oracle.grouped_mlp_rows(self.x, self.split, self.gates, self.w1q, self.w1s, self.w2q, self.w2s, rows,
                                     nthreads=self.threads, want_intermediate=False)
        return time.perf_counter() - t0

    def describe(self):
        return (f"{self.nrows} consecutive rows of expert 0 of the {self.name} workload per timed call "
                f"(binary64 GroupedLinear->ScaledSwiGLU->requant->GroupedLinear, {self.flops_per_row:.3g} flop/row); "
                "oracle weight quantization excluded")


def run_reference(args, world, rank):
    from mxfp8_block_scaled_03_gb300 import workloads as W
    if rank != 0:
        return
    w = W.moe_workload(args.workload, seed=0)
    s = OracleSample(w, nrows=args.oracle_rows)
    for _ in range(args.warmup):
        s.run()
    times = [s.run() for _ in range(args.steps)]
    total = sum(times)
    value = s.nrows * s.flops_per_row * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": s.threads, "kind": "oracle",
                         "sample": s.describe()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


WORKLOAD_TEXT = {
    "mixtral": "Mixtral-8x7B-shaped expert MLP layer, router logits N(0,1)+per-expert bias N(0,0.5), top-2 renormalized",
    "llama": "dense Llama-3.1-8B-shaped SwiGLU MLP as one group, gate 1",
    "fine": "fine-grained skewed MoE, Zipf(1.2) expert popularity (3 experts empty), top-8, Dirichlet(1) gates",
    "tiny": "tiny MoE expert MLP, router logits N(0,1), top-2 renormalized",
}


# ------------------------------------------------------------------------------------------------
# GPU leg
# ------------------------------------------------------------------------------------------------
def _events(n):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def gpu_numa_node(local: int):
    """NUMA node of the host memory closest to this GPU (the node of its PCI device), or None."""
    import torch
    pr = torch.cuda.get_device_properties(local)
    ids = [getattr(pr, a, None) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")]
    paths = []
    if None not in ids:
        paths.append(f"/sys/bus/pci/devices/{ids[0]:04x}:{ids[1]:02x}:{ids[2]:02x}.0/numa_node")
    try:
        uuid = str(getattr(pr, "uuid", ""))
        out = subprocess.run(["nvidia-smi", "--query-gpu=uuid,pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            u, bus = [t.strip() for t in line.split(",")]
            if uuid and uuid in u:
                dom, rest = bus.split(":", 1)
                paths.append(f"/sys/bus/pci/devices/{int(dom, 16):04x}:{rest.lower()}/numa_node")
    except Exception:
        pass
    for path in paths:
        try:
            node = int(open(path).read().strip())
            if node >= 0:
                return node
        except Exception:
            continue
    return None


def node_cpus(node: int):
    try:
        text = open(f"/sys/devices/system/node/node{node}/cpulist").read().strip()
    except Exception:
        return set()
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus


def numa_pages(ptr: int):
    """{node: pages} of the mapping of this process that holds address ptr (/proc/self/numa_maps)."""
    try:
        best = None
        for line in open("/proc/self/numa_maps"):
            parts = line.split()
            start = int(parts[0], 16)
            if start <= ptr and (best is None or start > best[0]):
                best = (start, parts)
        if best is None:
            return None
        nodes = {}
        for t in best[1]:
            if t.startswith("N") and "=" in t:
                k, v = t[1:].split("=")
                nodes[int(k)] = int(v)
        return nodes or None
    except Exception:
        return None


def library_mxfp8_gemms(R, H, F, dev, iters=10):
    """Context only: cuBLASLt's MXFP8 GEMM (through torch._scaled_mm) on the dense shapes of the two
    grouped GEMMs (M = routed rows, no expert grouping, bf16 output, no fused epilogue) and on the
    8192^3 square, timed with CUDA events on synthetic E4M3 codes with unit scales.  Nothing of the
    library's path runs here."""
    import torch
    if not hasattr(torch, "float8_e8m0fnu"):
        return {"unavailable": "this torch has no float8_e8m0fnu"}

    def rup(a, b):
        return (a + b - 1) // b * b

    out = {"kind": "cuBLASLt MXFP8 (torch._scaled_mm, block scale 1x32, bf16 out)", "note":
           "dense [M,K]x[K,N] without grouping, routing weight, SwiGLU or requantization"}
    for name, (M, N, K) in (("grouped_linear1_shape", (R, 2 * F, H)), ("grouped_linear2_shape", (R, H, F)),
                            ("square_8192", (8192, 8192, 8192))):
        try:
            g = torch.Generator(device=dev).manual_seed(3)
            a = (torch.randn(M, K, device=dev, generator=g) * 0.5).to(torch.float8_e4m3fn)
            b = (torch.randn(N, K, device=dev, generator=g) * 0.5).to(torch.float8_e4m3fn)
            sa = torch.full((rup(M, 128) * rup(K // 32, 4),), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
            sb = torch.full((rup(N, 128) * rup(K // 32, 4),), 127, dtype=torch.uint8, device=dev).view(torch.float8_e8m0fnu)
            run = lambda: torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
            for _ in range(3):
                run()
            torch.cuda.synchronize()
            e0, e1 = _events(2)
            e0.record()
            for _ in range(iters):
                run()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / iters
            out[name] = {"M": M, "N": N, "K": K, "ms": ms, "tflops": 2 * M * N * K / (ms * 1e-3) / 1e12}
            del a, b, sa, sb
        except Exception as ex:   # the library call is context, never a reason to fail the bench
            out[name] = {"unavailable": repr(ex)[:200]}
    torch.cuda.empty_cache()
    return out


def mma_loop_peak(mx, dev, fmt=0):
    """The library's own back-to-back block-scaled pair-MMA loop (mxfp8_mma_peak): TFLOP/s of the
    tensor pipe with operands resident in shared memory (fmt 0: MXFP8, K = 32 per MMA; fmt 1:
    NVFP4, K = 64 per MMA)."""
    import torch
    ws = torch.zeros(64, dtype=torch.uint8, device=dev)
    iters = 1 << 18
    kmma = 64 if fmt == 1 else 32
    mx.mxfp8_mma_peak(iters // 16, ws, fmt)
    torch.cuda.synchronize()
    best = None
    for _ in range(3):
        e0, e1 = _events(2)
        e0.record()
        n = mx.mxfp8_mma_peak(iters, ws, fmt)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        tf = n * iters * 4 * 2.0 * 256 * 256 * kmma / (ms * 1e-3) / 1e12
        best = tf if best is None else max(best, tf)
    st, bits = mx.mxfp8_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"MMA peak loop error word {bits:#x}")
    kind = "kind::mxf4nvf4.block_scale.scale_vec::4X M=256 N=256 K=64" if fmt == 1 else \
        "kind::mxf8f6f4.block_scale M=256 N=256 K=32"
    return {"tflops": best, "clusters": n, "mma_per_cluster": 4 * iters,
            "kind": f"mxfp8_mma_peak: tcgen05.mma.cta_group::2.{kind}, operands resident in shared memory, "
                    "best of 3 launches"}


def workload_config(w):
    return {"workload": f"{WORKLOAD_TEXT[w.name]}: E={w.E} top-{w.topk} T={w.T} (R={w.R} routed rows) "
                        f"H={w.H} F={w.F}, x~N(0,1), W~N(0,0.02)",
            "R": w.R, "H": w.H, "F": w.F, "E": w.E, "split_sizes": [int(v) for v in w.split_sizes],
            "l2": "no flush: inputs larger than L2 (x 256 MiB, W1+W2 1.3 GiB quantized)",
            "parallelism": "replicas"}


class Forward:
    """Device-resident inputs of one workload and its grouped_mlp_fwd step."""

    def __init__(self, mx, w, dev):
        import numpy as np
        import torch
        self.mx, self.w, self.dev = mx, w, dev
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        self.x = bf(w.x_sorted)
        self.split = torch.from_numpy(w.split_sizes).to(dev)
        self.gates = torch.from_numpy(w.gates).to(dev) if w.gates is not None else None
        w1, w2 = bf(w.w1), bf(w.w2)
        for _ in range(2):
            self.w1q, self.w1s, _, _ = mx.mxfp8_quantize(w1, sf_layout=mx.SF_MMA)
            self.w2q, self.w2s, _, _ = mx.mxfp8_quantize(w2, sf_layout=mx.SF_MMA)
        e0, e1 = _events(2)
        e0.record()
        mx.mxfp8_quantize(w1, sf_layout=mx.SF_MMA, out=[self.w1q, self.w1s, None, None])
        mx.mxfp8_quantize(w2, sf_layout=mx.SF_MMA, out=[self.w2q, self.w2s, None, None])
        e1.record()
        torch.cuda.synchronize()
        self.weight_quant_ms = e0.elapsed_time(e1)
        self.w1_bf16, self.w2_bf16 = w1, w2      # kept for the backward's transposed weights
        R, H, F, E = w.R, w.H, w.F, w.E
        self.ws = torch.empty(mx.grouped_mlp_workspace_size(R, H, F, E), dtype=torch.uint8, device=dev)
        self.y = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
        self.flops = 6.0 * R * H * F

    def step(self, events=None):
        self.mx.grouped_mlp_fwd(self.x, self.split, self.gates, self.w1q, self.w1s, self.w2q, self.w2s, y=self.y,
                                workspace=self.ws, stage_events=events)

    def check(self, when):
        st, bits = self.mx.mxfp8_check_device_error(self.ws)
        if st != 0:
            raise RuntimeError(f"device error word {bits:#x} {when}")

    def time(self, steps, warmup, world=1, clocks=None):
        """Per-step device time (events around K steps) and per-kernel times (events the library
        records between its kernels on the same stream)."""
        import torch
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        self.check("after warm-up")
        stage_ev = [_events(5) for _ in range(steps)]
        for evs in stage_ev:          # torch creates the CUDA event on first record; the library re-records it
            for ev in evs:
                ev.record()
        torch.cuda.synchronize()
        t_start, t_end = _events(2)
        ctx = ClockSampler(clocks) if clocks is not None else None
        if ctx is not None:
            ctx.__enter__()
        barrier(world)
        torch.cuda.synchronize()
        t_start.record()
        for i in range(steps):
            self.step(stage_ev[i])
        t_end.record()
        torch.cuda.synchronize()
        barrier(world)
        if ctx is not None:
            ctx.__exit__(None, None, None)
        self.clocks = ctx.summary() if ctx is not None else None
        step_ms = max_over_ranks(world, t_start.elapsed_time(t_end) / steps)
        names = ["schedule", "quantize_x", "grouped_linear1_swiglu_requant", "grouped_linear2"]
        kern_ms = {n: sum(ev[j].elapsed_time(ev[j + 1]) for ev in stage_ev) / steps for j, n in enumerate(names)}
        self.check("after timed steps")
        return step_ms, kern_ms


def forward_summary(fwd, step_ms, kern_ms, fp8_peak, mma_peak, world=1):
    w = fwd.w
    R, H, F = w.R, w.H, w.F
    g1 = 4.0 * R * H * F / (kern_ms["grouped_linear1_swiglu_requant"] * 1e-3) / 1e12
    g2 = 2.0 * R * H * F / (kern_ms["grouped_linear2"] * 1e-3) / 1e12
    value = world * fwd.flops / (step_ms * 1e-3) / 1e12
    out = {"workload": w.name, "R": R, "H": H, "F": F, "E": w.E, "ms": step_ms, "tflops": value,
           "frac_of_peak": value / world / fp8_peak, "kernel_ms": kern_ms,
           "grouped_linear1": {"tflops": g1, "frac": g1 / fp8_peak},
           "grouped_linear2": {"tflops": g2, "frac": g2 / fp8_peak}}
    if mma_peak:
        out["frac_of_measured_mxfp8_peak"] = value / world / mma_peak
        out["grouped_linear1"]["frac_of_measured_mxfp8_peak"] = g1 / mma_peak
        out["grouped_linear2"]["frac_of_measured_mxfp8_peak"] = g2 / mma_peak
    return out


def quantize_sweep(mx, dev, peaks, steps):
    """Stand-alone MXFP8 quantize of the sweep's three bf16 matrices, row-wise and row + column.
    Inputs that fit in L2 (the two smaller shapes) are timed one launch at a time with L2 flushed
    before each by reading a 512 MiB buffer (a read leaves L2 holding clean lines; a written
    flush buffer would leave about L2's size of dirty lines whose write-back then competes with
    the timed launch's reads); the largest (470 MB) is timed over back-to-back launches, its
    input far above L2."""
    import numpy as np
    import torch
    from mxfp8_block_scaled_03_gb300 import workloads as W
    flush = torch.ones(512 << 20, dtype=torch.uint8, device=dev)
    flush64 = flush.view(torch.int64)
    out = []
    for (M, K) in ((4096, 4096), (8192, 4096), (16384, 14336)):
        x = torch.from_numpy(W.quant_matrix(M, K, seed=0).view(np.int16)).to(dev).view(torch.bfloat16)
        small = M * K * 2 < 128 << 20
        for dirs, col in (("row", False), ("row+col", True)):
            buf = list(mx.mxfp8_quantize(x, rowwise=True, colwise=col))
            for _ in range(3):
                mx.mxfp8_quantize(x, rowwise=True, colwise=col, out=buf)
            torch.cuda.synchronize()
            n = max(10, steps)
            if small:
                tot = 0.0
                for _ in range(n):
                    torch.amax(flush64)
                    e0, e1 = _events(2)
                    e0.record()
                    mx.mxfp8_quantize(x, rowwise=True, colwise=col, out=buf)
                    e1.record()
                    torch.cuda.synchronize()
                    tot += e0.elapsed_time(e1)
                ms = tot / n
            else:
                e0, e1 = _events(2)
                e0.record()
                for _ in range(n):
                    mx.mxfp8_quantize(x, rowwise=True, colwise=col, out=buf)
                e1.record()
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / n
            nbytes = M * K * (2 + (2 if col else 1) * (1 + 1 / 32))
            gbs = nbytes / (ms * 1e-3) / 1e9
            out.append({"shape": [M, K], "directions": dirs, "ms": ms, "achieved": gbs, "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": nbytes,
                        "l2": "flushed (512 MiB read) before each launch" if small else "no flush: input above L2"})
            del buf
        del x
    del flush, flush64
    torch.cuda.empty_cache()
    return out


def nvfp4_forward(mx, fwd, steps, warmup, peaks):
    """The NVFP4 variant of the same forward (nvfp4_grouped_mlp_fwd) on the same resident inputs:
    weights quantized once to NVFP4 (timed apart), the intermediate's encode scale from the largest
    |h| a first call observed (the delayed scaling a training loop would use)."""
    import torch
    w = fwd.w
    R, H, F, E = w.R, w.H, w.F, w.E
    out = {}
    t0, t1 = _events(2)
    w1 = mx.nvfp4_quantize(fwd.w1_bf16, sf_layout=mx.SF_MMA)
    w2 = mx.nvfp4_quantize(fwd.w2_bf16, sf_layout=mx.SF_MMA)
    t0.record()
    mx.nvfp4_quantize(fwd.w1_bf16, sf_layout=mx.SF_MMA, out=w1)
    mx.nvfp4_quantize(fwd.w2_bf16, sf_layout=mx.SF_MMA, out=w2)
    t1.record()
    torch.cuda.synchronize()
    out["weight_quantize_ms"] = t0.elapsed_time(t1)
    ws = torch.empty(mx.nvfp4_grouped_mlp_workspace_size(R, H, F, E), dtype=torch.uint8, device=fwd.dev)
    y = torch.empty((R, H), dtype=torch.bfloat16, device=fwd.dev)
    lay = mx.nvfp4_grouped_mlp_workspace_layout(R, H, F, E)
    mx.nvfp4_grouped_mlp_fwd(fwd.x, fwd.split, fwd.gates, w1, w2, 1.0, y=y, workspace=ws)
    torch.cuda.synchronize()
    h_amax = float(ws[lay[1] + 4:lay[1] + 8].view(torch.float32).item())
    out["h_amax"] = h_amax

    def step(evs=None):
        mx.nvfp4_grouped_mlp_fwd(fwd.x, fwd.split, fwd.gates, w1, w2, h_amax, y=y, workspace=ws, stage_events=evs)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    st, bits = mx.mxfp8_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"device error word {bits:#x} in the NVFP4 forward")
    sev = [_events(5) for _ in range(steps)]
    for evs in sev:
        for ev in evs:
            ev.record()
    torch.cuda.synchronize()
    a0, a1 = _events(2)
    a0.record()
    for i in range(steps):
        step(sev[i])
    a1.record()
    torch.cuda.synchronize()
    ms = a0.elapsed_time(a1) / steps
    names = ["schedule", "amax_quantize_x", "grouped_linear1_swiglu_requant", "grouped_linear2"]
    km = {n: sum(e[j].elapsed_time(e[j + 1]) for e in sev) / steps for j, n in enumerate(names)}
    nominal = peaks["bf16_tflops"] * FP4_OVER_BF16
    g1 = 4.0 * R * H * F / (km["grouped_linear1_swiglu_requant"] * 1e-3) / 1e12
    g2 = 2.0 * R * H * F / (km["grouped_linear2"] * 1e-3) / 1e12
    out.update({"ms": ms, "tflops": fwd.flops / (ms * 1e-3) / 1e12, "kernel_ms": km,
                "grouped_linear1": {"tflops": g1, "frac": g1 / nominal},
                "grouped_linear2": {"tflops": g2, "frac": g2 / nominal},
                "peak": nominal, "peak_source": f"bf16_tflops x {FP4_OVER_BF16:.0f} (nominal dense fp4/bf16 ratio)",
                "dtype": "e2m1 (UE4M3 block scales, fp32 accumulate)"})
    del ws, y, w1, w2
    torch.cuda.empty_cache()
    return out


def run_native(args, world, rank, local):
    import numpy as np
    import torch

    import mxfp8_block_scaled_03_gb300 as mx
    from mxfp8_block_scaled_03_gb300 import build_ext
    from mxfp8_block_scaled_03_gb300 import workloads as W

    build_ext.build()
    mx.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16

    # run on the cores (and first-touch host memory on the NUMA node) next to this GPU
    numa = {"gpu_node": gpu_numa_node(local)}
    if numa["gpu_node"] is not None and hasattr(os, "sched_setaffinity"):
        cpus = node_cpus(numa["gpu_node"]) & set(os.sched_getaffinity(0))
        if cpus:
            os.sched_setaffinity(0, cpus)
            numa["bound_cpus"] = len(cpus)

    w = W.moe_workload(args.workload, seed=0)
    R, H, F, E = w.R, w.H, w.F, w.E
    flops = 6.0 * R * H * F
    fwd = Forward(mx, w, dev)
    x, split, gates, y, ws = fwd.x, fwd.split, fwd.gates, fwd.y, fwd.ws
    w1q, w1s, w2q, w2s = fwd.w1q, fwd.w1s, fwd.w2q, fwd.w2s
    step_ms, kern_ms = fwd.time(args.steps, args.warmup, world, clocks=local)
    clocks = fwd.clocks
    value = world * flops / (step_ms * 1e-3) / 1e12
    traffic = load_traffic()
    g1_flops = 4.0 * R * H * F
    g1_tflops = g1_flops / (kern_ms["grouped_linear1_swiglu_requant"] * 1e-3) / 1e12
    g2_tflops = 2.0 * R * H * F / (kern_ms["grouped_linear2"] * 1e-3) / 1e12
    roofline = {"kernel": "k_grouped_gemm_pair<GEMM_SWIGLU> (GroupedLinear 1 + ScaledSwiGLU + requant)",
                "bound": "tensor", "achieved": g1_tflops, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": g1_tflops / fp8_peak,
                "peak_source": f"{peak_src} bf16_tflops {peaks['bf16_tflops']:.1f} x {FP8_OVER_BF16:.0f} "
                               "(nominal dense fp8/bf16 ratio)",
                "algorithmic_flops_per_launch": g1_flops,
                "traffic": traffic.get("grouped_linear1_bytes_per_launch"),
                "step_frac_of_peak": value / world / fp8_peak,
                "kernel_ms": kern_ms,
                "grouped_linear2": {"achieved": g2_tflops, "frac": g2_tflops / fp8_peak,
                                    "traffic": traffic.get("grouped_linear2_bytes_per_launch")}}

    def measure_backward():
        # ---- backward (training): fwd_train saves [G | U]; the backward runs on a resident dy ----
        bwd = None
        if H % 256 == 0:
            w1b, w2b = fwd.w1_bf16, fwd.w2_bf16
            t0, t1 = _events(2)
            w1t = mx.mxfp8_quantize_colwise_t(w1b)
            w2t = mx.mxfp8_quantize_colwise_t(w2b)
            t0.record()
            mx.mxfp8_quantize_colwise_t(w1b, out=w1t)
            mx.mxfp8_quantize_colwise_t(w2b, out=w2t)
            t1.record()
            torch.cuda.synchronize()
            wt_ms = t0.elapsed_time(t1)
            gen = torch.Generator(device=dev)
            gen.manual_seed(1)
            dy = torch.randn((R, H), generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
            saved = torch.empty(mx.grouped_mlp_saved_bytes(R, H, F, E), dtype=torch.uint8, device=dev)
            bws = torch.empty(mx.grouped_mlp_bwd_workspace_size(R, H, F, E), dtype=torch.uint8, device=dev)
            dx = torch.empty((R, H), dtype=torch.bfloat16, device=dev)
            dgt = torch.empty(R, dtype=torch.float32, device=dev)
            dw1 = torch.empty((E, 2 * F, H), dtype=torch.float32, device=dev)
            dw2 = torch.empty((E, H, F), dtype=torch.float32, device=dev)

            def fwd_train():
                mx.grouped_mlp_fwd_train(x, split, gates, w1q, w1s, w2q, w2s, y=y, saved=saved, workspace=ws)

            def bwd_step(evs=None):
                mx.grouped_mlp_bwd(x, split, gates, saved, w1t[0], w1t[1], w2t[0], w2t[1], dy, dx=dx,
                                   dgates=dgt if gates is not None else False, dw1=dw1, dw2=dw2, workspace=bws,
                                   stage_events=evs)

            fwd_train()
            for _ in range(max(3, args.warmup)):
                bwd_step()
            torch.cuda.synchronize()
            for wsx in (ws, bws):
                st, bits = mx.mxfp8_check_device_error(wsx)
                if st != 0:
                    raise RuntimeError(f"device error word {bits:#x} in the backward")
            nb = max(3, args.steps)
            bev = [_events(7) for _ in range(nb)]
            for evs in bev:
                for ev in evs:
                    ev.record()
            torch.cuda.synchronize()
            f0, f1 = _events(2)
            f0.record()
            for _ in range(nb):
                fwd_train()
            f1.record()
            torch.cuda.synchronize()
            ftrain_ms = f0.elapsed_time(f1) / nb
            b0, b1 = _events(2)
            b0.record()
            for i in range(nb):
                bwd_step(bev[i])
            b1.record()
            torch.cuda.synchronize()
            bwd_ms = b0.elapsed_time(b1) / nb
            names = ["quantize_dy_x", "dgrad2_swiglu_bwd_quant", "dgate_reduce", "dgrad1", "wgrad2", "wgrad1"]
            stage = {n: sum(e[j].elapsed_time(e[j + 1]) for e in bev) / nb for j, n in enumerate(names)}
            bflops = 12.0 * R * H * F
            gemm_tf = {"dgrad2_swiglu_bwd_quant": 2.0 * R * H * F, "dgrad1": 4.0 * R * H * F, "wgrad2": 2.0 * R * H * F,
                       "wgrad1": 4.0 * R * H * F}
            bwd = {"ms": bwd_ms, "tflops": bflops / (bwd_ms * 1e-3) / 1e12, "flops_per_step": bflops,
                   "stage_ms": stage,
                   "gemm_frac_of_peak": {k: v / (stage[k] * 1e-3) / 1e12 / fp8_peak for k, v in gemm_tf.items()},
                   "fwd_train_ms": ftrain_ms,
                   "train_step_tflops": 18.0 * R * H * F / ((bwd_ms + ftrain_ms) * 1e-3) / 1e12,
                   "weight_quantize_transposed_ms": wt_ms,
                   "note": "flops = 12 R H F (dh, dx, dW2, dW1); dy resident, no L2 flush (operands above L2)"}
            del dy, saved, bws, dx, dgt, dw1, dw2, w1t, w2t
            torch.cuda.empty_cache()
        return bwd

    if args.only == "bwd":
        if rank == 0:
            print(json.dumps({"workload": args.workload, "backward": measure_backward()}), flush=True)
        return
    if args.only == "fwd":
        if rank == 0:
            print(json.dumps({"workload": args.workload, "ms_per_step": step_ms, "value": value,
                              "roofline": roofline}), flush=True)
        return
    if args.only == "nvfp4":
        nv = nvfp4_forward(mx, fwd, args.steps, args.warmup, peaks)
        if rank == 0:
            print(json.dumps({"workload": args.workload, "nvfp4": nv}), flush=True)
        return

    # ---- the measured MXFP8 peak: the larger of cuBLASLt at 8192^3 and the library's MMA loop ----
    lib = library_mxfp8_gemms(R, H, F, dev)
    mma = mma_loop_peak(mx, dev)
    cands = {"mma_loop": mma["tflops"]}
    sq = lib.get("square_8192", {}) if isinstance(lib, dict) else {}
    if "tflops" in sq:
        cands["cublaslt_8192"] = sq["tflops"]
    mpeak_src = max(cands, key=cands.get)
    mpeak = cands[mpeak_src]
    peak_measured = {"value": mpeak, "unit": "TFLOP/s", "source": mpeak_src, "candidates": cands, "mma_loop": mma}
    roofline["frac_of_measured_mxfp8_peak"] = g1_tflops / mpeak
    roofline["step_frac_of_measured_mxfp8_peak"] = value / world / mpeak
    roofline["grouped_linear2"]["frac_of_measured_mxfp8_peak"] = g2_tflops / mpeak

    # ---- stand-alone quantize (row + column) of the largest sweep shape: the headline quantize ----
    qx = torch.from_numpy(W.quant_matrix(*QUANT_SHAPE, seed=0).view(np.int16)).to(dev).view(torch.bfloat16)
    M, K = QUANT_SHAPE
    qout = list(mx.mxfp8_quantize(qx, rowwise=True, colwise=True))
    for _ in range(max(3, args.warmup)):
        mx.mxfp8_quantize(qx, rowwise=True, colwise=True, out=qout)
    q0, q1 = _events(2)
    torch.cuda.synchronize()
    qsteps = max(10, args.steps)
    q0.record()
    for _ in range(qsteps):
        mx.mxfp8_quantize(qx, rowwise=True, colwise=True, out=qout)
    q1.record()
    torch.cuda.synchronize()
    q_ms = q0.elapsed_time(q1) / qsteps
    q_bytes = M * K * (2 + 2 * (1 + 1 / 32))
    q_gbs = q_bytes / (q_ms * 1e-3) / 1e9
    quant = {"shape": [M, K], "directions": "row+col", "ms": q_ms, "achieved": q_gbs, "unit": "GB/s",
             "peak": peaks["hbm_gbs"], "frac": q_gbs / peaks["hbm_gbs"], "bound": "hbm",
             "algorithmic_bytes_per_launch": q_bytes, "traffic": traffic.get("quantize_bytes_per_launch"),
             "l2": "no flush: 470 MB input > L2"}
    del qx, qout
    torch.cuda.empty_cache()
    sweep = quantize_sweep(mx, dev, peaks, args.steps)

    # ---- the MoE layer around the forward: permute -> gathered forward -> combine ----
    layer = None
    if w.topk_experts is not None:
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        xt = bf(w.x_tokens)
        exd = torch.from_numpy(w.topk_experts).to(dev)
        gtd = torch.from_numpy(w.topk_gates).to(dev)
        T, k = w.topk_experts.shape
        pws = torch.empty(max(256, mx.moe_permute_workspace_size(T, k, E)), dtype=torch.uint8, device=dev)
        p_split = torch.empty(E, dtype=torch.int32, device=dev)
        p_ros = torch.empty((T, k), dtype=torch.int32, device=dev)
        p_tor = torch.empty(T * k, dtype=torch.int32, device=dev)
        p_gs = torch.empty(T * k, dtype=torch.float32, device=dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        p_out = (p_split, p_ros, p_tor, p_gs)

        def layer_step(evs):
            evs[0].record()
            mx.moe_permute(exd, gtd, E, workspace=pws, out=p_out)
            evs[1].record()
            mx.grouped_mlp_fwd_tokens(xt, p_tor, p_split, p_gs, w1q, w1s, w2q, w2s, y=y, workspace=ws)
            evs[2].record()
            mx.moe_combine(y, p_ros, out=out)
            evs[3].record()

        lev = [_events(4) for _ in range(max(3, args.steps))]
        for _ in range(max(3, args.warmup)):
            layer_step(lev[0])
        torch.cuda.synchronize()
        for evs in lev:
            layer_step(evs)
        torch.cuda.synchronize()
        for wsx in (pws, ws):
            st, bits = mx.mxfp8_check_device_error(wsx)
            if st != 0:
                raise RuntimeError(f"device error word {bits:#x} in the MoE layer")
        part = [sum(e[j].elapsed_time(e[j + 1]) for e in lev) / len(lev) for j in range(3)]
        c_bytes = T * k * H * 2 + T * H * 2 + T * k * 4
        layer = {"tokens": T, "topk": k, "ms": sum(part), "permute_ms": part[0], "fwd_tokens_ms": part[1],
                 "combine_ms": part[2], "tflops": flops / (sum(part) * 1e-3) / 1e12,
                 "combine": {"bound": "hbm", "algorithmic_bytes_per_launch": c_bytes,
                             "achieved": c_bytes / (part[2] * 1e-3) / 1e9, "unit": "GB/s",
                             "frac": c_bytes / (part[2] * 1e-3) / 1e9 / peaks["hbm_gbs"]},
                 "l2": "no flush: per-launch inputs above L2 except the permute's 128 KB of ids"}
        del xt, out

    bwd = measure_backward()

    # ---- the NVFP4 variant of the same forward ----
    nv = None
    if args.only == "all" and H % 256 == 0:
        nv = nvfp4_forward(mx, fwd, max(args.steps, 10), max(3, args.warmup), peaks)
        nv_mma = mma_loop_peak(mx, dev, fmt=1)
        nv["mma_loop_peak"] = nv_mma
        nv["frac_of_measured_nvfp4_peak"] = nv["tflops"] / nv_mma["tflops"]
        for k in ("grouped_linear1", "grouped_linear2"):
            nv[k]["frac_of_measured_nvfp4_peak"] = nv[k]["tflops"] / nv_mma["tflops"]

    # ---- the other configurations of the sweep: forward of each, per kernel ----
    configs = {}
    if args.workload == "mixtral" and args.only == "all" and not args.no_configs:
        for name in ("llama", "fine", "tiny"):
            wo = W.moe_workload(name, seed=0)
            f2 = Forward(mx, wo, dev)
            n = max(args.steps, 20)
            ms2, km2 = f2.time(n, max(3, args.warmup))
            configs[name] = forward_summary(f2, ms2, km2, fp8_peak, mpeak)
            configs[name]["steps"] = n
            if name == "tiny":
                configs[name]["note"] = "latency-bound (0.4 GFLOP): ms is the per-call device time"
            del f2
            torch.cuda.empty_cache()

    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs from pinned host memory and its output back.  Steps are
    # pipelined over three streams with double-buffered device x / y: the host->device copy of
    # step i+1 and the device->host copy of step i-1 run while step i computes.  The pinned
    # buffers are allocated (and first touched) by this process while it runs on the cores of
    # the GPU's NUMA node.
    xh = torch.from_numpy(np.ascontiguousarray(w.x_sorted).view(np.int16)).view(torch.bfloat16).pin_memory()
    sh = torch.from_numpy(w.split_sizes).pin_memory()
    gh = torch.from_numpy(w.gates).pin_memory() if w.gates is not None else None
    yh = torch.empty((R, H), dtype=torch.bfloat16).pin_memory()
    yh.zero_()
    numa["x_host_pages"] = numa_pages(xh.data_ptr())
    numa["y_host_pages"] = numa_pages(yh.data_ptr())
    xd = [torch.empty_like(x) for _ in range(2)]
    sd = [torch.empty_like(split) for _ in range(2)]
    gd = [torch.empty_like(gates) if gates is not None else None for _ in range(2)]
    yd = [torch.empty_like(y) for _ in range(2)]
    s_comp = torch.cuda.current_stream()
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()

    # each copy direction alone (same buffers, same streams)
    def copy_gbs(fn, nbytes, stream):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = _events(2)
        e0.record(stream)
        for _ in range(5):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 5
        return {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9}

    def h2d_only():
        with torch.cuda.stream(s_h2d):
            xd[0].copy_(xh, non_blocking=True)

    def d2h_only():
        with torch.cuda.stream(s_d2h):
            yh.copy_(yd[0], non_blocking=True)

    copies = {"h2d_x": copy_gbs(h2d_only, xh.numel() * 2, s_h2d), "d2h_y": copy_gbs(d2h_only, yh.numel() * 2, s_d2h)}

    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("h2d", "comp", "d2h")}
    for k in ev:
        for e in ev[k]:
            e.record(s_comp)

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_h2d):
            s_h2d.wait_event(ev["comp"][b])            # step i-2 finished reading xd[b]
            xd[b].copy_(xh, non_blocking=True)
            sd[b].copy_(sh, non_blocking=True)
            if gd[b] is not None:
                gd[b].copy_(gh, non_blocking=True)
            ev["h2d"][b].record(s_h2d)
        s_comp.wait_event(ev["h2d"][b])
        s_comp.wait_event(ev["d2h"][b])                # step i-2's result has left yd[b]
        mx.grouped_mlp_fwd(xd[b], sd[b], gd[b], w1q, w1s, w2q, w2s, y=yd[b], workspace=ws, stream=s_comp)
        ev["comp"][b].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev["comp"][b])
            yh.copy_(yd[b], non_blocking=True)
            ev["d2h"][b].record(s_d2h)

    for i in range(max(5, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    a0, a1 = _events(2)
    a0.record(s_comp)
    for i in range(args.steps):
        e2e_step(i)
    s_comp.wait_stream(s_d2h)
    a1.record(s_comp)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, a0.elapsed_time(a1) / args.steps)
    barrier(world)
    h2d = xh.numel() * 2 + sh.numel() * 4 + (gh.numel() * 4 if gh is not None else 0)
    d2h = yh.numel() * 2
    bound_ms = max(step_ms, copies["h2d_x"]["ms"], copies["d2h_y"]["ms"])
    e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "copy_alone": copies, "numa": numa,
           "expected_ms": bound_ms, "ratio_to_expected": e2e_ms / bound_ms,
           "path": "pinned host x/split_sizes/gates -> device, grouped_mlp_fwd, y -> pinned host; "
                   "three streams, copies of neighbouring steps overlap the forward; "
                   "expected_ms = max(device step, x copy alone, y copy alone)"}

    # ---- CPU oracle baseline on a bounded sample (rank 0 only, N=1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if hasattr(os, "sched_setaffinity") and "bound_cpus" in numa:
            os.sched_setaffinity(0, range(os.cpu_count() or 1))   # the oracle uses every host core
        # calibrate on a short call, then time one call sized to about --cpu-seconds
        s = OracleSample(w, nrows=args.oracle_rows)
        t = s.run()
        s.nrows = max(1, min(s.n_avail, int(s.nrows * args.cpu_seconds / max(t, 1e-3))))
        t = s.run()
        cpu = {"value": s.nrows * s.flops_per_row / t / 1e12, "unit": "TFLOP/s", "cores": s.threads,
               "kind": "oracle", "sample": s.describe(), "seconds": t}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)", "data": "synthetic",
            "config": workload_config(w), "roofline": roofline, "peak_mxfp8_measured": peak_measured,
            "quantize": quant, "quantize_sweep": sweep, "configs": configs, "nvfp4": nv, "moe_layer": layer,
            "backward": bwd,
            "e2e": e2e, "library_context": lib,
            "cpu_baseline": cpu, "clocks": clocks, "gpu_launches": 4 * args.steps,
            "weight_quantize_ms": fwd.weight_quant_ms, "peaks": {"source": peak_src, **peaks},
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--oracle-rows", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the forward of the other workloads")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="length of the timed oracle call behind cpu_baseline")
    ap.add_argument("--workload", choices=["mixtral", "llama", "fine", "tiny"], default=WORKLOAD,
                    help="workload of the timed step (the headline line uses mixtral)")
    ap.add_argument("--only", choices=["all", "fwd", "bwd", "nvfp4"], default="all",
                    help="fwd / bwd / nvfp4: time the MXFP8 forward (after it: the backward, or the NVFP4 "
                         "forward) only and print a short line (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_native(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
