"""Benchmark of the block-scaled GEMM hot path on GB300.

Default workload (one "step"): the dense MXFP8 NT GEMMs
    (M,N,K) = (4096,14336,4096), (4096,4096,14336), (8192,8192,8192)  E4M3 x E4M3
    (M,N,K) = (8192,8192,8192)                                        E4M3 x E5M2
each one pass of the path: scale relayout of sA and sB, then the tcgen05 GEMM.
Inputs are seeded N(0,1) values quantised per 32-wide K block (E8M0 scale
2^(floor(log2 amax) - emax)), resident in HBM before timing.  L2 is flushed (256
MiB write) before every GEMM, outside the timed events; a 256 MiB read follows the write,
so the flush's dirty lines are written back before the GEMM starts rather than during it.

Other workloads (``--workload``): mxfp4_dense (8192^3 and 1024x14336x4096),
grouped_fp8 (G=8, totM 128/1024/16384 x three (N,K)), grouped_bf16 (the same shapes
in BF16 without scales), linear_triple (fwd/dgrad/
wgrad of X[8192,4096], W[14336,4096], dY[8192,14336]), mxfp8_256 (256^3),
mxfp8_bias_gelu (the default GEMMs with a fused bias + GELU output stage), and
quantize (the quantisers that make the operands, in GB/s against HBM bandwidth).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead
(on a bounded row sample of the same workload, on the host cores).  Multi-GPU
runs are independent replicas (no collective on the data path).
"""
from __future__ import annotations

import argparse
import atexit
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MX/FP8 GEMM TFLOPS (2MNK/s) and % of GB300 block-scaled tensor peak"
FALLBACK_BF16_TFLOPS = 1900.0        # used only when MEASURED_PEAKS.json is absent
NOMINAL_RATIO = {"fp8": 4.5 / 2.25, "fp4": 13.5 / 2.25, "bf16": 1.0}


# ----------------------------------------------------------------------------- workloads
def workload_spec(name: str):
    """List of GEMM descriptions for one step."""
    if name == "mxfp8_dense":
        return [dict(kind="dense", M=4096, N=14336, K=4096, layout="NT", a="e4m3", b="e4m3", key=(2, 10)),
                dict(kind="dense", M=4096, N=4096, K=14336, layout="NT", a="e4m3", b="e4m3", key=(2, 11)),
                dict(kind="dense", M=8192, N=8192, K=8192, layout="NT", a="e4m3", b="e4m3", key=(2, 12)),
                dict(kind="dense", M=8192, N=8192, K=8192, layout="NT", a="e4m3", b="e5m2", key=(2, 13))]
    if name == "mxfp8_bias_gelu":
        out = workload_spec("mxfp8_dense")
        for g in out:
            g.update(act="gelu", bias=True)
        return out
    if name == "mxfp8_256":
        return [dict(kind="dense", M=256, N=256, K=256, layout="NT", a="e4m3", b="e4m3", key=(1, 0))]
    if name == "mxfp4_dense":
        return [dict(kind="dense", M=8192, N=8192, K=8192, layout="NT", a="e2m1", b="e2m1", key=(3, 10)),
                dict(kind="dense", M=1024, N=14336, K=4096, layout="NT", a="e2m1", b="e2m1", key=(3, 11))]
    if name == "linear_triple":
        return [dict(kind="triple", part=p, key=(5, 0)) for p in ("fwd", "dgrad", "wgrad")]
    if name == "grouped_fp8":
        out = []
        for i, (t, n, k) in enumerate((t, n, k) for t in (128, 1024, 16384)
                                      for (n, k) in ((2048, 7168), (7168, 2304), (16384, 6656))):
            out.append(dict(kind="grouped", T=t, N=n, K=k, case=i))
        return out
    if name == "grouped_fp8_packed":
        out = workload_spec("grouped_fp8")
        for g in out:
            g["packed"] = True
        return out
    if name == "grouped_bf16":
        out = workload_spec("grouped_fp8")
        for g in out:
            g["kind"] = "grouped_bf16"
        return out
    raise SystemExit(f"unknown workload {name}")


WORKLOAD_TEXT = {
    "mxfp8_dense": "MXFP8 dense NT: (4096,14336,4096),(4096,4096,14336),(8192,8192,8192) E4M3xE4M3 "
                   "+ (8192,8192,8192) E4M3xE5M2; E8M0 per 32 along K; BF16 out",
    "mxfp8_bias_gelu": "the mxfp8_dense GEMMs with the fused output stage: D = GELU(acc + bias[n]) "
                       "(erf form), BF16 bias [N] from seeded N(0,1)",
    "mxfp8_256": "MXFP8 NT 256^3 E4M3xE4M3",
    "mxfp4_dense": "MXFP4 dense NT: 8192^3 and (1024,14336,4096), packed E2M1, E8M0 per 32",
    "linear_triple": "MXFP8 Linear triple: fwd NT (8192,14336,4096), dgrad NN (8192,4096,14336), "
                     "wgrad TN (14336,4096,8192)",
    "grouped_fp8": "grouped groupwise FP8, G=8, totM in {128,1024,16384} x (N,K) in "
                   "{(2048,7168),(7168,2304),(16384,6656)}; seeded uneven m_sizes with 2 empty groups",
    "grouped_fp8_packed": "the grouped_fp8 GEMMs on weights packed once outside the timed region "
                          "(grouped_fp8_pack_weights: each 128x128 weight tile one contiguous "
                          "block), as the pages' preshuffled grouped op packs at load time",
    "grouped_bf16": "grouped BF16 (no scales), the grouped_fp8 shapes: G=8, totM in "
                    "{128,1024,16384} x (N,K) in {(2048,7168),(7168,2304),(16384,6656)}; seeded "
                    "uneven m_sizes with 2 empty groups; FP32 accumulation, BF16 out",
}


def describe(g) -> str:
    if g["kind"].startswith("grouped"):
        return f'{g["kind"]} G=8 totM={g["T"]} N={g["N"]} K={g["K"]}'
    return f'{g["M"]}x{g["N"]}x{g["K"]} {g.get("layout", "")} {g.get("a", "")}x{g.get("b", "")}'


def flops_of(g) -> float:
    if g["kind"].startswith("grouped"):
        return 2.0 * g["T"] * g["N"] * g["K"]
    return 2.0 * g["M"] * g["N"] * g["K"]


def grouped_bytes(g, m_sizes) -> float:
    """Algorithmic HBM bytes of one grouped GEMM: W and its scales of the non-empty
    groups, X and its scales, D, m_sizes."""
    T, N, K = g["T"], g["N"], g["K"]
    live = int(sum(1 for m in m_sizes if m > 0))
    if g["kind"] == "grouped_bf16":      # BF16 X and W, no scales
        return live * N * K * 2 + T * K * 2 + 2 * T * N + 8 * len(m_sizes)
    return (live * (N * K + 4 * N * K / 128 ** 2) + T * K + 4 * T * K / 128 + 2 * T * N
            + 8 * len(m_sizes))


def make_inputs(g):
    """Host numpy operands for one GEMM description."""
    import synthetic
    if g["kind"] == "dense":
        c = synthetic.mx_operands(g["key"], g["M"], g["N"], g["K"], g["layout"], g["a"], g["b"])
        if g.get("bias"):
            import torch
            c["bias"] = torch.from_numpy(synthetic.normal((*g["key"], 9), (g["N"],))).to(
                torch.bfloat16).float().numpy()
        return c
    if g["kind"] == "triple":
        global _TRIPLE
        if "_TRIPLE" not in globals() or _TRIPLE is None:
            _TRIPLE = synthetic.linear_triple(g["key"])
        c = _TRIPLE[g["part"]]
        g.update(M=c["M"], N=c["N"], K=c["K"])
        return c
    ms = synthetic.gen_m_sizes(g["T"], g["case"])
    if g["kind"] == "grouped_bf16":
        return synthetic.grouped_bf16_operands((5, g["case"]), ms, g["N"], g["K"])
    return synthetic.grouped_operands((4, g["case"]), ms, g["N"], g["K"])


_TRIPLE = None


# ----------------------------------------------------------------------------- helpers
class L2Flush:
    """Empties L2 of the step's inputs between timed GEMMs: a 256 MiB write (twice the
    129 MB L2), then a 256 MiB read, which writes the first buffer's dirty lines back to
    DRAM before the GEMM starts instead of during it, and leaves only clean lines behind."""

    def __init__(self, torch, dev):
        self.w = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 * 1024 * 1024, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.max()

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("hbm_gbs", 6800.0)), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 6800.0, "fallback"


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every 50 ms.  Started before the
    warm-up (nvidia-smi's start-up can stall CUDA calls of this process for tens of ms, so
    it must not fall inside the timed region); only samples that arrive inside the timed
    window set by window() are summarised."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []          # (arrival time, line)
        self.t0 = self.t1 = None

    def start(self, settle_s: float = 5.0):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            deadline = time.perf_counter() + settle_s
            while not self.lines and time.perf_counter() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        if self.proc:
            atexit.register(self.stop)   # also on an error before the timed region ends
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def window(self, t0: float, t1: float):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc and self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def __enter__(self):
        return self.start()

    def __exit__(self, *exc):
        self.stop()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        if self.t0 is not None:
            # a sample arrives up to one period after it was taken
            inside = [(t, ln) for t, ln in lines if self.t0 <= t <= self.t1 + 0.06]
            lines = inside if inside else lines
        for _, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws):
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("gloo")
        return dist
    return None


def reduce_max(values, dist):
    """Element-wise max over ranks (gloo all-reduce on CPU); identity for one process."""
    if dist is None:
        return list(values)
    import torch
    v = torch.tensor(list(values), dtype=torch.float64)
    dist.all_reduce(v, op=dist.ReduceOp.MAX)
    return v.tolist()


# The sources each workload's dominant kernel is built from (the traffic record is
# valid only while they are unchanged).
KERNEL_SOURCES = {
    "grouped_fp8": ("grouped_gemm.cu", "grouped_sched.cuh", "ptx.cuh", "internal.h"),
    "grouped_fp8_packed": ("grouped_gemm.cu", "grouped_sched.cuh", "ptx.cuh", "internal.h"),
    "grouped_bf16": ("grouped_bf16.cu", "grouped_sched.cuh", "ptx.cuh", "internal.h"),
    "quantize": ("quantize.cu", "ptx.cuh", "internal.h"),
    "dense": ("mx_gemm_2sm.cu", "mx_gemm.cu", "epilogue.cuh", "store_stage.cuh", "stream_k.cuh",
              "ptx.cuh", "internal.h"),
}


def _code_only(text: str) -> str:
    """C++ source without its comments (a record stays valid across comment edits)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (line.split("//", 1)[0].rstrip() for line in text.splitlines())
    return "\n".join(line for line in lines if line)


def kernel_source_hash(workload: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_scaled_precision_mma_gb300", "csrc")
    for f in KERNEL_SOURCES[workload if workload in KERNEL_SOURCES else "dense"]:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary, if
    it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    try:
        kv = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_sources_sha256_16") != kernel_source_hash(workload):
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import block_scaled_precision_mma_gb300 as bs

    ws, rank, local = dist_env()
    dist = init_dist(ws)
    torch.cuda.set_device(local)
    bs.build()
    bs.load()
    bs.set_dense_variant(args.dense_variant)
    bs.set_grouped_tile_width(args.grouped_width)
    bs.set_grouped_variant(args.grouped_variant)
    dev = torch.device("cuda", local)
    spec = workload_spec(args.workload)
    if args.gemm is not None:
        spec = [spec[args.gemm]]    # one GEMM of the step (profiling a single shape)

    gemms = []
    for g in spec:
        c = make_inputs(g)
        if g["kind"] == "grouped_bf16":
            def bf16(a):
                return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
            t = {"X": bf16(c["X"]).to(dev), "W": bf16(c["W"]).to(dev),
                 "m_sizes": torch.from_numpy(c["m_sizes"]).to(dev)}
            t["D"] = torch.empty((g["T"], g["N"]), dtype=torch.bfloat16, device=dev)
            host = {"X": bf16(c["X"]).pin_memory(), "W": bf16(c["W"]).pin_memory(),
                    "m_sizes": torch.from_numpy(c["m_sizes"]).pin_memory()}
        elif g["kind"] == "grouped":
            t = {k: torch.from_numpy(np.ascontiguousarray(c[k])).to(dev)
                 for k in ("X", "sX", "W", "sW", "m_sizes")}
            t["D"] = torch.empty((g["T"], g["N"]), dtype=torch.bfloat16, device=dev)
            host = {k: torch.from_numpy(np.ascontiguousarray(c[k])).pin_memory()
                    for k in ("X", "sX", "W", "sW", "m_sizes")}
            if g.get("packed"):
                # weights packed once, as at load time; the host keeps the packed copy
                t["W"] = bs.grouped_fp8_pack_weights(t["W"])
                torch.cuda.synchronize()
                host["W"] = t["W"].cpu().pin_memory()
        else:
            t = {k: torch.from_numpy(np.ascontiguousarray(c[k])).to(dev) for k in ("A", "sA", "B", "sB")}
            t["D"] = torch.empty((g["M"], g["N"]), dtype=torch.bfloat16, device=dev)
            t["bias"] = (torch.from_numpy(c["bias"]).to(torch.bfloat16).to(dev)
                         if "bias" in c else None)
            t["tA"] = torch.empty(bs.mx_scale_tiled_bytes(g["M"], g["K"] // 32, "A"), dtype=torch.uint8,
                                  device=dev)
            t["tB"] = torch.empty(bs.mx_scale_tiled_bytes(g["N"], g["K"] // 32, "B"), dtype=torch.uint8,
                                  device=dev)
            host = {k: torch.from_numpy(np.ascontiguousarray(c[k])).pin_memory()
                    for k in ("A", "sA", "B", "sB")}
            g.setdefault("layout", c["layout"])
            g.setdefault("a", c["a_fmt"])
            g.setdefault("b", c["b_fmt"])
        host["D"] = torch.empty(t["D"].shape, dtype=torch.bfloat16).pin_memory()
        gemms.append((g, t, host))
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()
    step_flops = sum(flops_of(g) for g, _, _ in gemms)

    def one_gemm(g, t, ev):
        """Relayout (a2) + GEMM (a3-a6); events: [start, after relayout, end]."""
        ev[0].record(stream)
        if g["kind"] == "grouped_bf16":
            ev[1].record(stream)
            bs.grouped_bf16_gemm(t["X"], t["W"], t["m_sizes"], out=t["D"])
        elif g["kind"] == "grouped":
            ev[1].record(stream)
            bs.grouped_fp8_gemm(t["X"], t["sX"], t["W"], t["sW"], t["m_sizes"], out=t["D"],
                                    packed=g.get("packed", False))
        else:
            bs.mx_scale_relayout(t["sA"], "A", out=t["tA"])
            bs.mx_scale_relayout(t["sB"], "B", out=t["tB"])
            ev[1].record(stream)
            bs.mx_gemm_tiled(t["A"], t["tA"], t["B"], t["tB"], g["layout"], g["a"], g["b"],
                             out=t["D"], M=g["M"], N=g["N"], K=g["K"], bias=t.get("bias"),
                             act=g.get("act", "none"))
        ev[2].record(stream)

    def step(events):
        for (g, t, _), ev in zip(gemms, events):
            flush()
            one_gemm(g, t, ev)

    mk = lambda: [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in gemms]
    clk = ClockSampler(local).start()
    for _ in range(args.warmup):
        step(mk())
    torch.cuda.synchronize()
    if bs.device_status() != 0:
        raise SystemExit("device status error during warm-up")
    all_events = [mk() for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    n_launch0 = bs.launch_count()
    try:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            step(all_events[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    finally:
        clk.stop()
    clk.window(wall0, wall0 + wall)
    n_launch = bs.launch_count() - n_launch0
    st = bs.device_status()
    if st != 0:
        raise SystemExit(f"device status {bs.status_string(st)}")
    total_ms = sum(ev[0].elapsed_time(ev[2]) for evs in all_events for ev in evs)
    gemm_ms = sum(ev[1].elapsed_time(ev[2]) for evs in all_events for ev in evs)
    per_gemm_ms = [sum(evs[j][1].elapsed_time(evs[j][2]) for evs in all_events) / args.steps
                   for j in range(len(gemms))]

    # ------------------------------------------------------------- end to end (host buffers)
    e2e_events = []
    h2d = sum(sum(v.numel() * v.element_size() for k, v in h.items() if k != "D") for _, _, h in gemms)
    d2h = sum(h["D"].numel() * h["D"].element_size() for _, _, h in gemms)
    e2e_steps = max(3, min(args.steps, 20))

    # Every GEMM's inputs go host->device on one copy stream while the previous GEMM
    # computes, and its result goes device->host on a second copy stream while the next
    # one computes; events order each reuse of a device buffer across steps.
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in gemms]
    comp_done = [torch.cuda.Event() for _ in gemms]
    d2h_done = [torch.cuda.Event() for _ in gemms]
    recorded = [False] * len(gemms)

    def e2e_step():
        for i, (g, t, h) in enumerate(gemms):
            with torch.cuda.stream(h2d_stream):
                if recorded[i]:
                    h2d_stream.wait_event(comp_done[i])     # the last step's GEMM i read its inputs
                keys = {"grouped": ("X", "sX", "W", "sW", "m_sizes"), "grouped_bf16": ("X", "W", "m_sizes")
                        }.get(g["kind"], ("A", "sA", "B", "sB"))
                for k in keys:
                    t[k].copy_(h[k], non_blocking=True)
                h2d_done[i].record(h2d_stream)
            stream.wait_event(h2d_done[i])
            if recorded[i]:
                stream.wait_event(d2h_done[i])              # the last step's result i is on the host
            if g["kind"] == "grouped_bf16":
                bs.grouped_bf16_gemm(t["X"], t["W"], t["m_sizes"], out=t["D"])
            elif g["kind"] == "grouped":
                bs.grouped_fp8_gemm(t["X"], t["sX"], t["W"], t["sW"], t["m_sizes"], out=t["D"],
                                    packed=g.get("packed", False))
            else:
                bs.mx_gemm(t["A"], t["sA"], t["B"], t["sB"], g["layout"], g["a"], g["b"],
                           out=t["D"], M=g["M"], N=g["N"], K=g["K"], bias=t.get("bias"),
                           act=g.get("act", "none"))
            comp_done[i].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(comp_done[i])
                h["D"].copy_(t["D"], non_blocking=True)
                d2h_done[i].record(d2h_stream)
            recorded[i] = True

    if args.no_e2e:
        e2e_steps = 0
    else:
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    e0.record(stream)
    h2d_stream.wait_stream(stream)      # no copy of the timed steps starts before e0
    for _ in range(e2e_steps):
        e2e_step()
    stream.wait_stream(d2h_stream)      # e1 follows the last result's arrival on the host
    stream.wait_stream(h2d_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps if e2e_steps else float("nan")

    ms_per_step, gemm_step_ms, e2e_ms = reduce_max(
        [total_ms / args.steps, gemm_ms / args.steps, e2e_ms], dist)
    if rank != 0:
        return

    bf16_peak, _, peak_src = measured_peaks()
    is_fp4 = args.workload == "mxfp4_dense"
    is_bf16 = args.workload == "grouped_bf16"
    kind = "fp4" if is_fp4 else "bf16" if is_bf16 else "fp8"
    peak = bf16_peak * NOMINAL_RATIO[kind]
    # the dominant launch: the GEMM of the step with the most flops
    dom = max(range(len(gemms)), key=lambda j: flops_of(gemms[j][0]))
    dom_g = gemms[dom][0]
    achieved = flops_of(dom_g) / (per_gemm_ms[dom] * 1e-3) / 1e12
    step_achieved = step_flops / (gemm_step_ms * 1e-3) / 1e12
    value = ws * step_flops / (ms_per_step * 1e-3) / 1e12
    if args.workload.startswith("grouped_fp8"):
        kernel = "grouped_fp8_kernel"
    elif is_bf16:
        kernel = "grouped_bf16_kernel"
    else:
        kernel = "mx_gemm_2sm_kernel" if args.dense_variant in (0, 3) else "mx_gemm_kernel"
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOPS",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"fp4": "mxfp4(e2m1)+e8m0->f32acc", "bf16": "bf16->f32acc",
                  "fp8": "mxfp8(e4m3/e5m2)+e8m0->f32acc"}[kind],
        "data": "synthetic (seeded N(0,1) truncated to BF16)" if is_bf16
                else "synthetic (seeded N(0,1), MX-quantised)",
        "config": {"workload": args.workload + ": " + WORKLOAD_TEXT[args.workload]
                   + ("" if args.gemm is None else f" -- only GEMM {args.gemm}: {describe(spec[0])}"),
                   "l2": "flushed before every GEMM by a 256 MiB write, then a 256 MiB read (the "
                         "write's dirty lines leave L2 before the GEMM), outside the timed events",
                   "parallelism": f"replicas x{ws}",
                   "dense_variant": args.dense_variant,
                   "grouped_width": args.grouped_width,
                   "grouped_variant": args.grouped_variant,
                   "per_gemm_kernel_ms": [round(x, 4) for x in per_gemm_ms]},
        "roofline": {"bound": "tensor", "kernel": kernel,
                     "launch": describe(dom_g),
                     "achieved": round(achieved, 1),
                     "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_src} bf16 dense, burst" if is_bf16 else
                                    f"{peak_src} bf16 dense x nominal {kind}/bf16 ratio, burst",
                     "traffic": recorded_traffic(args.workload),
                     "all_gemm_kernels_achieved": round(step_achieved, 1)},
        "e2e": None if args.no_e2e else {
            "value": round(ws * step_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOPS",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "api": "mx_gemm / grouped_fp8_gemm / grouped_bf16_gemm with host->device copies of every input "
                   "and device->host copy of D inside the timed region; the copies run on two "
                   "copy streams, overlapping the neighbouring GEMMs' compute"},
        "gpu_launches": int(n_launch),
        "clocks": clk.summary(),
        "wall_s_timed": round(wall, 3),
    }
    if args.workload.startswith("grouped"):
        # each shape against its own bound: compute at the FP8 peak or its algorithmic
        # bytes at the measured HBM copy bandwidth, whichever takes longer
        _, hbm_peak, _ = measured_peaks()
        shapes = []
        for (g, t, _), ms_ in zip(gemms, per_gemm_ms):
            msz = t["m_sizes"].cpu().numpy()
            b = grouped_bytes(g, msz)
            t_hbm = b / (hbm_peak * 1e9)
            t_mma = flops_of(g) / (peak * 1e12)
            bound = "hbm" if t_hbm >= t_mma else "tensor"
            shapes.append({"launch": describe(g), "ms": round(ms_, 4), "bound": bound,
                           "achieved": round(b / (ms_ * 1e-3) / 1e9, 1) if bound == "hbm"
                           else round(flops_of(g) / (ms_ * 1e-3) / 1e12, 1),
                           "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                           "frac": round(max(t_hbm, t_mma) / (ms_ * 1e-3), 4)})
        line["roofline"]["per_shape"] = shapes
        line["roofline"]["hbm_peak_gbs"] = hbm_peak
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- quantisers
QUANT_METRIC = "quantiser GB/s (algorithmic bytes read + written per second) and % of measured HBM copy bandwidth"
QUANT_TEXT = ("quantisers on BF16 inputs: MX E4M3 rowwise and columnwise of X[8192,8192] (the Linear "
              "forward and wgrad operands), groupwise E4M3 of X[16384,7168] with G=8 seeded m_sizes "
              "(1x128 FP32 scales, per-group block layout), blockwise E4M3 of W[8,2048,7168] "
              "(128x128 FP32 scales)")


def quant_ops():
    """The quantiser calls of one step: (name, input shape, seed, kind)."""
    return [("mx_rows_e4m3", (8192, 8192), 0, "rows"), ("mx_cols_e4m3", (8192, 8192), 0, "cols"),
            ("group_x_e4m3", (16384, 7168), 1, "group"), ("block_w_e4m3", (8, 2048, 7168), 2, "block")]


def quant_bytes(kind, shape, in_bytes=2):
    n = int(np.prod(shape))
    if kind in ("rows", "cols"):
        return n * in_bytes + n + n // 32
    if kind == "group":
        return n * in_bytes + n + (n // 128) * 4
    return n * in_bytes + n + (n // (128 * 128)) * 4


def quant_input(shape, seed):
    import synthetic
    return synthetic.normal((6, seed), shape)


def quant_call(bs, kind, x, out, m_sizes, stream=None):
    if kind == "rows":
        bs.mx_quantize(x, "e4m3", codes=out[0], scales=out[1], stream=stream)
    elif kind == "cols":
        bs.mx_quantize(x, "e4m3", colwise=True, codes=out[0], scales=out[1], stream=stream)
    elif kind == "group":
        bs.fp8_group_quantize(x, m_sizes, codes=out[0], scales=out[1], stream=stream)
    else:
        bs.fp8_block_quantize(x, codes=out[0], scales=out[1], stream=stream)


def quant_outputs(torch, kind, shape, dev, pinned=False):
    def mk(sh, dt):
        t = torch.empty(sh, dtype=dt, device="cpu" if pinned else dev)
        return t.pin_memory() if pinned else t
    if kind == "rows":
        return mk(shape, torch.uint8), mk((shape[0], shape[1] // 32), torch.uint8)
    if kind == "cols":
        return mk(shape, torch.uint8), mk((shape[1], shape[0] // 32), torch.uint8)
    if kind == "group":
        return mk(shape, torch.uint8), mk((shape[0] * (shape[1] // 128),), torch.float32)
    return mk(shape, torch.uint8), mk((shape[0], shape[1] // 128, shape[2] // 128), torch.float32)


def quant_oracle_sample(cache, frac, nthreads=None):
    """Oracle quantisation of a `frac` share of every call's rows (rows, columns or weight
    blocks are independent); returns (seconds, algorithmic bytes)."""
    import oracle
    import synthetic
    secs, nbytes = 0.0, 0.0
    for name, shape, seed, kind in quant_ops():
        if name not in cache:
            x = quant_input(shape, seed)
            import torch
            cache[name] = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
        x = cache[name]
        if kind in ("rows", "group"):
            r = max(1, int(shape[0] * frac))
            sub = x[:r]
            t0 = time.perf_counter()
            if kind == "rows":
                oracle.mx_quantize(sub, "e4m3")
            else:
                oracle.fp8_group_quantize(sub, np.array([r // 3, 0, r - r // 3]))
            secs += time.perf_counter() - t0
            nbytes += quant_bytes(kind, sub.shape)
        elif kind == "cols":
            c = max(16, int(shape[1] * frac) // 16 * 16)
            sub = np.ascontiguousarray(x[:, :c])
            t0 = time.perf_counter()
            oracle.mx_quantize(sub, "e4m3", colwise=True)
            secs += time.perf_counter() - t0
            nbytes += quant_bytes(kind, sub.shape)
        else:
            n = max(128, int(shape[1] * frac) // 128 * 128)
            sub = np.ascontiguousarray(x[:1, :n])
            t0 = time.perf_counter()
            oracle.fp8_block_quantize(sub)
            secs += time.perf_counter() - t0
            nbytes += quant_bytes(kind, sub.shape)
    return secs, nbytes


def run_quantize(args):
    import torch
    import block_scaled_precision_mma_gb300 as bs

    ws, rank, local = dist_env()
    dist = init_dist(ws)
    torch.cuda.set_device(local)
    bs.build()
    bs.load()
    dev = torch.device("cuda", local)
    import synthetic
    ms_host = torch.from_numpy(synthetic.gen_m_sizes(16384, 6)).pin_memory()
    ms = ms_host.to(dev)
    ops = []
    for name, shape, seed, kind in quant_ops():
        xh = torch.from_numpy(quant_input(shape, seed)).to(torch.bfloat16).pin_memory()
        ops.append(dict(name=name, kind=kind, shape=shape, x=xh.to(dev), xh=xh,
                        out=quant_outputs(torch, kind, shape, dev),
                        outh=quant_outputs(torch, kind, shape, dev, pinned=True),
                        bytes=quant_bytes(kind, shape)))
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()
    step_bytes = sum(o["bytes"] for o in ops)

    def step(events):
        for o, ev in zip(ops, events):
            flush()
            ev[0].record(stream)
            quant_call(bs, o["kind"], o["x"], o["out"], ms)
            ev[1].record(stream)

    mk = lambda: [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in ops]
    clk = ClockSampler(local).start()
    for _ in range(args.warmup):
        step(mk())
    torch.cuda.synchronize()
    if bs.device_status() != 0:
        raise SystemExit("device status error during warm-up")
    all_events = [mk() for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = bs.launch_count()
    try:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            step(all_events[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    finally:
        clk.stop()
    clk.window(wall0, wall0 + wall)
    n_launch = bs.launch_count() - n0
    st = bs.device_status()
    if st != 0:
        raise SystemExit(f"device status {bs.status_string(st)}")
    per_op_ms = [sum(evs[j][0].elapsed_time(evs[j][1]) for evs in all_events) / args.steps
                 for j in range(len(ops))]

    # end to end: inputs up on one copy stream, codes and scales down on another
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in ops]
    comp_done = [torch.cuda.Event() for _ in ops]
    d2h_done = [torch.cuda.Event() for _ in ops]
    recorded = [False] * len(ops)

    def e2e_step():
        for i, o in enumerate(ops):
            with torch.cuda.stream(h2d_stream):
                if recorded[i]:
                    h2d_stream.wait_event(comp_done[i])
                o["x"].copy_(o["xh"], non_blocking=True)
                h2d_done[i].record(h2d_stream)
            stream.wait_event(h2d_done[i])
            if recorded[i]:
                stream.wait_event(d2h_done[i])
            quant_call(bs, o["kind"], o["x"], o["out"], ms)
            comp_done[i].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(comp_done[i])
                for dst, src in zip(o["outh"], o["out"]):
                    dst.copy_(src, non_blocking=True)
                d2h_done[i].record(d2h_stream)
            recorded[i] = True

    e2e_steps = 0 if args.no_e2e else max(3, min(args.steps, 20))
    h2d = sum(o["xh"].numel() * o["xh"].element_size() for o in ops)
    d2h = sum(t.numel() * t.element_size() for o in ops for t in o["outh"])
    if e2e_steps:
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    e0.record(stream)
    h2d_stream.wait_stream(stream)
    for _ in range(e2e_steps):
        e2e_step()
    stream.wait_stream(d2h_stream)
    stream.wait_stream(h2d_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps if e2e_steps else float("nan")

    step_ms = sum(per_op_ms)
    step_ms, e2e_ms = reduce_max([step_ms, e2e_ms], dist)
    if rank != 0:
        return
    _, hbm_peak, peak_src = measured_peaks()
    dom = max(range(len(ops)), key=lambda j: ops[j]["bytes"])
    achieved = ops[dom]["bytes"] / (per_op_ms[dom] * 1e-3) / 1e9
    kernel = {"rows": "mx_quant_rows_kernel", "cols": "mx_quant_cols_kernel",
              "group": "group_quant_kernel", "block": "block_quant_kernel"}[ops[dom]["kind"]]
    line = {
        "metric": QUANT_METRIC,
        "value": round(ws * step_bytes / (step_ms * 1e-3) / 1e9, 1),
        "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in, e4m3 + e8m0/f32 scales out",
        "data": "synthetic (seeded N(0,1) as BF16)",
        "config": {"workload": "quantize: " + QUANT_TEXT,
                   "l2": "flushed before every call by a 256 MiB write, then a 256 MiB read (the "
                         "write's dirty lines leave L2 before the call), outside the timed events",
                   "parallelism": f"replicas x{ws}",
                   "per_call_ms": {o["name"]: round(t, 4) for o, t in zip(ops, per_op_ms)},
                   "per_call_gbs": {o["name"]: round(o["bytes"] / (t * 1e-3) / 1e9, 1)
                                    for o, t in zip(ops, per_op_ms)}},
        "roofline": {"bound": "hbm", "kernel": kernel, "launch": ops[dom]["name"],
                     "achieved": round(achieved, 1), "peak": round(hbm_peak, 1), "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4),
                     "peak_source": f"{peak_src} HBM copy bandwidth",
                     "traffic": recorded_traffic("quantize")},
        "e2e": None if args.no_e2e else {
            "value": round(ws * step_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "api": "mx_quantize / fp8_group_quantize / fp8_block_quantize with the BF16 input "
                   "copied host->device and codes + scales device->host inside the timed "
                   "region, on two copy streams overlapping the neighbouring calls"},
        "gpu_launches": int(n_launch),
        "clocks": clk.summary(),
        "wall_s_timed": round(wall, 3),
    }
    if not args.no_cpu_baseline and rank == 0:
        cache = {}
        s0, _ = quant_oracle_sample(cache, 1 / 512)            # calibration
        frac = min(1.0, (1 / 512) * args.cpu_seconds / max(s0, 1e-3))
        secs, nb = quant_oracle_sample(cache, frac)
        line["cpu_baseline"] = {"value": round(nb / secs / 1e9, 4), "unit": "GB/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"{frac:.4f} of each call's rows / columns / weight rows "
                                          f"({nb / 1e6:.1f} MB algorithmic, {secs:.1f} s, "
                                          f"single-threaded C oracle)"}
    print(json.dumps(line), flush=True)


def run_quantize_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cache = {}
    s0, _ = quant_oracle_sample(cache, 1 / 1024)
    per_step = max(0.2, args.ref_seconds / max(1, args.steps + args.warmup))
    frac = min(1.0, (1 / 1024) * per_step / max(s0, 1e-3))
    for _ in range(args.warmup):
        quant_oracle_sample(cache, frac)
    secs, nb = 0.0, 0.0
    for _ in range(args.steps):
        a, b = quant_oracle_sample(cache, frac)
        secs += a
        nb += b
    value = nb / secs / 1e9
    line = {
        "impl": "reference", "metric": QUANT_METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 in, e4m3 + scales out",
        "data": "synthetic (seeded N(0,1) as BF16)",
        "config": {"workload": "quantize: " + QUANT_TEXT, "parallelism": "host core"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step: {frac:.4f} of each call's rows / columns / weight rows"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- oracle timing
def time_oracle_sample(spec, rows_per_gemm: int, inputs_cache: dict, nthreads: int):
    """Runs the oracle on `rows_per_gemm` sampled output rows (all columns) of every
    GEMM of the step; returns (seconds, flops)."""
    import oracle
    secs, flops = 0.0, 0.0
    for i, g in enumerate(spec):
        if i not in inputs_cache:
            inputs_cache[i] = make_inputs(dict(g))
        c = inputs_cache[i]
        if g["kind"].startswith("grouped"):
            T = int(np.asarray(c["m_sizes"]).sum())
            rows = np.random.default_rng([8, i]).choice(T, size=min(rows_per_gemm, T), replace=False)
            t0 = time.perf_counter()
            if g["kind"] == "grouped_bf16":
                oracle.grouped_bf16_gemm(c["X"], c["W"], c["m_sizes"], g["N"], g["K"],
                                         rows=np.sort(rows), nthreads=nthreads)
            else:
                oracle.grouped_fp8_gemm(c["X"], c["sX"], c["W"], c["sW"], c["m_sizes"], g["N"],
                                        g["K"], rows=np.sort(rows), nthreads=nthreads)
            secs += time.perf_counter() - t0
            flops += 2.0 * len(rows) * g["N"] * g["K"]
        else:
            M = c["M"]
            rows = np.random.default_rng([8, i]).choice(M, size=min(rows_per_gemm, M), replace=False)
            t0 = time.perf_counter()
            d = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], c["M"], c["N"], c["K"], c["layout"],
                               c["a_fmt"], c["b_fmt"], rows=np.sort(rows), nthreads=nthreads)
            if g.get("act"):
                oracle.bias_act(d, c.get("bias"), g["act"])
            secs += time.perf_counter() - t0
            flops += 2.0 * len(rows) * c["N"] * c["K"]
    return secs, flops


def cpu_baseline(spec, budget_s: float = 15.0):
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    cache = {}
    s, f = time_oracle_sample(spec, 4, cache, cores)       # calibration
    rows = int(max(4, min(4096, 4 * budget_s / max(s, 1e-3))))
    s, f = time_oracle_sample(spec, rows, cache, cores)
    return {"value": round(f / s / 1e12, 6), "unit": "TFLOPS", "cores": cores, "kind": "oracle",
            "sample": f"{rows} random output rows x all N columns of each GEMM of the step "
                      f"({f / 2:.3e} MACs, {s:.1f} s, FP64 table-decode oracle)"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    spec = workload_spec(args.workload)
    cores = os.cpu_count() or 1
    cache = {}
    s, _ = time_oracle_sample(spec, 2, cache, cores)        # calibration + input generation
    per_step_budget = max(0.2, args.ref_seconds / max(1, args.steps + args.warmup))
    rows = int(max(1, min(4096, 2 * per_step_budget / max(s, 1e-3))))
    for _ in range(args.warmup):
        time_oracle_sample(spec, rows, cache, cores)
    secs, flops = 0.0, 0.0
    for _ in range(args.steps):
        a, b = time_oracle_sample(spec, rows, cache, cores)
        secs += a
        flops += b
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) truncated to BF16)" if args.workload == "grouped_bf16"
                else "synthetic (seeded N(0,1), MX-quantised)",
        "config": {"workload": args.workload + ": " + WORKLOAD_TEXT[args.workload],
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {rows} random output rows x all N columns of each GEMM"},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mxfp8_dense",
                    choices=["mxfp8_dense", "mxfp8_bias_gelu", "mxfp8_256", "mxfp4_dense",
                             "linear_triple", "grouped_fp8", "grouped_fp8_packed", "grouped_bf16",
                             "quantize"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling)")
    ap.add_argument("--grouped-width", type=int, default=0, choices=[0, 128, 256],
                    help="grouped tile width: 0 automatic, 128 or 256 (tuning only)")
    ap.add_argument("--grouped-variant", type=int, default=0, choices=[0, 1, 3],
                    help="grouped BF16 tiles: 0 automatic, 1 one CTA, 3 SM pairs (tuning only)")
    ap.add_argument("--dense-variant", type=int, default=0, choices=[0, 1, 3],
                    help="0 automatic, 1 single-CTA tiles, 3 SM-pair MMAs (tuning only)")
    ap.add_argument("--gemm", type=int, default=None,
                    help="run only this GEMM (index into the workload's list) in each step; "
                         "for profiling one shape, not a bench line of the workload")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload == "quantize":
        run_quantize_reference(args) if args.impl == "reference" else run_quantize(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
