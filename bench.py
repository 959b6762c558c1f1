"""Benchmark of the dropless MoE layer (forward + backward) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config mixtral|moe_xs|tiny|skewed|fine] [--no-cpu-baseline]
                    [--depth L] [--block 64|128|256] [--gate] [--tokens T] [--experts E]
                    [--pair 0|1|2|3]

One step = one pass of the whole hot path over one batch: route -> permute+pad
-> topology -> SDD(+act) -> DSD -> combine, then combine backward -> router
backward (d logits) -> SDD(+act') -> DSTD (dW2) -> DSD^T (dx) -> DSTD (dW1[,
dW3]) -> un-permute of dx.  The
default workload is the Mixtral-8x7B-shaped layer (T=8192, d=4096, E=8,
F=14336, top-2 SwiGLU with renormalised weights), the largest of the five
workloads and the one whose products are bound by the tensor cores.  Inputs and weights are seeded synthetic data already resident
in HBM; L2 is flushed (256 MB write) between timed steps, outside the timed
events.  Every op is bracketed by CUDA events on the launching stream, which
gives the per-kernel times used for the roofline of the dominant kernel.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs an
independent replica on its own GPU (the layer has no data-path exchange on
one GPU); the value is the sum of all ranks' work over the slowest rank's
time.  ``--impl reference`` times the fp64 CPU oracle on a bounded sample of
the same workload instead.
"""

from __future__ import annotations

import argparse
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import dmoe_synth as syn  # noqa: E402

METRIC = "dMoE layer fwd+bwd useful TFLOP/s and % of GB300 BF16 peak; permute GB/s vs HBM"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ cost model

def workload_name(cfg, depth=1, block=128, gate=False) -> str:
    return (f"{cfg.name}: T={cfg.T} d={cfg.d} E={cfg.E} F={cfg.F} top-{cfg.k} {cfg.act}"
            + (" renorm" if cfg.renorm else "") + (f" depth={depth}" if depth > 1 else "")
            + (f" block={block}" if block != 128 else "") + (" linear-gate" if gate else ""))


def gate_weights(cfg):
    """Router weights of the linear gate [E, d] (bf16 bits), N(0, 1/d)."""
    return syn.normal_bf16(cfg.seed, 90, (cfg.E, cfg.d), 1.0 / np.sqrt(cfg.d))


def useful_flops(cfg) -> float:
    """2*A*d*F per GEMM (padding excluded); 2 (GELU) or 3 (SwiGLU) GEMMs forward, x3 for fwd+bwd."""
    g = 3 if cfg.act == "swiglu" else 2
    return 3.0 * g * 2.0 * cfg.A * cfg.d * cfg.F


def op_costs(cfg, P: int, nnz: int, live_experts: int, block: int = 128):
    """Algorithmic (bytes, flops) of one launch of each op for this routing.

    Bytes count every operand read once and every output written once;
    flops count the block-sparse products as executed (padded rows
    included, 2 flops per multiply-add).  Weights count only the live
    experts' slices.
    """
    T, d, E, F, k, A = cfg.T, cfg.d, cfg.E, cfg.F, cfg.k, cfg.A
    bf, i4 = 2, 4
    blk = nnz * block * block * bf
    W = live_experts * d * F * bf
    gemm = 2.0 * P * d * F
    swi = cfg.act == "swiglu"
    c = {}
    c["route_topk"] = (T * E * 4 + A * (i4 + 4), 0.0)
    # the router with its own linear gate: x and w_gate in, logits and the
    # routing out
    c["gate_route_topk"] = (T * d * bf + E * d * bf + T * E * 4 + A * (i4 + 4), 2.0 * T * d * E)
    c["permute_pad"] = (T * d * bf + A * i4 + P * d * bf + (A + P) * i4 + (2 * E + 1) * i4, 0.0)
    # padded offsets and token counts in; row offsets, row fill, four
    # per-block index arrays and the transposed column offsets out
    c["build_topology"] = ((2 * E + 1) * i4 + (2 * (P // block) + 1 + 4 * nnz + E * (F // block) + 1) * i4, 0.0)
    # the fused launch: the router's logits in, the permutation and the
    # topology out (expert ids are not read back)
    c["dispatch"] = (c["route_topk"][0] + c["permute_pad"][0] - A * i4 + c["build_topology"][0] - (2 * E + 1) * i4, 0.0)
    if swi:
        c["sdd_fwd"] = (P * d * bf + 2 * W + 3 * blk, 2 * gemm)
    else:
        c["sdd_fwd"] = (P * d * bf + W + 2 * blk, gemm)
    c["dsd_fwd"] = (blk + W + P * d * bf, gemm)
    c["unpermute_combine"] = (A * d * bf + A * (i4 + 4) + T * d * bf, 0.0)
    c["combine_backward"] = (T * d * bf + P * d * bf + P * i4 + A * 4 + P * d * bf + A * 4, 0.0)
    if swi:
        c["sdd_bwd"] = (P * d * bf + W + 2 * blk + 2 * blk, gemm)
        c["dsd_t_dx"] = (2 * blk + 2 * W + P * d * bf, 2 * gemm)
    else:
        c["sdd_bwd"] = (P * d * bf + W + blk + blk, gemm)
        c["dsd_t_dx"] = (blk + W + P * d * bf, gemm)
    c["dstd_dw2"] = (blk + P * d * bf + W, gemm)
    c["dstd_dw1"] = (blk + P * d * bf + W, gemm)
    if swi:
        c["dstd_dw3"] = (blk + P * d * bf + W, gemm)
    c["unpermute_dx"] = (A * d * bf + A * i4 + T * d * bf, 0.0)
    c["route_backward"] = (2 * T * E * 4 + A * (i4 + 4 + 4), 0.0)
    return c


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


OP_SOURCES = {
    "route_topk": ["route.cu", "route.cuh"], "route_backward": ["route.cu", "route.cuh"],
    "permute_pad": ["permute.cu", "route.cuh", "topology.cuh"],
    "dispatch": ["permute.cu", "route.cuh", "topology.cuh"],
    "build_topology": ["topology.cu", "topology.cuh"], "unpermute_combine": ["combine.cu"],
    "combine_backward": ["combine.cu"], "unpermute_dx": ["combine.cu"],
    "gate_route_topk": ["gate.cu", "route.cuh", "tc.cuh", "tmap.cuh"],
}
# the block-sparse products (every other op): the kernel, its tcgen05 / TMA
# helpers and the host code that encodes its tensor maps
BSMM_SOURCES = ["bsmm.cu", "tc.cuh", "tmap.cuh"]


def kernel_source_hash(op: str = "sdd_fwd") -> str:
    """Short hash of the CUDA sources an op's kernel is built from (its own
    .cu file plus the shared device headers): identifies that kernel build."""
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "dropless_moe_block_gb300", "csrc")
    for name in OP_SOURCES.get(op, BSMM_SOURCES) + ["common.cuh"]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:12]


def load_traffic():
    """ncu DRAM traffic per launch, from profiles/traffic.txt lines
    ``<op> <workload> <bytes_per_launch> <kernel_source_hash>``; entries taken
    on other kernel sources are ignored (their counters no longer apply)."""
    out = {}
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if os.path.exists(path):
        for line in open(path):
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if len(parts) >= 4 and parts[3] == kernel_source_hash(parts[0]):
                try:
                    out[(parts[0], parts[1])] = float(parts[2])
                except ValueError:
                    pass
    return out


# ------------------------------------------------------- multi-rank helpers

def max_over_ranks(x: float, device) -> float:
    """Largest x over all ranks (identity without an initialised process group)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flops_per_rank: float, world: int, ms_slowest: float) -> float:
    """Useful TFLOP/s of all replicas together, timed by the slowest rank."""
    return world * flops_per_rank / (ms_slowest * 1e-3) / 1e12


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clock, power and clock-event reasons every ~2 ms through
    NVML (ctypes on libnvidia-ml) while the timed region runs; read-only."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_device: int):
        self.cuda_device = cuda_device
        self.samples = []
        self.window = None
        self._stop = threading.Event()
        self._nvml = None
        self._dev = None
        self.error = None

    def _open(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        dev = ctypes.c_void_p()
        try:
            import torch
            p = torch.cuda.get_device_properties(self.cuda_device)
            bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0".encode()
            rc = nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(dev))
        except Exception:
            rc = -1
        if rc != 0 and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.cuda_device), ctypes.byref(dev)) != 0:
            raise RuntimeError("no NVML handle")
        self._nvml, self._dev = nv, dev
        mx = ctypes.c_uint(0)
        nv.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons

    def _run(self):
        import ctypes
        nv, dev = self._nvml, self._dev
        clk, pw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not self._stop.is_set():
            t = time.perf_counter()
            nv.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(clk))
            nv.nvmlDeviceGetPowerUsage(dev, ctypes.byref(pw))
            self._reasons_fn(dev, ctypes.byref(rs))
            self.samples.append((t, float(clk.value), pw.value / 1000.0, int(rs.value)))
            time.sleep(0.002)

    def __enter__(self):
        try:
            self._open()
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        except Exception as e:  # no NVML: report it, never fall back silently
            self.error = str(e)
        return self

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def __exit__(self, *a):
        self._stop.set()
        if self._nvml is not None:
            self._thread.join(timeout=2)

    def summary(self):
        if self.error:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"unsampled: {self.error}"], "samples": 0}
        t0, t1 = self.window or (-1e30, 1e30)
        inside = [s for s in self.samples if t0 <= s[0] <= t1] or self.samples[-3:]
        reasons = sorted({name for s in inside for bit, name in self.REASONS.items() if s[3] & bit})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "power_w_max": max(s[2] for s in inside), "reasons": reasons, "samples": len(inside),
                "source": "NVML, 2 ms period, inside the timed region"}


# ----------------------------------------------------------- CPU oracle leg

def oracle_sample(cfg, inp, n_tokens, depth=1):
    """Run the fp64 oracle layer (fwd + bwd) on the first n tokens; returns (seconds, useful flops)."""
    import oracle as O
    n = int(n_tokens)
    t0 = time.perf_counter()
    # with a linear gate the router logits are part of the work
    logits = (O.gate_logits(inp["x"][:n], inp["w_gate"]).astype(np.float32) if "w_gate" in inp
              else inp["logits"][:n])
    if depth == 1:
        # weight gradients computed but not kept: at the large workloads
        # their float64 copies alone would exceed host memory
        O.layer_per_expert(inp["x"][:n], logits, inp["w1"], inp["w2"], inp["dy"][:n], cfg.k, cfg.act,
                           cfg.renorm, w3=inp.get("w3"), keep_weight_grads=False)
    else:
        O.layer_deep_per_expert(inp["x"][:n], logits, inp["w1s"], inp["w2s"], inp["dy"][:n], cfg.k,
                                cfg.act, cfg.renorm, w3s=inp.get("w3s"))
    dt = time.perf_counter() - t0
    return dt, depth * useful_flops(cfg.scaled(n))


def cpu_cores():
    """Cores this process may run on (its CPU affinity)."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cgroup_cpu_quota():
    """CPU limit of this process's cgroup in cores (cgroup v2 cpu.max, else
    v1 cfs quota / period), or None when unlimited or unreadable."""
    try:
        with open("/sys/fs/cgroup/cpu.max") as f:
            q, per = f.read().split()[:2]
        return None if q == "max" else round(int(q) / int(per), 2)
    except Exception:
        pass
    try:
        with open("/sys/fs/cgroup/cpu/cpu.cfs_quota_us") as f:
            q = int(f.read())
        with open("/sys/fs/cgroup/cpu/cpu.cfs_period_us") as f:
            per = int(f.read())
        return None if q <= 0 else round(q / per, 2)
    except Exception:
        return None


def host_cpus():
    """The host's CPU figures beside the affinity count the lines report as
    ``cores``: every online CPU of the machine and the cgroup's quota."""
    return {"cpu_count": os.cpu_count(), "affinity": cpu_cores(), "cgroup_quota_cores": cgroup_cpu_quota()}


def per_token_flops(cfg, depth=1) -> float:
    """Useful fwd+bwd flops of one token (all k of its assignments)."""
    return depth * useful_flops(cfg) / cfg.T


def sample_tokens(cfg, gflop: float, depth=1, cap=None) -> int:
    """Tokens whose fwd+bwd is about `gflop` GFLOP: at least 64, at most
    `cap` (default T)."""
    n = int(gflop * 1e9 / per_token_flops(cfg, depth))
    return max(64, min(cap or cfg.T, n))


class CpuUse:
    """Effective parallelism of the code run inside the block: process CPU
    time (user + system, all threads) over wall time."""

    def __enter__(self):
        self.t, self.w = os.times(), time.perf_counter()
        return self

    def __exit__(self, *exc):
        t = os.times()
        cpu = (t.user - self.t.user) + (t.system - self.t.system)
        self.threads = cpu / max(time.perf_counter() - self.w, 1e-9)
        return False


def cpu_baseline(cfg, inp, target_s=12.0, depth=1):
    """The oracle on a token prefix grown until one pass takes about
    target_s / 4 (at most the whole layer), then repeated until about
    target_s of CPU work has been timed."""
    n = sample_tokens(cfg, 5.0, depth, cap=max(64, cfg.T // 64))
    with CpuUse() as use:  # over every pass, the sizing ones included
        dt, fl = oracle_sample(cfg, inp, n, depth)
        while dt < target_s / 4 and n < cfg.T:
            n = min(cfg.T, int(n * min(8.0, max(2.0, target_s / max(dt, 1e-3) / 2))))
            dt, fl = oracle_sample(cfg, inp, n, depth)
        total, reps = dt, 1
        while total < target_s:
            total += oracle_sample(cfg, inp, n, depth)[0]
            reps += 1
    return {"value": fl * reps / total / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "threads_effective": round(use.threads, 1), "host": host_cpus(),
            "sample": f"fp64 numpy oracle, forward+backward of the first {n} of {cfg.T} tokens "
                      f"(all weights, decoded to fp64 one expert at a time inside the timed call), "
                      f"{reps} pass(es), {total:.2f} s"}


# ---------------------------------------------------------------- GPU arm

def bf16_dev(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def isolated_kernel_us(fns, device, reps=10, rounds=3):
    """Per-launch device time of each call on its own: a CUDA graph of
    reps x [256 MB read-only pass over a flush buffer, call] minus a graph of
    the passes alone, timed with CUDA events around the replay (best of
    `rounds`).  Every launch starts with a cold L2 holding no dirty lines and
    still pays for writing back its own output; no event sits between the
    kernels, so the number carries no per-node event overhead."""
    import torch
    buf = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    acc = torch.zeros((), dtype=torch.float32, device=device)

    def flush():
        torch.sum(buf, dim=0, out=acc)

    def timed(f):
        for _ in range(2):
            flush()
            f()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            for _ in range(reps):
                flush()
                f()
        best = []
        for _ in range(rounds):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            b.synchronize()
            best.append(a.elapsed_time(b))
        del g
        return 1e3 * min(best) / reps

    base = timed(lambda: None)
    return {n: max(0.0, timed(f) - base) for n, f in fns.items()}


def run_ours(args, cfg, rank, world, local_rank):
    import torch
    import dropless_moe_block_gb300 as dm

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dm.set_pair(args.pair)
    depth = args.depth
    inp = syn.make_inputs(cfg)
    x = bf16_dev(inp["x"], device)
    logits = torch.from_numpy(inp["logits"]).to(device)
    if depth == 1:
        w1 = bf16_dev(inp["w1"], device)
        w2 = bf16_dev(inp["w2"], device)
        w3 = bf16_dev(inp["w3"], device) if cfg.act == "swiglu" else None
    else:  # lists of expert blocks
        inp.update(syn.make_deep_weights(cfg, depth))
        w1 = [bf16_dev(w, device) for w in inp["w1s"]]
        w2 = [bf16_dev(w, device) for w in inp["w2s"]]
        w3 = [bf16_dev(w, device) for w in inp["w3s"]] if cfg.act == "swiglu" else None
    dy = bf16_dev(inp["dy"], device)
    wg = None
    if args.gate:
        inp["w_gate"] = gate_weights(cfg)
        wg = bf16_dev(inp["w_gate"], device)
    layer = dm.DMoELayer(cfg.T, cfg.d, cfg.E, cfg.F, cfg.k, cfg.act, cfg.renorm, device=device, depth=depth,
                         block=args.block)
    calls = layer.forward_calls(x, logits, w1, w2, w3, wg) + layer.backward_calls(dy, x, w1, w2, w3)
    names = [n for n, _ in calls]
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        for _, f in calls:
            f()
    torch.cuda.synchronize()
    if dm.get_error(clear=True) != 0:
        raise RuntimeError("device error word set during warm-up")

    K = args.steps
    per_op = {n: [] for n in names}
    step_ms = []
    # The step as one CUDA graph (timed per replay from outside), plus a
    # second graph with an event node around every call for the per-kernel
    # times; the eager loop (host-queued behind a GPU-side wait) is the
    # fallback when capture is not available.
    graph, graph_ev, evs, exec_mode = None, None, None, "eager"
    try:
        graph, graph_launches = layer.capture(x, logits, w1, w2, w3, dy=dy, concurrent=True, w_gate=wg)
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(calls) + 1)]
        graph_ev, _ = layer.capture(x, logits, w1, w2, w3, dy=dy, events=evs, w_gate=wg)
        exec_mode = "cuda_graph (forward combine and independent backward products on a second stream)"
    except Exception as e:  # noqa: BLE001 - reported in the JSON line
        exec_mode = f"eager (graph capture failed: {type(e).__name__}: {str(e)[:120]})"
        graph = graph_ev = None
        torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(K)]
    ends = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    n_launch0 = dm.launch_count()
    with ClockSampler(device.index) as clocks:
        time.sleep(0.02)
        wall0 = time.perf_counter()
        for s in range(K):
            flush.fill_(float(s))  # L2 flush, outside the timed events
            if graph is not None:
                ends[s][0].record(stream)
                graph.replay()
                ends[s][1].record(stream)
            else:
                # a GPU-side wait (outside the timed events) lets the host queue
                # the whole step, so the events time the kernels, not the host
                torch.cuda._sleep(2_000_000)
                ev[s][0].record(stream)
                for i, (_, f) in enumerate(calls):
                    f()
                    ev[s][i + 1].record(stream)
        if graph is not None:
            # per-kernel times: the same step with event nodes between calls
            for s in range(K):
                flush.fill_(float(s))
                graph_ev.replay()
                evs[-1].synchronize()
                for i, n in enumerate(names):
                    per_op[n].append(evs[i].elapsed_time(evs[i + 1]))
        torch.cuda.synchronize()
        wall1 = time.perf_counter()
        clocks.mark(wall0, wall1)
    wall = wall1 - wall0
    launches = graph_launches * 2 * K if graph is not None else dm.launch_count() - n_launch0
    if world > 1:
        torch.distributed.barrier()
    err = dm.get_error(clear=True)
    if err:
        raise RuntimeError(f"device error word {err:#x}")
    for s in range(K):
        if graph is not None:
            step_ms.append(ends[s][0].elapsed_time(ends[s][1]))
        else:
            step_ms.append(ev[s][0].elapsed_time(ev[s][-1]))
            for i, n in enumerate(names):
                per_op[n].append(ev[s][i].elapsed_time(ev[s][i + 1]))
    ms_step = float(np.mean(step_ms))

    ms_max = max_over_ranks(ms_step, device)  # slowest rank decides

    P = int(layer.P_dev.item())
    nnz = layer.topo.nnz()
    live = int((layer.tokens_per_expert > 0).sum().item())
    costs = op_costs(cfg, P, nnz, live, args.block)
    # the calls of expert block l carry the suffix _l; they cost what block 1 does
    costs.update({n: costs[re.sub(r"_\d+$", "", n)] for n in names if n not in costs})
    peaks, peak_src = load_peaks()
    mean_us = {n: 1e3 * float(np.mean(v)) for n, v in per_op.items()}
    kernel_sum_us = sum(mean_us.values())
    # each call alone (cold L2, no event nodes between kernels): the
    # duration the roofline of the dominant kernel is computed from
    try:
        iso_us = isolated_kernel_us(dict(calls), device)
        iso_note = ("graph of 10 x [256 MB read-only L2 flush, kernel] minus the flushes alone, "
                    "CUDA events around the replay, best of 3")
    except Exception as e:  # noqa: BLE001 - reported in the JSON line
        iso_us, iso_note = dict(mean_us), f"in-step event times (isolated timing failed: {type(e).__name__})"
        torch.cuda.synchronize()
    if dm.get_error(clear=True):
        raise RuntimeError("device error word set during the isolated kernel timing")
    dom = max(mean_us, key=mean_us.get)
    b, f = costs[dom]
    t_dom = iso_us[dom] * 1e-6
    hbm_t = b / (peaks["hbm_gbs"] * 1e9)
    ten_t = f / (peaks["bf16_tflops"] * 1e12) if f else 0.0
    traffic = load_traffic().get((dom, cfg.name)) if depth == 1 and args.block == 128 else None
    if ten_t > hbm_t:
        roof = {"bound": "tensor", "achieved": f / t_dom / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": b / t_dom / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    # the same kernel inside the timed step, against the peak for work timed
    # inside a long step (sustained, under the power cap)
    if roof["bound"] == "tensor":
        sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
        roof["in_step"] = {"achieved": f / (mean_us[dom] * 1e-6) / 1e12, "peak": sus,
                           "frac": f / (mean_us[dom] * 1e-6) / 1e12 / sus,
                           "peak_source": "MEASURED_PEAKS.json bf16_tflops_sustained" if peak_src == "measured"
                           else peak_src}
    else:
        roof["in_step"] = {"achieved": b / (mean_us[dom] * 1e-6) / 1e9, "peak": peaks["hbm_gbs"],
                           "frac": b / (mean_us[dom] * 1e-6) / 1e9 / peaks["hbm_gbs"]}
    roof.update({"traffic": traffic, "kernel": dom, "kernel_source": kernel_source_hash(re.sub(r"_\d+$", "", dom)), "algorithmic_bytes": b, "algorithmic_flops": f,
                 "peak_source": f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" else peak_src,
                 "mean_us": iso_us[dom], "timing": iso_note, "mean_us_in_step": mean_us[dom]})

    flops = depth * useful_flops(cfg)
    value = whole_job_value(flops, world, ms_max)
    # the permutation runs inside the fused dispatch launch (route + permute +
    # topology) unless the layer was built with the three separate calls
    front = "permute_pad" if "permute_pad" in mean_us else "dispatch"
    perm_gbs = costs[front][0] / (mean_us[front] * 1e-6) / 1e9
    comb_gbs = costs["unpermute_combine"][0] / (mean_us["unpermute_combine"] * 1e-6) / 1e9
    gemm_names = [n for n in names if n.startswith(("sdd", "dsd", "dstd"))]
    gemm_us = sum(mean_us[n] for n in gemm_names)
    gemm_tflops = flops / (gemm_us * 1e-6) / 1e12

    e2e = run_e2e(args, cfg, layer, inp, device, x, logits, w1, w2, w3, dy, flops, wg)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights; shapes of the workload)",
        "config": {"workload": workload_name(cfg, depth, args.block, args.gate), "depth": depth,
                   "block": args.block, "router_logits": "linear gate in the router" if args.gate else "given",
                   "cta_pairs": ["per call", "never", "wherever allowed",
                                 "wherever allowed, 256 x 512 tiles wherever allowed"][args.pair],
                   "T": cfg.T, "d": cfg.d, "E": cfg.E, "F": cfg.F, "k": cfg.k, "act": cfg.act, "P": P, "nnz": nnz,
                   "pad_share": 1.0 - cfg.A / P, "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "flushed between steps by a 256 MB write outside the timed events",
                   "exec": exec_mode},
        "pct_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
        "pct_bf16_peak_sustained": 100.0 * value / world / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]),
        "gemm_useful_tflops": gemm_tflops,
        "permute_gbs": perm_gbs, "permute_frac_hbm": perm_gbs / peaks["hbm_gbs"], "permute_kernel": front,
        "combine_gbs": comb_gbs, "combine_frac_hbm": comb_gbs / peaks["hbm_gbs"],
        "topology_us": mean_us.get("build_topology"), "dispatch_us": mean_us.get("dispatch"),
        "kernels_us": {n: round(v, 2) for n, v in mean_us.items()},
        "kernels_isolated_us": {n: round(v, 2) for n, v in iso_us.items()},
        "kernels_sum_us": round(kernel_sum_us, 2),
        "roofline": roof,
        "gpu_launches": launches,
        "wall_s_timed_region": wall,
        "clocks": clocks.summary(),
        "e2e": e2e,
    }
    return result, inp


def run_e2e(args, cfg, layer, inp, device, x, logits, w1, w2, w3, dy, flops, wg=None):
    """Same metric through the public API with host buffers: every step
    copies its inputs (x, logits, dy) in from pinned host memory and its
    results (y, dx, d_gate, d_logits) out to pinned host memory; the
    weights and the weight gradients stay in device memory.  dm.StepRunner
    overlaps those copies with the neighbouring steps' compute (inputs of
    step s+1 in, results of step s-1 out, on their own streams)."""
    import torch
    import dropless_moe_block_gb300 as dm
    hx = torch.from_numpy(np.ascontiguousarray(inp["x"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    hl = None if wg is not None else torch.from_numpy(inp["logits"]).pin_memory()
    hdy = torch.from_numpy(np.ascontiguousarray(inp["dy"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    runner = dm.StepRunner(layer, w1, w2, w3, w_gate=wg)
    hout = runner.host_outputs()
    stream = torch.cuda.current_stream()
    steps = max(1, args.steps)
    runner.run(hx, hl, hdy, hout, 2)  # warm the copy engines and both graphs
    runner.finish()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    runner.run(hx, hl, hdy, hout, steps)
    runner.finish()
    e1.record(stream)
    e1.synchronize()
    if dm.get_error(clear=True):
        raise RuntimeError("device error word set during the end-to-end steps")
    ms = e0.elapsed_time(e1) / steps
    bi = hx.numel() * 2 + (hl.numel() * 4 if hl is not None else 0) + hdy.numel() * 2
    bo = sum(t.numel() * t.element_size() for t in hout[0])
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "inputs_copied": ["x", "dy"] + ([] if hl is None else ["logits"]),
            "results_copied": list(dm.StepRunner.RESULTS),
            "resident": "weights and weight gradients (dW1, dW2" + (", dW3" if w3 is not None else "") +
                        ") stay in device memory, as in a training step whose optimizer runs on the GPU",
            "pipelining": "step s+1's inputs copied in and step s-1's results copied out while step s computes"}


def run_reference(args, cfg):
    """The fp64 CPU oracle as the reference arm, a bounded sample per step."""
    inp = syn.make_inputs(cfg)
    depth = args.depth
    if depth > 1:
        inp.update(syn.make_deep_weights(cfg, depth))
    if args.gate:
        inp["w_gate"] = gate_weights(cfg)
    # about 50 GFLOP of fp64 work per step, at most T/16 tokens
    n = sample_tokens(cfg, 50.0, depth, cap=max(64, cfg.T // 16 // depth))
    for _ in range(args.warmup):
        oracle_sample(cfg, inp, min(n, 64), depth)
    times, flops = [], 0.0
    with CpuUse() as use:
        for _ in range(args.steps):
            dt, fl = oracle_sample(cfg, inp, n, depth)
            times.append(dt)
            flops = fl
    sec = float(np.mean(times))
    value = flops / sec / 1e12
    sample = (f"fp64 numpy oracle, forward+backward of the first {n} of {cfg.T} tokens (all weights, decoded "
              f"to fp64 one expert at a time inside the timed call) per step")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": workload_name(cfg, depth, args.block, args.gate), "sampled_tokens": n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "threads_effective": round(use.threads, 1), "host": host_cpus(), "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def parser():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="mixtral", choices=sorted(syn.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0, help="override T (smaller cases for profiling)")
    ap.add_argument("--experts", type=int, default=0, help="override E (smaller cases for profiling)")
    ap.add_argument("--depth", type=int, default=1,
                    help="expert blocks per expert (SDD -> act -> DSD, repeated; 1 = the two-layer MLP)")
    ap.add_argument("--gate", action="store_true",
                    help="the layer computes its router logits with a linear gate (fused into the router)")
    ap.add_argument("--block", type=int, default=128, choices=[64, 128, 256],
                    help="B of the B x B sparse blocks (expert groups padded to multiples of B)")
    ap.add_argument("--pair", type=int, default=0, choices=[0, 1, 2, 3],
                    help="CTA pairs in the block-sparse products: 0 chosen per call, 1 never, 2 wherever allowed "
                         "(256 x 256 pair tiles), 3 wherever allowed with 256 x 512 tiles wherever allowed")
    return ap


def main():
    ap = parser()
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.depth < 1:
        ap.error("--depth must be >= 1")
    cfg = syn.CONFIGS[args.config]
    if args.tokens or args.experts:
        import dataclasses
        T = args.tokens or cfg.T
        E = args.experts or cfg.E
        cfg = dataclasses.replace(cfg, T=T, E=E, name=f"{cfg.name}_T{T}_E{E}")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, cfg)), flush=True)
        return

    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    result, inp = run_ours(args, cfg, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(cfg, inp, depth=args.depth)
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
