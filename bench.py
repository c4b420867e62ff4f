"""Benchmark of the fused row-parallel GEMM + partial channel-reduce hot path.

One step = one pass of the whole path over one synthetic batch of the chosen
workload.  Default: the Llama2-7B-shaped layers at prefill (h = 4096, t = 8
emulated tensor-parallel ranks, N = 4096 tokens, p = 0.5, contiguous S): the
fused forward (GEMM + partial channel-reduce into t rank outputs) of the
attention out-projection (K = 4096) and of the MLP down-projection (K = 11008).
The training workloads (130M, 1.1B) add each layer's backward (partial reduce
of the upstream gradient, dX, dW).  Metric: algorithmic TFLOP/s (2NKh forward,
4NKh backward per layer, independent of p).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl caat|reference]
                  [--workload 7b_prefill|130m|1.1b|7b_decode8|7b_prefill256|130m_stack]
                  [--layout contiguous|random] [--p P] [--t T] [--placement reduce_dout|column]
                  [--no-extras] [--no-stack]

Under torchrun (N GPUs) the workload's t ranks are spread over the GPUs, t / N on
each: every process runs the fused forward of its own ranks and the partial
channel-reduce across processes (NCCL all-to-all and all-gather of the S
channels, folded in rank order); the channels outside S never leave their GPU.
The layer is the same for every N (strong scaling); rank 0 prints one JSON line
with the slowest rank's time.  ``--impl reference`` times the CPU oracle on the
host cores instead.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import caat_inputs as ci  # noqa: E402

METRIC = "fused rowpar-GEMM+partial-reduce TFLOP/s & reduce GB/s (% of GB300 peak), 1 GPU"
L2_BYTES = 129 * 2**20


# untimed spin before each timed step (clock cycles, about 0.5 ms): the host needs
# 140 - 330 us to queue a training step of four calls, and the spin keeps it ahead of
# the GPU so that no host gap falls inside a timed call
STEP_SPIN_CYCLES = 1000000

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# dominant forward kernel, from an ncu capture of the same workload with the
# kernels as they are now (7B prefill: the full capture of one step, plain and
# compact outputs, and at 256 tokens; 130M: the one-pass launch list, averaged
# over its steps); a
# workload or layer without a capture reports null.  Output lines still dirty in
# L2 when the kernel ends are not in the count.
DRAM_TRAFFIC = {
    ("7b_prefill", "out_proj"): 118.40e6 + 208.71e6,
    ("7b_prefill", "down_proj"): 419.26e6 + 221.02e6,
    ("7b_prefill_compact", "out_proj"): 80.22e6 + 100.05e6,
    ("7b_prefill_compact", "down_proj"): 404.57e6 + 115.12e6,
    ("130m", "out_proj"): 13.85e6 + 36.30e6,
    ("130m", "down_proj"): 57.29e6 + 38.94e6,
    ("7b_prefill256", "out_proj"): 35.69e6 + 0.06e6,
    ("7b_prefill256", "down_proj"): 95.91e6 + 3.93e6,
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- GPU arm

class LayerData:
    def __init__(self, torch, w, li, device):
        L = w.layers[li]
        X, Wl, G = ci.layer_tensors(w, li)
        self.K = L.K
        self.name = L.name
        self.S = None
        bf = torch.bfloat16

        def dev(a):
            return torch.from_numpy(ci.bf16_words(a).view(np.int16)).to(device).view(bf)

        self.X_host = ci.bf16_words(X)
        self.X = dev(X)
        self.Wstore = dev(np.ascontiguousarray(Wl.T))     # nn.Linear layout [h, K]
        self.W = self.Wstore.t()
        self.G_host = [ci.bf16_words(G[r]) for r in range(w.t)] if G is not None else None
        self.G = [dev(G[r]) for r in range(w.t)] if G is not None else None
        self.Y = [torch.empty((w.N, w.h), dtype=bf, device=device) for _ in range(w.t)]
        self.dX = torch.empty((w.N, L.K), dtype=bf, device=device)
        self.dWstore = torch.empty((w.h, L.K), dtype=bf, device=device)
        self.dW = self.dWstore.t()
        self.flops_fwd = 2.0 * w.N * L.K * w.h
        self.flops_bwd = 4.0 * w.N * L.K * w.h if w.backward else 0.0
        self.bytes_fwd = 2.0 * (w.N * L.K + L.K * w.h + w.t * w.N * w.h)

    def make_compact(self, torch, w, S, device):
        """Compact outputs (the S channels once, YS, and each rank's others, YN[r])
        in place of Y, and the gradient in the same form: dYS = the sum over ranks
        of G_r on S, dYN[r] = G_r outside S (device tensors and host words)."""
        bf = torch.bfloat16
        U = np.setdiff1d(np.arange(w.h), S)
        ns = int(S.size)
        self.Y = None
        self.YS = torch.empty((w.N, ns), dtype=bf, device=device)
        self.YN = [torch.empty((w.N, w.h - ns), dtype=bf, device=device) for _ in range(w.t)]
        self.bytes_fwd = 2.0 * (w.N * self.K + self.K * w.h + w.N * ns + w.t * w.N * (w.h - ns))
        if self.G_host is None:
            return
        G = [ci.words_to_f32(g) for g in self.G_host]
        gs = np.zeros((w.N, ns), dtype=np.float32)
        for g in G:
            gs += g[:, S]
        self.dYS_host = ci.bf16_words(gs)
        self.dYN_host = [ci.bf16_words(np.ascontiguousarray(g[:, U])) for g in G]

        def dev(a):
            return torch.from_numpy(a.view(np.int16)).to(device).view(bf)
        self.dYS = dev(self.dYS_host)
        self.dYN = [dev(a) for a in self.dYN_host]
        self.G = None


def job_rate(dist, device, ms_local, flops_per_step, steps):
    """Whole-job time and throughput of a weak-scaling run: every rank did
    `steps` steps of `flops_per_step`, so the job did world times one rank's work,
    in the time of its slowest rank (the maximum over ranks of `ms_local`).
    Returns (ms, TFLOP/s); dist is torch.distributed or None for one process."""
    ms, world = float(ms_local), 1
    if dist is not None:
        import torch
        tt = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms, world = float(tt.item()), dist.get_world_size()
    return ms, flops_per_step * steps * world / (ms * 1e-3) / 1e12


def _setup_dist():
    """(dist or None, rank, world, device) of this process (one GPU per rank)."""
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return dist, rank, world, torch.device("cuda", torch.cuda.current_device())


class LayerStep:
    """One workload's layers resident on the device, with its channel set and the
    backward workspace: `run(evs)` issues one step (every layer's fused forward,
    then its backward when the workload trains), recording an event before each
    call and one after the last."""

    def __init__(self, torch, caat, w, device, compact=False):
        self.torch, self.caat, self.w = torch, caat, w
        self.compact = compact
        S = caat.select_channels(w.h, w.p, w.layout, w.seeds()["perm"])
        # a contiguous S is passed by its size (the library's null-index form)
        self.sel = int(S.size) if w.layout == 0 else torch.from_numpy(S).to(device)
        self.layers = [LayerData(torch, w, i, device) for i in range(len(w.layers))]
        ws_bytes = max([caat.rowpar_linear_bwd_workspace(w.t, w.N, L.K, w.h, 1, 0) for L in w.layers] + [256])
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        self.wsf = self.ws
        if compact:
            idx = w.layout != 0 and 0 < S.size < w.h
            for L in self.layers:
                L.make_compact(torch, w, S, device)
            self.wsf = torch.empty(max([caat.rowpar_linear_compact_workspace(w.t, w.N, L.K, w.h, 1, idx, False)
                                        for L in w.layers] + [256]), dtype=torch.uint8, device=device)
            self.ws = torch.empty(max([caat.rowpar_linear_compact_workspace(w.t, w.N, L.K, w.h, 1, idx, True)
                                       for L in w.layers] + [256]), dtype=torch.uint8, device=device)
        self.names = []
        for L in self.layers:
            self.names.append("fwd_" + L.name)
            if w.backward:
                self.names.append("bwd_" + L.name)
        self.flops = sum(L.flops_fwd + L.flops_bwd for L in self.layers)

    def run(self, evs=None):
        caat, w, stream = self.caat, self.w, self.torch.cuda.current_stream()
        k = 0
        for L in self.layers:
            if evs is not None:
                evs[k].record(stream); k += 1
            if self.compact:
                caat.rowpar_linear_fwd_compact(L.X, L.W, w.t, self.sel, YS=L.YS, YN=L.YN, workspace=self.wsf)
            else:
                caat.rowpar_linear_fwd(L.X, L.W, w.t, self.sel, outs=L.Y)
            if w.backward:
                if evs is not None:
                    evs[k].record(stream); k += 1
                if self.compact:
                    caat.rowpar_linear_bwd_compact(L.X, L.W, L.dYS, L.dYN, w.t, sel=self.sel, dX=L.dX, dW=L.dW,
                                                   workspace=self.ws)
                else:
                    caat.rowpar_linear_bwd(L.X, L.W, L.G, w.t, self.sel, caat.CAAT_BWD_REDUCE_DOUT,
                                           dX=L.dX, dW=L.dW, workspace=self.ws)
        if evs is not None:
            evs[k].record(stream)


class TPLayer:
    """One layer's data on process g of `world`: the t ranks of the workload are
    spread over the processes, t / world on each GPU; this process holds the input
    columns and weight rows of its own ranks (the same seeded draws as one GPU
    holding all t)."""

    def __init__(self, torch, w, li, device, g, world):
        L = w.layers[li]
        X, Wl, G = ci.layer_tensors(w, li)
        self.t_local = w.t // world
        kl = L.K // world
        cols = slice(g * kl, (g + 1) * kl)
        bf = torch.bfloat16

        def dev(a):
            return torch.from_numpy(ci.bf16_words(np.ascontiguousarray(a)).view(np.int16)).to(device).view(bf)

        self.name, self.K, self.kl = L.name, L.K, kl
        self.X_host = ci.bf16_words(np.ascontiguousarray(X[:, cols]))
        self.X = dev(X[:, cols])
        self.Wstore = dev(np.ascontiguousarray(Wl[cols, :].T))      # nn.Linear layout [h, kl]
        self.W = self.Wstore.t()
        ranks = range(g * self.t_local, (g + 1) * self.t_local)
        self.G_host = [ci.bf16_words(G[r]) for r in ranks] if G is not None else None
        self.G = [dev(G[r]) for r in ranks] if G is not None else None
        self.Y = [torch.empty((w.N, w.h), dtype=bf, device=device) for _ in range(self.t_local)]
        self.dY = [torch.empty((w.N, w.h), dtype=bf, device=device) for _ in range(self.t_local)] \
            if G is not None else None
        self.dX = torch.empty((w.N, kl), dtype=bf, device=device)
        self.dWstore = torch.empty((w.h, kl), dtype=bf, device=device)
        self.dW = self.dWstore.t()
        # this process's share of the layer's algorithmic work
        self.flops_fwd = 2.0 * w.N * kl * w.h
        self.flops_bwd = 4.0 * w.N * kl * w.h if w.backward else 0.0
        self.bytes_fwd = 2.0 * (w.N * kl + kl * w.h + self.t_local * w.N * w.h)


class TPStep:
    """The workload's step with its t ranks spread over the processes of the
    default group (one GPU each): per layer the forward with the partial
    channel-reduce across processes, then (training workloads) the backward with
    the reduce on the upstream gradient across processes."""

    def __init__(self, torch, caat, w, device, g, world):
        from partial_activation_sync_gb300 import tp
        if w.t % world != 0:
            raise SystemExit("bench: %d ranks do not split over %d GPUs" % (w.t, world))
        self.torch, self.caat, self.w, self.tp = torch, caat, w, tp
        S = caat.select_channels(w.h, w.p, w.layout, w.seeds()["perm"])
        self.sel = int(S.size) if w.layout == 0 else torch.from_numpy(S).to(device)
        self.layers = [TPLayer(torch, w, i, device, g, world) for i in range(len(w.layers))]
        self.pr = tp.PartialReduce()
        self.side = torch.cuda.Stream(device=device)
        self.names = []
        for L in self.layers:
            self.names.append("fwd_" + L.name)
            if w.backward:
                self.names.append("bwd_" + L.name)
        self.flops = sum(L.flops_fwd + L.flops_bwd for L in self.layers)

    def run(self, evs=None, io=None):
        stream = self.torch.cuda.current_stream()
        k = 0
        for li, L in enumerate(self.layers):
            B = io[li] if io is not None else L
            if evs is not None:
                evs[k].record(stream); k += 1
            self.tp.rowpar_linear_fwd_tp(B.X, L.W, L.t_local, self.sel, self.pr, outs=B.Y, side=self.side)
            if self.w.backward:
                if evs is not None:
                    evs[k].record(stream); k += 1
                self.tp.rowpar_linear_bwd_tp(B.X, L.W, B.G, L.t_local, self.sel, self.pr, dX=B.dX, dW=B.dW,
                                             dY=L.dY)
        if evs is not None:
            evs[k].record(stream)


def time_steps(torch, caat, ls, steps, warmup, device, dist=None, clocks=None):
    """W untimed warm-up steps, then exactly `steps` timed steps between a barrier
    and a synchronize on both sides.  Every call of a step is bracketed by CUDA
    events on the launching stream; an untimed spin kernel before each step lets
    the host queue the whole step (its calls then run back to back), and the L2 is
    flushed between steps by reading a buffer twice its size (untimed).
    Returns (per-call ms summed over the steps, library launches in the region,
    clock record or None)."""
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    n_calls = len(ls.names)
    for _ in range(warmup):
        ls.run()
        flush.sum()
    torch.cuda.synchronize()
    assert caat.device_status() == 0
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    launches0 = caat.launch_count()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    all_evs = []
    for _ in range(steps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_calls + 1)]
        torch.cuda._sleep(STEP_SPIN_CYCLES)
        ls.run(evs)
        all_evs.append(evs)
        flush.sum()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    launches = caat.launch_count() - launches0
    clk = clocks.stop() if clocks is not None else None
    assert caat.device_status() == 0
    per_call = np.zeros(n_calls)
    for evs in all_evs:
        for i in range(n_calls):
            per_call[i] += evs[i].elapsed_time(evs[i + 1])
    del flush
    return per_call, launches, clk


def roofline_of(ls, per_call, steps, peaks, kernel_name):
    """Roofline object of the dominant forward call of a step: algorithmic FLOPs
    (or bytes, below the ridge) per launch over its mean event-timed duration."""
    w = ls.w
    fwd_idx = [i for i, n in enumerate(ls.names) if n.startswith("fwd_")]
    dom = max(fwd_idx, key=lambda i: per_call[i])
    Ld = ls.layers[fwd_idx.index(dom)]
    t_dom = per_call[dom] / steps * 1e-3
    ai = Ld.flops_fwd / Ld.bytes_fwd
    ridge = peaks["bf16"] * 1e12 / (peaks["hbm"] * 1e9)
    if ai >= ridge:
        ach = Ld.flops_fwd / t_dom / 1e12
        roof = {"kernel": "%s (%s forward)" % (kernel_name, Ld.name), "bound": "tensor",
                "achieved": round(ach, 2), "peak": peaks["bf16"], "unit": "TFLOP/s",
                "frac": round(ach / peaks["bf16"], 4)}
        roof["peak_kind"] = "dense bf16 burst (cuBLAS 8192^3, best of 10)"
    else:
        ach = Ld.bytes_fwd / t_dom / 1e9
        roof = {"kernel": "%s (%s forward)" % (kernel_name, Ld.name), "bound": "hbm",
                "achieved": round(ach, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm"], 4)}
        roof["peak_kind"] = "copy bandwidth (read + write)"
    roof["peak_source"] = "of measured (MEASURED_PEAKS.json)" if peaks["source"] == "measured" else "of fallback"
    # DRAM counters exist for the one-GPU launch configuration only
    roof["traffic"] = (DRAM_TRAFFIC.get((w.name + ("_compact" if ls.compact else ""), Ld.name))
                       if isinstance(ls, LayerStep) else None)
    roof["algorithmic_per_launch"] = {"flops": Ld.flops_fwd, "bytes": Ld.bytes_fwd}
    roof["us_per_launch"] = round(t_dom * 1e6, 2)
    return roof


def run_gpu(args, w):
    import torch
    import partial_activation_sync_gb300 as caat

    dist, rank, world, device = _setup_dist()
    peaks = _peaks()
    # one GPU: the t ranks emulated in its memory; several: the ranks spread over
    # the GPUs, with the partial channel-reduce across them (strong scaling: the
    # layer is the same whatever the GPU count)
    compact = bool(args.compact) and world == 1      # the compact outputs are a one-GPU form
    ls = LayerStep(torch, caat, w, device, compact) if world == 1 else TPStep(torch, caat, w, device, rank, world)
    clocks = ClockSampler(device.index)
    per_call, launches, clk = time_steps(torch, caat, ls, args.steps, args.warmup, device, dist, clocks)
    kernel_name = caat.last_kernel()
    total_ms, tflops = job_rate(dist, device, float(per_call.sum()), ls.flops, args.steps)
    ms_step = total_ms / args.steps
    breakdown = {n: round(float(v) / args.steps, 4) for n, v in zip(ls.names, per_call)}
    # a forward-only step on one GPU ends with its dominant call (the down-proj), so
    # the last kernel is that call's; a training step ends with a backward kernel
    # and the split step with the exchange, and their forward calls (thousands of
    # tokens) run on the tile kernel
    fwd_kernel = kernel_name if (not w.backward and world == 1) else "rowpar_fwd_tc"
    roof = roofline_of(ls, per_call, args.steps, peaks, fwd_kernel + ("" if world == 1 else " + exchange"))

    result = {
        "metric": METRIC, "value": round(tflops, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak" if world == 1 else "strong", "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations/gradients, N(0,0.02) weights)",
        "config": {"workload": w.name, "t": w.t, "N": w.N, "h": w.h,
                   "layers": {L.name: L.K for L in ls.layers}, "p": w.p,
                   "S": "contiguous" if w.layout == 0 else "random",
                   "outputs": ("compact: the S channels once [N, |S|] + each rank's other channels "
                               "[N, h - |S|]" if compact else "t full rank outputs [N, h]"),
                   "fwd_and_bwd": bool(w.backward),
                   "l2": "flushed between timed steps by reading a 2x L2 buffer (untimed)",
                   "timing": "CUDA events around each call of a step; an untimed spin kernel before "
                             "each step lets the host queue it, so the calls run back to back",
                   "parallelism": ("1 GPU, t ranks emulated" if world == 1 else
                                   "tp%d: %d ranks per GPU, partial channel-reduce across GPUs (NCCL "
                                   "all-to-all + all-gather of the S channels, fold in rank order)"
                                   % (world, w.t // world))},
        "breakdown_ms": breakdown,
        "gpu_launches": int(launches),
        "clocks": clk,
        "roofline": roof,
    }

    # end to end through the public API with host buffers (pinned), per step
    if world == 1:
        result["e2e"] = run_e2e(torch, caat, w, ls.layers, ls.sel, ls.ws, args, device, dist,
                                compact=compact, wsf=ls.wsf)
    else:
        result["e2e"] = run_e2e_tp(torch, ls, args, device, dist)
    del ls
    torch.cuda.empty_cache()

    if rank == 0 and not args.no_extras:
        result["extras"] = run_extras(torch, caat, device, peaks, args)
    if rank == 0:
        result["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    return result if rank == 0 else None


def run_e2e(torch, caat, w, layers, sel, ws, args, device, dist, compact=False, wsf=None):
    """End to end through the public API with host buffers: every step copies its
    inputs (X and the t upstream gradients of every layer) from pinned host memory
    and reads its results (dX and dW; without a backward, all t rank outputs) back.
    compact: the compact calls, whose outputs (and gradients) hold the S channels
    once: YS and the t YN[r] come back, dYS and the t dYN[r] go in.

    The copies run on their own streams and overlap the compute of the neighbouring
    steps: step i+1's inputs go in while step i computes, and step i-1's results come
    out meanwhile.  Two device buffer sets alternate, and events order every reuse.
    The timed region runs from before the first input copy to after the last read."""
    comp = torch.cuda.current_stream()
    h2d_s = torch.cuda.Stream(device=device)
    d2h_s = torch.cuda.Stream(device=device)
    hostX = [torch.from_numpy(L.X_host.view(np.int16)).pin_memory() for L in layers]
    if compact:
        # [dYS, dYN[0], ..., dYN[t-1]] per layer
        hostG = [[torch.from_numpy(a.view(np.int16)).pin_memory() for a in [L.dYS_host] + L.dYN_host]
                 if w.backward else [] for L in layers]
    else:
        hostG = [[torch.from_numpy(g.view(np.int16)).pin_memory() for g in L.G_host]
                 if w.backward else [] for L in layers]

    def dev_set(own):
        """One device buffer set per layer: the layer's own buffers, or fresh ones."""
        out = []
        for L in layers:
            # the device gradients in the order of hostG; the outputs that come back
            G = ([L.dYS] + L.dYN if w.backward else []) if compact else (L.G or [])
            Y = [L.YS] + L.YN if compact else L.Y
            if own:
                out.append({"X": L.X, "G": G, "Y": Y, "dX": L.dX, "dW": L.dW, "dWs": L.dWstore})
                continue
            dWs = torch.empty_like(L.dWstore)
            out.append({"X": torch.empty_like(L.X), "G": [torch.empty_like(g) for g in G],
                        "Y": [torch.empty_like(y) for y in Y], "dX": torch.empty_like(L.dX),
                        "dW": dWs.t(),
                        "dWs": dWs})
        return out

    sets = [dev_set(True), dev_set(False)]
    outs = [[{"dX": torch.empty(L.dX.shape, dtype=torch.int16).pin_memory(),
              "dW": torch.empty(L.dWstore.shape, dtype=torch.int16).pin_memory(),
              "Y": ([torch.empty(y.shape, dtype=torch.int16).pin_memory() for y in sets[0][li]["Y"]]
                    if not w.backward else [])} for li, L in enumerate(layers)]
            for _ in range(2)]
    h2d = sum(x.numel() * 2 for x in hostX) + sum(g.numel() * 2 for gs in hostG for g in gs)
    if w.backward:
        d2h = sum(L.dX.numel() * 2 + L.dWstore.numel() * 2 for L in layers)
    else:
        d2h = sum(y.numel() * 2 for st in sets[0] for y in st["Y"])
    in_ready = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        j = i % 2
        S, O = sets[j], outs[j]
        with torch.cuda.stream(h2d_s):
            if i >= 2:
                h2d_s.wait_event(comp_done[j])          # step i-2 is done with these inputs
            for li in range(len(layers)):
                S[li]["X"].view(torch.int16).copy_(hostX[li], non_blocking=True)
                for r in range(len(hostG[li])):
                    S[li]["G"][r].view(torch.int16).copy_(hostG[li][r], non_blocking=True)
            in_ready[j].record(h2d_s)
        comp.wait_event(in_ready[j])
        if i >= 2:
            comp.wait_event(out_done[j])                # step i-2's results have been read
        for li in range(len(layers)):
            L, B = layers[li], S[li]
            if compact:
                caat.rowpar_linear_fwd_compact(B["X"], L.W, w.t, sel, YS=B["Y"][0], YN=B["Y"][1:], workspace=wsf)
                if w.backward:
                    caat.rowpar_linear_bwd_compact(B["X"], L.W, B["G"][0], B["G"][1:], w.t, sel=sel, dX=B["dX"],
                                                   dW=B["dW"], workspace=ws)
                continue
            caat.rowpar_linear_fwd(B["X"], L.W, w.t, sel, outs=B["Y"])
            if w.backward:
                caat.rowpar_linear_bwd(B["X"], L.W, B["G"], w.t, sel, caat.CAAT_BWD_REDUCE_DOUT,
                                       dX=B["dX"], dW=B["dW"], workspace=ws)
        comp_done[j].record(comp)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(comp_done[j])
            for li in range(len(layers)):
                B = S[li]
                if w.backward:
                    O[li]["dX"].copy_(B["dX"].view(torch.int16), non_blocking=True)
                    O[li]["dW"].copy_(B["dWs"].view(torch.int16), non_blocking=True)
                else:
                    for r in range(len(B["Y"])):
                        O[li]["Y"][r].copy_(B["Y"][r].view(torch.int16), non_blocking=True)
            out_done[j].record(d2h_s)

    def run(n):
        for i in range(n):
            step(i)
        comp.wait_event(out_done[(n - 1) % 2])
        if n >= 2:
            comp.wait_event(out_done[n % 2])

    run(max(2, args.warmup))
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    h2d_s.wait_event(e0)
    d2h_s.wait_event(e0)
    run(args.steps)
    e1.record(comp)
    torch.cuda.synchronize()
    flops = sum(L.flops_fwd + L.flops_bwd for L in layers)
    ms, rate = job_rate(dist, device, e0.elapsed_time(e1), flops, args.steps)
    return {"value": round(rate, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms / args.steps, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "overlap": "inputs of step i+1 and results of step i-1 copy on two streams while step i computes"}


def run_e2e_tp(torch, ls, args, device, dist):
    """End to end for the step spread over processes: every step copies this
    process's inputs (its columns of X, its ranks' upstream gradients) in from
    pinned host memory, runs the step, and reads its results (dX and dW, or its
    ranks' outputs without a backward) back, all on one stream."""
    import types
    w = ls.w
    hostX = [torch.from_numpy(L.X_host.view(np.int16)).pin_memory() for L in ls.layers]
    hostG = [[torch.from_numpy(g.view(np.int16)).pin_memory() for g in L.G_host] if w.backward else []
             for L in ls.layers]
    outs = []
    for L in ls.layers:
        if w.backward:
            outs.append([torch.empty(L.dX.shape, dtype=torch.int16).pin_memory(),
                         torch.empty(L.dWstore.shape, dtype=torch.int16).pin_memory()])
        else:
            outs.append([torch.empty(y.shape, dtype=torch.int16).pin_memory() for y in L.Y])
    io = [types.SimpleNamespace(X=L.X, G=L.G, Y=L.Y, dX=L.dX, dW=L.dW) for L in ls.layers]

    def step():
        for li, L in enumerate(ls.layers):
            L.X.view(torch.int16).copy_(hostX[li], non_blocking=True)
            for r, g in enumerate(hostG[li]):
                L.G[r].view(torch.int16).copy_(g, non_blocking=True)
        ls.run(io=io)
        for li, L in enumerate(ls.layers):
            src = [L.dX, L.dWstore] if w.backward else L.Y
            for o, d in zip(outs[li], src):
                o.copy_(d.view(torch.int16), non_blocking=True)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    h2d = sum(x.numel() * 2 for x in hostX) + sum(g.numel() * 2 for gs in hostG for g in gs)
    d2h = sum(o.numel() * 2 for os_ in outs for o in os_)
    ms, rate = job_rate(dist, device, e0.elapsed_time(e1), ls.flops, args.steps)
    return {"value": round(rate, 3), "unit": "TFLOP/s", "ms_per_step": round(ms / args.steps, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "overlap": "none: copies in, step, copies out on one stream (per process)"}


def _time_call(torch, fn, reps, flush=None, spin=100000):
    """Median device time of fn() (CUDA events on the current stream).  Before each
    timed call the GPU gets an untimed head start (a spin kernel of `spin` cycles,
    ~50 us by default; a step of several calls takes STEP_SPIN_CYCLES) so that the
    host's launch work does not leave the GPU idle inside the timed region."""
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush.sum()
        torch.cuda._sleep(spin)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ts) * 1e-3


def _compact_step(torch, caat, w, device, flush, peaks, random_s):
    """Forward + backward of the workload's layers with compact outputs (S stored
    once; the gradient at it already summed over the ranks), p = w.p.  Returns
    TFLOP/s (6 N K h per layer) and ms per step, median of 10, L2 flushed."""
    S = caat.select_channels(w.h, w.p, caat.CAAT_S_RANDOM if random_s else caat.CAAT_S_CONTIGUOUS,
                             w.seeds()["perm"])
    ns = int(S.size)
    sel = torch.from_numpy(S).to(device) if random_s else ns
    lay = []
    for L in w.layers:
        lay.append({
            "X": torch.randn((w.N, L.K), device=device).to(torch.bfloat16),
            "W": (torch.randn((w.h, L.K), device=device) * 0.02).to(torch.bfloat16).t(),
            "YS": torch.empty((w.N, ns), dtype=torch.bfloat16, device=device),
            "YN": [torch.empty((w.N, w.h - ns), dtype=torch.bfloat16, device=device) for _ in range(w.t)],
            "dYS": torch.randn((w.N, ns), device=device).to(torch.bfloat16),
            "dYN": [torch.randn((w.N, w.h - ns), device=device).to(torch.bfloat16) for _ in range(w.t)],
            "dX": torch.empty((w.N, L.K), dtype=torch.bfloat16, device=device),
            "dW": torch.empty((w.h, L.K), dtype=torch.bfloat16, device=device).t(),
            "wsf": torch.empty(max(caat.rowpar_linear_compact_workspace(w.t, w.N, L.K, w.h, caat.CAAT_BF16,
                                                                        random_s, False), 1),
                               dtype=torch.uint8, device=device),
            "wsb": torch.empty(caat.rowpar_linear_compact_workspace(w.t, w.N, L.K, w.h, caat.CAAT_BF16,
                                                                    random_s, True),
                               dtype=torch.uint8, device=device)})

    def step():
        for d in lay:
            caat.rowpar_linear_fwd_compact(d["X"], d["W"], w.t, sel, YS=d["YS"], YN=d["YN"], workspace=d["wsf"])
            caat.rowpar_linear_bwd_compact(d["X"], d["W"], d["dYS"], d["dYN"], w.t, sel=sel, dX=d["dX"],
                                           dW=d["dW"], workspace=d["wsb"])
    step()
    sec = _time_call(torch, step, 10, flush, spin=STEP_SPIN_CYCLES)
    fl = sum(6.0 * w.N * L.K * w.h for L in w.layers)
    del lay
    torch.cuda.empty_cache()
    return {"TFLOP/s": round(fl / sec / 1e12, 1), "ms": round(sec * 1e3, 4),
            "frac_bf16": round(fl / sec / 1e12 / peaks["bf16"], 4), "S": "random" if random_s else "contiguous"}


def run_extras(torch, caat, device, peaks, args):
    """Side measurements next to the headline step: the 130M-shaped training step
    (forward and backward of both row-parallel layers) with its own roofline, the
    standalone reduce on a working set far above L2 (HBM-bound) and at the small
    fp32 configuration, Llama2-7B decode, the column-parallel layer, and the
    full 130M CAAT-Net training step in both placements of the backward reduce."""
    out = {}
    # 130M-shaped layers, forward + backward, p = 0.5 contiguous
    w130 = ci.WORKLOADS["130m"]
    ls = LayerStep(torch, caat, w130, device)
    steps130 = 10
    per_call, launches, _ = time_steps(torch, caat, ls, steps130, 3, device)
    ms = float(per_call.sum()) / steps130
    out["130m_step"] = {
        "TFLOP/s": round(ls.flops / (ms * 1e-3) / 1e12, 1), "ms": round(ms, 4),
        "frac_bf16": round(ls.flops / (ms * 1e-3) / 1e12 / peaks["bf16"], 4),
        "breakdown_ms": {n: round(float(v) / steps130, 4) for n, v in zip(ls.names, per_call)},
        "roofline_fwd": roofline_of(ls, per_call, steps130, peaks, "rowpar_fwd_tc"),
        "gpu_launches_per_step": int(launches) // steps130}
    del ls
    torch.cuda.empty_cache()
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    # standalone PCR, bf16 and fp32, t=8, [4096, 4096], p=0.5, out of place
    for dt_name, dt, es in (("bf16", torch.bfloat16, 2), ("f32", torch.float32, 4)):
        t, N, h = 8, 4096, 4096
        ins = [torch.randn((N, h), device=device).to(dt) for _ in range(t)]
        outs = [torch.empty_like(x) for x in ins]
        sel = torch.from_numpy(caat.select_channels(h, 0.5)).to(device)
        fn = lambda: caat.partial_channel_reduce(ins, sel, outs=outs)  # noqa: E731
        fn()
        sec = _time_call(torch, fn, 20, flush)
        gbs = 2.0 * t * N * h * es / sec / 1e9
        out["pcr_%s_t8_4096x4096" % dt_name] = {
            "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm"], 4),
            "us": round(sec * 1e6, 2), "kernel": caat.last_kernel()}
        del ins, outs
    # config-1 PCR (fp32, t=2, [256, 768]), L2-resident, launch-latency bound
    Y = ci.normal(1001, (2, 256, 768))
    ins = [torch.from_numpy(Y[r]).to(device) for r in range(2)]
    outs = [torch.empty_like(x) for x in ins]
    sel = torch.from_numpy(caat.select_channels(768, 0.5)).to(device)
    fn = lambda: caat.partial_channel_reduce(ins, sel, outs=outs)  # noqa: E731
    fn()
    sec = _time_call(torch, fn, 50)
    # the same call 100 times in one CUDA graph: device time per call without the
    # launch cost of each (the case is launch-latency bound)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(100):
            fn()
    graph.replay()
    sec_g = _time_call(torch, graph.replay, 20) / 100
    pcr_bytes = 2.0 * 2 * 256 * 768 * 4
    out["pcr_f32_t2_256x768"] = {"GB/s": round(pcr_bytes / sec / 1e9, 1), "us": round(sec * 1e6, 2),
                                 "graph_GB/s": round(pcr_bytes / sec_g / 1e9, 1),
                                 "graph_us": round(sec_g * 1e6, 3)}
    del graph
    # 7B prefill forward with a random S (seeded permutation), p = 0.5
    w = ci.WORKLOADS["7b_prefill"]
    S = caat.select_channels(w.h, w.p, caat.CAAT_S_RANDOM, w.seeds()["perm"])
    sel = torch.from_numpy(S).to(device)
    for li, L in enumerate(w.layers):
        X = torch.randn((w.N, L.K), device=device).to(torch.bfloat16)
        Wst = (torch.randn((w.h, L.K), device=device) * 0.02).to(torch.bfloat16)
        Ys = [torch.empty((w.N, w.h), dtype=torch.bfloat16, device=device) for _ in range(w.t)]
        fn = lambda: caat.rowpar_linear_fwd(X, Wst.t(), w.t, sel, outs=Ys)  # noqa: E731
        fn()
        sec = _time_call(torch, fn, 10, flush)
        tf = 2.0 * w.N * L.K * w.h / sec / 1e12
        out["7b_prefill_random_S_fwd_" + L.name] = {
            "TFLOP/s": round(tf, 1), "frac_bf16": round(tf / peaks["bf16"], 4),
            "us": round(sec * 1e6, 1), "kernel": caat.last_kernel()}
        del X, Wst, Ys
    # compact outputs (the S channels, the same on every rank, stored once): the 7B
    # prefill forward and the 130M layers' forward + backward, p = 0.5 contiguous
    n_sel = int(caat.select_channels(w.h, w.p).size)
    for li, L in enumerate(w.layers):
        X = torch.randn((w.N, L.K), device=device).to(torch.bfloat16)
        Wst = (torch.randn((w.h, L.K), device=device) * 0.02).to(torch.bfloat16)
        YS = torch.empty((w.N, n_sel), dtype=torch.bfloat16, device=device)
        YN = [torch.empty((w.N, w.h - n_sel), dtype=torch.bfloat16, device=device) for _ in range(w.t)]
        fn = lambda: caat.rowpar_linear_fwd_compact(X, Wst.t(), w.t, n_sel, YS=YS, YN=YN)  # noqa: E731
        fn()
        sec = _time_call(torch, fn, 10, flush)
        tf = 2.0 * w.N * L.K * w.h / sec / 1e12
        out["7b_prefill_compact_fwd_" + L.name] = {
            "TFLOP/s": round(tf, 1), "frac_bf16": round(tf / peaks["bf16"], 4), "us": round(sec * 1e6, 1),
            "MB_written": round(2.0 * w.N * (n_sel + w.t * (w.h - n_sel)) / 1e6, 1), "kernel": caat.last_kernel()}
        del X, Wst, YS, YN
    out["130m_step_compact"] = _compact_step(torch, caat, ci.WORKLOADS["130m"], device, flush, peaks, False)
    # the 1.1B layers, S contiguous and a seeded random S (index lists: W's channels
    # renamed S-first once per call, dW's rows put back)
    for rnd in (False, True):
        out["1.1b_step_compact_" + ("random_S" if rnd else "contiguous_S")] = _compact_step(
            torch, caat, ci.WORKLOADS["1.1b"], device, flush, peaks, rnd)
    # 7B decode: N in {1, 8, 64} tokens, p = 0.5, contiguous S -- weight streaming (HBM
    # bound).  Each call alone (CUDA events around one launch, so the launch latency
    # is in the time), and per call inside a CUDA graph that runs the layer for 8
    # different weight sets in turn (8 layers of a decode step: 269 / 722 MB of
    # weights, more than L2, so every call streams its weights from HBM; the launch
    # cost is paid once per graph)
    sel = torch.from_numpy(caat.select_channels(w.h, w.p, caat.CAAT_S_CONTIGUOUS)).to(device)
    nsets = 8
    for li, L in enumerate(w.layers):
        Wsets = [(torch.randn((w.h, L.K), device=device) * 0.02).to(torch.bfloat16) for _ in range(nsets)]
        Wst = Wsets[0]
        for Nd in w.decode_N:
            X = torch.randn((Nd, L.K), device=device).to(torch.bfloat16)
            Ys = [torch.empty((Nd, w.h), dtype=torch.bfloat16, device=device) for _ in range(w.t)]
            fn = lambda: caat.rowpar_linear_fwd(X, Wst.t(), w.t, sel, outs=Ys)  # noqa: E731
            fn()
            sec = _time_call(torch, fn, 10, flush)
            byt = 2.0 * (L.K * w.h + Nd * L.K + w.t * Nd * w.h)
            rec = {"GB/s": round(byt / sec / 1e9, 1), "frac_hbm": round(byt / sec / 1e9 / peaks["hbm"], 4),
                   "us": round(sec * 1e6, 1), "TFLOP/s": round(2.0 * Nd * L.K * w.h / sec / 1e12, 2),
                   "kernel": caat.last_kernel()}
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for Wk in Wsets:
                    caat.rowpar_linear_fwd(X, Wk.t(), w.t, sel, outs=Ys)
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for Wk in Wsets:
                    caat.rowpar_linear_fwd(X, Wk.t(), w.t, sel, outs=Ys)
            graph.replay()
            sec_g = _time_call(torch, graph.replay, 10, flush) / nsets
            rec.update({"graph_us": round(sec_g * 1e6, 2), "graph_GB/s": round(byt / sec_g / 1e9, 1),
                        "graph_frac_hbm": round(byt / sec_g / 1e9 / peaks["hbm"], 4)})
            # the same graph with the inference opt-in CAAT_PDL_WEIGHTS=1 (no launch
            # writes the weights, so each call may start streaming them before the
            # previous call has finished)
            prev = os.environ.get("CAAT_PDL_WEIGHTS")
            os.environ["CAAT_PDL_WEIGHTS"] = "1"
            try:
                graph_w = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph_w):
                    for Wk in Wsets:
                        caat.rowpar_linear_fwd(X, Wk.t(), w.t, sel, outs=Ys)
            finally:
                if prev is None:
                    os.environ.pop("CAAT_PDL_WEIGHTS", None)
                else:
                    os.environ["CAAT_PDL_WEIGHTS"] = prev
            graph_w.replay()
            sec_w = _time_call(torch, graph_w.replay, 10, flush) / nsets
            rec.update({"graph_static_weights_us": round(sec_w * 1e6, 2),
                        "graph_static_weights_frac_hbm": round(byt / sec_w / 1e9 / peaks["hbm"], 4)})
            out["7b_decode_N%d_%s" % (Nd, L.name)] = rec
            del X, Ys, graph, graph_w
        # a short prefill, 256 tokens, S by its size: the few-token kernel in two
        # chunks of 128 tokens against the tile kernel (CAAT_FWD_SKINNY=0), per call
        # in the graph
        Np = 256
        n_sel = int(sel.numel())
        X = torch.randn((Np, L.K), device=device).to(torch.bfloat16)
        Ys = [torch.empty((Np, w.h), dtype=torch.bfloat16, device=device) for _ in range(w.t)]
        rec = {}
        for key, env in (("", None), ("tile_kernel_", "0")):
            prev = os.environ.get("CAAT_FWD_SKINNY")
            if env is not None:
                os.environ["CAAT_FWD_SKINNY"] = env
            try:
                caat.rowpar_linear_fwd(X, Wst.t(), w.t, n_sel, outs=Ys)
                kern = caat.last_kernel()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    for Wk in Wsets:
                        caat.rowpar_linear_fwd(X, Wk.t(), w.t, n_sel, outs=Ys)
            finally:
                if prev is None:
                    os.environ.pop("CAAT_FWD_SKINNY", None)
                else:
                    os.environ["CAAT_FWD_SKINNY"] = prev
            graph.replay()
            sec_g = _time_call(torch, graph.replay, 10, flush) / nsets
            rec.update({key + "kernel": kern, key + "graph_us": round(sec_g * 1e6, 2),
                        key + "graph_TFLOP/s": round(2.0 * Np * L.K * w.h / sec_g / 1e12, 1)})
            del graph
        out["7b_prefill_N%d_%s" % (Np, L.name)] = rec
        del X, Ys
        del Wsets, Wst
    # column-parallel layer at the 130M MLP up-projection (N = 8192, h = 768,
    # FFN 3072, t = 8, p = 0.5): forward, and the backward with the partial reduce
    # on its input gradient (Megatron's placement)
    t, N, h, K = 8, 8192, 768, 3072
    A = torch.randn((t, N, h), device=device).to(torch.bfloat16)
    W1 = (torch.randn((h, K), device=device) * 0.02).to(torch.bfloat16)
    dZ = torch.randn((N, K), device=device).to(torch.bfloat16)
    Z = torch.empty((N, K), dtype=torch.bfloat16, device=device)
    dA = torch.empty((t, N, h), dtype=torch.bfloat16, device=device)
    dW1 = torch.empty_like(W1)
    ws = torch.empty(max(caat.colpar_linear_bwd_workspace(t, N, h, K, 1), 1), dtype=torch.uint8,
                     device=device)
    for name, fn, flops in (
            ("130m_colpar_up_fwd", lambda: caat.colpar_linear_fwd(A, W1, t, Z=Z), 2.0 * N * h * K),
            ("130m_colpar_up_bwd", lambda: caat.colpar_linear_bwd(A, W1, dZ, t, h // 2, dA=dA, dW1=dW1,
                                                                  workspace=ws), 4.0 * N * h * K)):
        fn()
        sec = _time_call(torch, fn, 10, flush)
        tf = flops / sec / 1e12
        out[name] = {"TFLOP/s": round(tf, 1), "frac_bf16": round(tf / peaks["bf16"], 4),
                     "us": round(sec * 1e6, 1), "kernel": caat.last_kernel()}
    del A, W1, dZ, Z, dA, dW1, ws, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    # the full 130M CAAT-Net training step (forward, backward, AdamW), both
    # placements of the backward reduce
    # (and, default placement, with a seeded random S: the layers given its index
    # list, then the same model relabelled so that S comes first)
    if not args.no_stack:
        for placement, layout, relabel in (("reduce_dout", "contiguous", False), ("column", "contiguous", False),
                                           ("reduce_dout", "random", False), ("reduce_dout", "random", True)):
            r = stack_rate(placement, steps=5, warmup=3, layout=layout, relabel=relabel)
            key = "130m_stack_" + placement + ("" if layout == "contiguous" else "_random_S")
            out[key + ("_relabelled" if relabel else "")] = {
                "tokens/s": r["value"], "ms_per_step": r["ms_per_step"],
                "gpu_launches_per_step": r["gpu_launches"] // 5, "loss_last": r["loss_last"]}
            torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------- CPU oracle arm

def _oracle_sample(w, rows, threads):
    """The oracle on `rows` token rows of every layer of the workload, fwd and
    (for training workloads) bwd.  Returns (algorithmic FLOPs, seconds)."""
    from oracle import oracle as orc
    orc.set_threads(threads)
    S = orc.select_channels(w.h, w.p, w.layout, w.seeds()["perm"])
    flops, sec = 0.0, 0.0
    for li, L in enumerate(w.layers):
        X, Wl, G = ci.layer_tensors(w, li, N=rows)
        Xd = ci.words_to_f32(ci.bf16_words(X)).astype(np.float64)
        Wd = ci.words_to_f32(ci.bf16_words(Wl)).astype(np.float64)
        t0 = time.perf_counter()
        orc.rowpar_fwd(Xd, Wd, w.t, S)
        flops += 2.0 * rows * L.K * w.h
        if w.backward:
            Gd = ci.words_to_f32(ci.bf16_words(G)).astype(np.float64)
            orc.rowpar_bwd(Xd, Wd, Gd, w.t, S, 0)
            flops += 4.0 * rows * L.K * w.h
        sec += time.perf_counter() - t0
    return flops, sec


def _calibrate_rows(w, threads, budget_s):
    """Rows of the workload the oracle processes in about budget_s seconds."""
    rows = min(w.N, 4 * max(threads, 4))
    while True:      # grow until a sample costs a quarter of the budget (cost is not linear)
        _, s = _oracle_sample(w, rows, threads)
        if s >= budget_s / 4 or rows >= w.N:
            break
        rows = int(min(w.N, rows * min(8.0, max(2.0, budget_s / 4 / max(s, 1e-3)))))
    rows = int(min(w.N, max(threads, rows * budget_s / max(s, 1e-3))))
    if rows >= threads:
        rows = rows // threads * threads     # whole rows per thread
    return max(1, min(w.N, rows))


def cpu_baseline(w, budget_s=12.0):
    from oracle import oracle as orc
    threads = os.cpu_count() or 1
    orc.set_threads(threads)
    rows2 = _calibrate_rows(w, threads, budget_s)
    f, s = _oracle_sample(w, rows2, threads)
    return {"value": round(f / s / 1e12, 6), "unit": "TFLOP/s", "cores": orc.get_threads(),
            "kind": "oracle",
            "sample": "%d of %d token rows of every layer (%s), fwd%s, float64 naive loops, %.1f s"
                      % (rows2, w.N, ",".join(L.name for L in w.layers),
                         "+bwd" if w.backward else "", s)}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    from oracle import oracle as orc
    threads = os.cpu_count() or 1
    orc.set_threads(threads)
    # a bounded sample per step so the K timed steps stay within about two minutes
    per_step_s = max(1.0, min(10.0, 120.0 / max(1, args.steps)))
    rows = _calibrate_rows(w, threads, per_step_s)
    for _ in range(args.warmup):
        _oracle_sample(w, min(rows, threads), threads)
    tot_f, tot_s = 0.0, 0.0
    for _ in range(args.steps):
        f, s = _oracle_sample(w, rows, threads)
        tot_f += f
        tot_s += s
    v = tot_f / tot_s / 1e12
    sample = "%d of %d token rows of every layer per step, float64 naive loops" % (rows, w.N)
    return {"metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_s / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "t": w.t, "N": w.N, "h": w.h, "p": w.p,
                       "layers": {L.name: L.K for L in w.layers},
                       "fwd_and_bwd": bool(w.backward)},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": orc.get_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


PCR_WORKLOADS = {"pcr_bf16_t8_4096x4096": ("bf16", 8, 4096, 4096),
                 "pcr_f32_t8_4096x4096": ("f32", 8, 4096, 4096)}


def run_pcr(args):
    """The standalone partial channel-reduce as the step: t = 8 partial tensors of
    [4096, 4096], p = 0.5 (S = the first 2048 channels, as an index list), out of
    place.  Metric: algorithmic GB/s = 2 t N h bytes per call (every input read
    once, every output written once) over its event-timed duration."""
    import torch
    import partial_activation_sync_gb300 as caat
    dist, rank, world, device = _setup_dist()
    peaks = _peaks()
    dname, t, N, h = PCR_WORKLOADS[args.workload]
    dt, es = (torch.bfloat16, 2) if dname == "bf16" else (torch.float32, 4)
    Y = [torch.from_numpy(ci.normal(5000 + r, (N, h))).to(device).to(dt) for r in range(t)]
    outs = [torch.empty_like(y) for y in Y]
    sel = torch.from_numpy(caat.select_channels(h, 0.5)).to(device)
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    for _ in range(args.warmup):
        caat.partial_channel_reduce(Y, sel, outs=outs)
        flush.sum()
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index)
    clocks.start()
    time.sleep(0.3)
    launches0 = caat.launch_count()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(100000)
        a.record(stream)
        caat.partial_channel_reduce(Y, sel, outs=outs)
        b.record(stream)
        evs.append((a, b))
        flush.sum()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    launches = caat.launch_count() - launches0
    clk = clocks.stop()
    assert caat.device_status() == 0
    ms_local = sum(a.elapsed_time(b) for a, b in evs)
    byts = 2.0 * t * N * h * es
    ms, world_n = float(ms_local), 1
    if dist is not None:
        tt = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms, world_n = float(tt.item()), dist.get_world_size()
    gbs = byts * args.steps * world_n / (ms * 1e-3) / 1e9
    per = ms / args.steps
    res = {"metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world_n,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per, 5),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dname,
           "data": "synthetic (seeded N(0,1) partial tensors)",
           "config": {"workload": args.workload, "t": t, "N": N, "h": h, "p": 0.5,
                      "S": "first 2048 channels (index list)", "in_place": False,
                      "l2": "flushed between timed steps by reading a 2x L2 buffer (untimed)"},
           "gpu_launches": int(launches), "clocks": clk,
           "roofline": {"kernel": caat.last_kernel(), "bound": "hbm",
                        "achieved": round(byts / (per * 1e-3) / 1e9, 1), "peak": peaks["hbm"],
                        "unit": "GB/s", "frac": round(byts / (per * 1e-3) / 1e9 / peaks["hbm"], 4),
                        "peak_source": "of measured (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
                        else "of fallback",
                        "traffic": DRAM_TRAFFIC.get((args.workload, "pcr")),
                        "algorithmic_per_launch": {"bytes": byts}}}
    if dist is not None:
        dist.destroy_process_group()
    return res if rank == 0 else None


STACK_METRIC = "130M CAAT-Net training step tokens/s (t=8 emulated ranks, p=0.5), 1 GPU"


def run_stack(args):
    """The full 130M block stack as the step (see stack_rate), with clocks and e2e."""
    return stack_rate(args.placement, args.steps, args.warmup, full=True, layout=args.layout or "contiguous")


def stack_rate(placement, steps, warmup, full=False, layout="contiguous", relabel=False):
    """The full 130M block stack, one training step = forward, backward, AdamW:
    12 layers, 16 heads, h = 768, FFN 3072, RoPE, sequence 1024, batch 8, t = 8
    emulated ranks, p = 0.5; token ids uniform over a 32000 vocabulary; random
    N(0, 0.02) weights.  The two row-parallel layers of every block run the fused
    kernels (with --placement column, the column-parallel layers' backward with the
    partial reduce too); attention, norms, embedding and loss are PyTorch ops.
    layout "random": S a seeded random subset (index lists in the layers);
    relabel: that model after relabel_channels (S first, passed by size)."""
    import torch
    import partial_activation_sync_gb300 as caat
    from partial_activation_sync_gb300.caatnet import CAATNet, relabel_channels, train_step
    torch.cuda.set_device(0)
    torch.manual_seed(5)
    vocab, batch, seq = 32000, 8, 1024
    model = CAATNet(vocab=vocab, h=768, heads=16, layers=12, ffn=3072, t=8, p=0.5, seq=seq,
                    placement=placement, layout=layout, seed=4003)
    model = model.cuda().to(torch.bfloat16)
    if relabel:
        model, _ = relabel_channels(model)
    opt = torch.optim.AdamW(model.parameters(), lr=6e-4, fused=True)
    rng = np.random.default_rng(5005)
    host_tok = [torch.from_numpy(rng.integers(0, vocab, (batch, seq))).pin_memory()
                for _ in range(steps + warmup)]
    tok = torch.empty((batch, seq), dtype=torch.int64, device="cuda")
    tok.copy_(host_tok[0])
    for i in range(warmup):
        train_step(model, opt, tok)
    torch.cuda.synchronize()
    launches0 = caat.launch_count()
    clocks = ClockSampler(0) if full else None
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        train_step(model, opt, tok)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    clk = clocks.stop() if clocks is not None else None
    launches = caat.launch_count() - launches0
    # end to end: each step copies its tokens in and reads the loss back
    out = torch.empty(1, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(steps):
        tok.copy_(host_tok[warmup + i], non_blocking=True)
        loss = train_step(model, opt, tok)
        out.copy_(loss.float().reshape(1), non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = f0.elapsed_time(f1)
    ntok = batch * seq
    return {"metric": STACK_METRIC, "value": round(ntok * steps / (ms * 1e-3), 1), "unit": "tokens/s",
            "n_gpus": 1, "steps": steps, "warmup": warmup,
            "ms_per_step": round(ms / steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (token ids uniform over 32000, N(0,0.02) weights)",
            "config": {"workload": "130m_stack", "layers": 12, "heads": 16, "h": 768, "ffn": 3072,
                       "seq": seq, "batch": batch, "t": 8, "p": 0.5, "optimizer": "AdamW (fused)",
                       "placement": placement, "S": layout + (" (relabelled)" if relabel else ""),
                       "l2": "working set far above L2"},
            "gpu_launches": int(launches), "clocks": clk,
            "loss_last": round(float(out.item()), 4),
            "e2e": {"value": round(ntok * steps / (ms_e2e * 1e-3), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": ntok * 8, "d2h_bytes_per_step": 4}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["caat", "reference"], default="caat")
    ap.add_argument("--workload", default="7b_prefill",
                    choices=["7b_prefill", "130m", "1.1b", "7b_decode8", "7b_prefill256", "130m_stack"]
                    + list(PCR_WORKLOADS))
    ap.add_argument("--layout", choices=["contiguous", "random"], default=None,
                    help="channel-set layout (default: the workload's own)")
    ap.add_argument("--p", type=float, default=None, help="synchronized fraction (default: workload's)")
    ap.add_argument("--compact", action="store_true",
                    help="layer workloads with compact outputs: the S channels stored once (one GPU)")
    ap.add_argument("--t", type=int, default=None, help="tensor-parallel ranks (default: the workload's 8)")
    ap.add_argument("--placement", choices=["reduce_dout", "column"], default="reduce_dout",
                    help="130m_stack: where the backward reduce sits")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-stack", action="store_true", help="leave the 130M stack out of the extras")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload == "130m_stack":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the block-stack workload has no CPU arm; "
                              "the reference arm times the layer workloads"}), flush=True)
        elif int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(run_stack(args)), flush=True)
        return
    if args.workload in PCR_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the standalone-reduce workloads have no "
                              "CPU arm; the reference arm times the layer workloads"}), flush=True)
            return
        res = run_pcr(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    w = ci.WORKLOADS[args.workload]
    if args.layout is not None or args.p is not None or args.t is not None:
        import dataclasses
        if args.t is not None and (args.t < 1 or any(L.K % args.t for L in w.layers)):
            ap.error("--t must divide every layer's K")
        w = dataclasses.replace(w, layout=(1 if args.layout == "random" else 0) if args.layout else w.layout,
                                p=args.p if args.p is not None else w.p,
                                t=args.t if args.t is not None else w.t)
    if args.impl == "reference":
        res = run_reference(args, w)
    else:
        res = run_gpu(args, w)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
