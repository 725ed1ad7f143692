"""Benchmark of the tensor-parallel block on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-rows]

Prints ONE JSON line (rank 0).  The headline step is one forward + backward of
the tensor-parallel MLP block (tp_mlp_fwd + tp_mlp_bwd) at the pages' model
width: b=2, s=2048, h=4096, h'=16384, N=2 shards, bf16 with fp32
accumulation; the metric is its throughput in TFLOP/s (12*M*h*h' algorithmic
FLOPs per step).
Inputs are synthetic and seeded (synthetic_inputs.py) and resident in HBM when
the timed region starts; L2 is flushed (a 256 MiB write) before every timed
step and the flush is outside the per-step events.

The same line carries: the roofline of the dominant kernel (per-launch CUDA
events taken by the library on the launching stream during the timed region),
the end-to-end number through the C ABI with host buffers (pinned host->device
copies of the step's inputs and device->host reads of its outputs inside the
timed region), the clocks sampled by nvidia-smi during the timed region, the
embedding gather's GB/s (the metric's second half) at top level, one short
entry per other row (the smaller MLP, attention projections, logits and tied
gradient, cross-entropy, attention core, transformer layer, Adam step), and
the fp64 CPU oracle timed on a bounded sample as a reported baseline.  The
line is kept short; every row's full per-kernel list goes to the file named
by --detail.

Multi-GPU: the block runs on one GPU; under torchrun every rank runs an
independent replica (no collective on the data path) and the line reports the
units all ranks processed over the slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
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

import synthetic_inputs as SI  # noqa: E402

METRIC = "TP-MLP fwd+bwd TFLOP/s (% BF16 peak); embed gather GB/s (% HBM)"
DEFAULT_WORKLOAD = "mlp_b2_s2048_h4096_hp16384_N2"
DEFAULT_DETAIL = os.path.join("gpurun_out", "bench_detail.json")
L2_FLUSH_BYTES = 256 << 20
SUSTAINED_AFTER_S = 1.0  # timed loops at least this long are compared with the sustained bf16 peak
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ----------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(backend):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    """Max over ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate_throughput(units_per_rank_sum: float, max_seconds: float) -> float:
    """Whole-job throughput: units all ranks processed / slowest rank's time."""
    return units_per_rank_sum / max_seconds if max_seconds > 0 else float("nan")


# ----------------------------------------------------------------------------
# measurement helpers
# ----------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# The sources that define each kind of work's kernels and launches: a DRAM
# traffic figure stays valid while these files are unchanged.
_GEMM_SRC = ("tp_gemm_tc.cu", "tp_api.cu", "tp_internal.h", "tp_device.cuh")
KERNEL_SOURCES = {"gemm": _GEMM_SRC, "embed": ("tp_embed.cu", "tp_internal.h"),
                  "ce_reduce": ("tp_embed.cu", "tp_internal.h"),
                  "attn_norm": ("tp_attn.cu", "tp_internal.h", "tp_philox.cuh"),
                  "attn_rowdot": ("tp_attn.cu", "tp_internal.h"),
                  "layer": ("tp_layer.cu", "tp_internal.h", "tp_philox.cuh"),
                  "attn_keep": ("tp_layer.cu", "tp_internal.h", "tp_philox.cuh"),
                  "adam": ("tp_opt.cu", "tp_internal.h")}


def kernel_sources(kernel: str):
    for prefix, files in KERNEL_SOURCES.items():
        if kernel.startswith(prefix):
            return files
    return None


def kernel_source_hash(kernel: str = None):
    """Hash of the sources of `kernel` (all library sources when None or unknown)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "megatron_tensor_transformer_tp_gb300", "csrc")
    files = kernel_sources(kernel) if kernel else None
    for name in sorted(files or os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when absent or taken on a different source of that kernel."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get("kernels", {}).get(f"{workload}/{kernel}")
    if rec is None:
        return None
    want = rec.get("source_hash", d.get("kernel_source_hash"))
    have = kernel_source_hash(kernel) if "source_hash" in rec else kernel_source_hash()
    if want != have:
        return None
    return rec.get("dram_bytes_per_call", rec.get("dram_bytes_per_launch"))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
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
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------
# workloads: device state, one step, algorithmic work
# ----------------------------------------------------------------------------
class MLPBench:
    kind = "mlp"

    def __init__(self, name, tp, torch):
        self.name, self.tp, self.torch = name, tp, torch
        cfg = SI.WORKLOADS[name]
        inp = SI.mlp_inputs(cfg)
        d = lambda t: t.cuda().contiguous()
        M, h, hp, N = inp["M"], inp["h"], inp["hp"], inp["N"]
        self.M, self.h, self.hp, self.N = M, h, hp, N
        bf, f = torch.bfloat16, torch.float32
        self.X, self.dOut = d(inp["X"]), d(inp["dOut"])
        self.W = [d(t) for t in inp["W_shards"]]
        self.U = [d(t) for t in inp["U_shards"]]
        self.a = [d(t) for t in inp["a_shards"]]
        self.b = d(inp["b"])
        self.Z = torch.empty(M, hp, dtype=bf, device="cuda")
        self.Y = torch.empty_like(self.Z)
        self.Out = torch.empty(M, h, dtype=bf, device="cuda")
        self.dZ = torch.empty_like(self.Z)
        self.dX = torch.empty(M, h, dtype=bf, device="cuda")
        self.dW = [torch.empty(hp // N, h, dtype=f, device="cuda") for _ in range(N)]
        self.dU = [torch.empty(h, hp // N, dtype=f, device="cuda") for _ in range(N)]
        self.da = [torch.empty(hp // N, dtype=f, device="cuda") for _ in range(N)]
        self.db = torch.empty(h, dtype=f, device="cuda")
        # pinned host buffers for the end-to-end path
        self.hX = inp["X"].pin_memory()
        self.hdOut = inp["dOut"].pin_memory()
        self.hOut = torch.empty(M, h, dtype=bf).pin_memory()
        self.hdX = torch.empty(M, h, dtype=bf).pin_memory()

    def step(self):
        self.step_on(self.X, self.dOut, self.Out, self.dX)

    def step_on(self, X, dOut, Out, dX):
        tp = self.tp
        tp.tp_mlp_fwd(X, self.W, self.a, self.U, self.b, self.Z, self.Y, Out)
        tp.tp_mlp_bwd(dOut, X, self.W, self.U, self.Z, self.Y, self.dZ, dX, self.dW,
                      self.da, self.dU, self.db)

    def e2e_run(self, steps):
        """`steps` end-to-end steps through the C ABI, each copying its own
        inputs from pinned host memory and reading its results (Out, dX) back,
        pipelined the way a training loop prefetches its next batch: two device
        buffer sets, the inputs of step i copied on one stream while step i-1
        computes, the results of step i read back on another while step i+1
        computes.  Returns device milliseconds from the first copy to the last
        read (CUDA events)."""
        torch = self.torch
        if not hasattr(self, "sets"):
            e = lambda t: torch.empty_like(t)
            self.sets = [(self.X, self.dOut, self.Out, self.dX),
                         (e(self.X), e(self.dOut), e(self.Out), e(self.dX))]
        cur = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set k are on the device
        ev_done = [torch.cuda.Event() for _ in range(2)]  # step on set k finished
        ev_read = [torch.cuda.Event() for _ in range(2)]  # results of set k are on the host
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_in.wait_stream(cur)
        t0.record(s_in)
        for i in range(steps):
            k = i % 2
            X, dOut, Out, dX = self.sets[k]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_done[k])  # step i-2 no longer reads this set's inputs
                X.copy_(self.hX, non_blocking=True)
                dOut.copy_(self.hdOut, non_blocking=True)
                ev_in[k].record(s_in)
            cur.wait_event(ev_in[k])
            cur.wait_event(ev_read[k])  # step i-2's results have left this set
            self.step_on(X, dOut, Out, dX)
            ev_done[k].record(cur)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[k])
                self.hOut.copy_(Out, non_blocking=True)
                self.hdX.copy_(dX, non_blocking=True)
                ev_read[k].record(s_out)
        cur.wait_stream(s_out)
        cur.wait_stream(s_in)
        t1.record(cur)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    def e2e_bytes(self):
        b = lambda t: t.numel() * t.element_size()
        return b(self.hX) + b(self.hdOut), b(self.hOut) + b(self.hdX)

    def units(self):
        return 12.0 * self.M * self.h * self.hp, "TFLOP/s", 1e12

    def kernel_work(self):
        # algorithmic FLOPs only: the bias column sums the backward also
        # computes on the tensor cores are not counted
        f = 2.0 * self.M * self.h * self.hp
        return {"gemm_mlp_fwd": ("tensor", 2 * f), "gemm_mlp_bwd": ("tensor", 4 * f)}


class AttnBench:
    kind = "attn"

    def __init__(self, name, tp, torch):
        self.name, self.tp, self.torch = name, tp, torch
        inp = SI.attn_inputs(SI.WORKLOADS[name])
        d = lambda t: t.cuda().contiguous()
        M, h, N = inp["M"], inp["h"], inp["N"]
        self.M, self.h, self.N, self.nh = M, h, N, inp["n_heads"]
        bf, f = torch.bfloat16, torch.float32
        self.X, self.C, self.dQKV, self.dO = d(inp["X"]), d(inp["C"]), d(inp["dQKV"]), d(inp["dO"])
        self.Wq = [d(t) for t in inp["Wqkv_shards"]]
        self.Wo = [d(t) for t in inp["Wo_shards"]]
        self.bq = [d(t) for t in inp["bqkv_shards"]]
        self.bo = d(inp["bo"])
        dd = h // N
        self.QKV = torch.empty(M, 3 * h, dtype=bf, device="cuda")
        self.O = torch.empty(M, h, dtype=bf, device="cuda")
        self.dX = torch.empty(M, h, dtype=bf, device="cuda")
        self.dC = torch.empty(M, h, dtype=bf, device="cuda")
        self.dWq = [torch.empty(3 * dd, h, dtype=f, device="cuda") for _ in range(N)]
        self.dWo = [torch.empty(h, dd, dtype=f, device="cuda") for _ in range(N)]
        self.dbq = [torch.empty(3 * dd, dtype=f, device="cuda") for _ in range(N)]
        self.dbo = torch.empty(h, dtype=f, device="cuda")

    def step(self):
        tp = self.tp
        tp.tp_attn_proj_fwd(self.X, self.Wq, self.bq, self.C, self.Wo, self.bo, self.QKV, self.O, self.nh)
        tp.tp_attn_proj_bwd(self.dQKV, self.dO, self.X, self.C, self.Wq, self.Wo, self.dX, self.dC,
                            self.dWq, self.dbq, self.dWo, self.dbo, self.nh)

    def units(self):
        return 24.0 * self.M * self.h * self.h, "TFLOP/s", 1e12

    def kernel_work(self):
        f = 8.0 * self.M * self.h * self.h
        return {"gemm_attn_fwd": ("tensor", f), "gemm_attn_bwd": ("tensor", 2 * f)}


class EmbedBench:
    """Vocab-parallel lookup, per-range logits and tied gradient."""
    kind = "embed"

    def __init__(self, name, tp, torch):
        self.name, self.tp, self.torch = name, tp, torch
        inp = SI.embed_inputs(SI.WORKLOADS[name])
        d = lambda t: t.cuda().contiguous()
        bf = torch.bfloat16
        self.T, self.V, self.h, self.N, self.rs = inp["T"], inp["V"], inp["h"], inp["N"], inp["ranges"]
        self.ids = d(inp["ids"])
        self.unique = int(torch.unique(inp["ids"]).numel())
        self.E = [d(t) for t in inp["E_shards"]]
        self.X, self.dEmb = d(inp["X"]), d(inp["dEmb"])
        self.out = torch.empty(self.T, self.h, dtype=bf, device="cuda")
        widths = [self.rs[r + 1] - self.rs[r] for r in range(self.N)]
        self.L = [torch.empty(self.T, tp.logits_pitch(w, bf), dtype=bf, device="cuda") for w in widths]
        self.dL = []
        for r, w in enumerate(widths):
            buf = torch.zeros(self.T, tp.logits_pitch(w, bf), dtype=bf, device="cuda")
            buf[:, :w] = inp["dLogits_shards"][r].cuda()
            self.dL.append(buf)
        self.dE = [torch.empty(w, self.h, dtype=torch.float32, device="cuda") for w in widths]
        self.ws = torch.empty(tp.tied_embed_grad_workspace_size(self.T, self.V), dtype=torch.uint8,
                              device="cuda")

    def gather(self):
        self.tp.vocab_parallel_embed(self.ids, self.E, self.rs, self.out)

    def step(self):
        tp = self.tp
        self.gather()
        tp.tp_vocab_logits(self.X, self.E, self.rs, self.L)
        tp.tied_embed_grad(self.ids, self.dEmb, self.X, self.dL, self.rs, self.dE, workspace=self.ws)

    def gather_bytes(self):
        # unique rows read once + every output row written + the ids
        return self.unique * self.h * 2.0 + self.T * self.h * 2.0 + self.T * 8.0

    def units(self):
        return 4.0 * self.T * self.V * self.h, "TFLOP/s", 1e12

    def kernel_work(self):
        f = 2.0 * self.T * self.V * self.h
        return {"embed_gather": ("hbm", self.gather_bytes()), "gemm_logits": ("tensor", f),
                "gemm_tied_grad_segsum": ("tensor", f),
                "embed_sort": ("hbm", self.T * 8.0 + self.T * 4.0 + (self.V + 1) * 4.0)}


class CEBench:
    """Vocab-parallel cross-entropy: forward (loss without stored logits) and
    backward (dLogits per range and the logits-side dX)."""
    kind = "ce"

    def __init__(self, name, tp, torch):
        self.name, self.tp, self.torch = name, tp, torch
        inp = SI.ce_inputs(SI.WORKLOADS[name])
        d = lambda t: t.cuda().contiguous()
        bf = torch.bfloat16
        self.T, self.V, self.h, self.N, self.rs = inp["T"], inp["V"], inp["h"], inp["N"], inp["ranges"]
        self.X, self.E = d(inp["X"]), [d(t) for t in inp["E_shards"]]
        self.targets, self.dloss = d(inp["targets"]), d(inp["dloss"])
        self.loss = torch.empty(self.T, device="cuda")
        self.lse = torch.empty(self.T, device="cuda")
        self.ws = torch.empty(tp.tp_vocab_cross_entropy_workspace_size(self.T, self.V, self.rs),
                              dtype=torch.uint8, device="cuda")
        widths = [self.rs[r + 1] - self.rs[r] for r in range(self.N)]
        self.dL = [torch.empty(self.T, tp.logits_pitch(w, bf), dtype=bf, device="cuda") for w in widths]
        self.dX = torch.empty(self.T, self.h, dtype=bf, device="cuda")
        self.parts = sum((w + 63) // 64 for w in widths)

    def step(self):
        tp = self.tp
        tp.tp_vocab_cross_entropy_fwd(self.X, self.E, self.rs, self.targets, self.loss, self.lse, self.ws)
        tp.tp_vocab_cross_entropy_bwd(self.X, self.E, self.rs, self.targets, self.lse, self.dloss,
                                      self.dL, self.dX)

    def units(self):
        # forward logits, recomputed logits, dX = sum_r dLogits_r E_r
        return 6.0 * self.T * self.V * self.h, "TFLOP/s", 1e12

    def kernel_work(self):
        f = 2.0 * self.T * self.V * self.h
        # the reduction reads every (max, sum) pair and the target logit, reads
        # the targets and writes loss and lse
        red = self.parts * self.T * 8.0 + self.T * (4.0 + 8.0 + 4.0 + 4.0)
        return {"gemm_ce_fwd": ("tensor", f), "gemm_ce_bwd": ("tensor", 2 * f), "ce_reduce": ("hbm", red)}


def attn_norm_bytes(pairs, s, causal, dropout):
    """Algorithmic bytes of one attn_norm call: the per-part statistics its rows
    merge (8 B per part), the lse it writes, the stored exponentials it reads
    (the causal part of each row) and the probabilities it writes (whole rows,
    zeros after the causal limit), plus, with dropout, the keep words of the
    causal part and the dropped probabilities."""
    parts = sum(r // 64 + 1 for r in range(s)) if causal else s * ((s + 63) // 64)
    kept = s * (s + 1) / 2.0 if causal else float(s * s)
    b = parts * 8.0 + s * 4.0 + kept * 2.0 + s * s * 2.0
    if dropout:
        b += kept / 8.0 + s * s * 2.0
    return pairs * b


class AttnCoreBench:
    """Causal attention core per head: forward (scores with per-part
    statistics and exponentials, their normalisation into P, C = P V) and
    backward (dS with dV, then dQ and dK).  The step's FLOPs are the method's:
    4 b H s^2 d forward and 8 b H s^2 d backward, times the causal fraction
    (s + 1) / 2s."""
    kind = "attn_core"

    def __init__(self, name, tp, torch):
        self.name, self.tp, self.torch = name, tp, torch
        cfg = SI.WORKLOADS[name]
        a = SI.attn_core_inputs(cfg)
        self.s, self.H, self.N, self.causal = a["s"], a["n_heads"], a["N"], cfg["causal"]
        self.T, self.h = a["T"], a["h"]
        self.b, self.d = self.T // self.s, self.h // self.H
        self.QKV, self.dC = a["QKV"].cuda(), a["dC"].cuda()
        bf = torch.bfloat16
        self.P = torch.empty(self.b, self.H, self.s, self.s, dtype=bf, device="cuda")
        self.C = torch.empty(self.T, self.h, dtype=bf, device="cuda")
        self.dQKV = torch.empty(self.T, 3 * self.h, dtype=bf, device="cuda")
        self.ws = torch.empty(tp.tp_attn_core_workspace_size(self.T, self.s, self.h, self.H),
                              dtype=torch.uint8, device="cuda")
        self.frac = (self.s + 1) / (2.0 * self.s) if self.causal else 1.0

    def step(self):
        tp = self.tp
        tp.tp_attn_core_fwd(self.QKV, self.s, self.H, self.N, self.causal, self.P, self.C, None, self.ws)
        tp.tp_attn_core_bwd(self.QKV, self.P, self.C, self.dC, self.s, self.H, self.N, self.causal,
                            self.dQKV, self.ws)

    def units(self):
        return 12.0 * self.b * self.H * self.s * self.s * self.d * self.frac, "TFLOP/s", 1e12

    def kernel_work(self):
        u = 2.0 * self.b * self.H * self.s * self.s * self.d * self.frac  # one s x s x d contraction
        rows = self.b * self.H * self.s
        return {"gemm_attn_scores": ("tensor", u), "gemm_attn_pv": ("tensor", u),
                "gemm_attn_bwd": ("tensor", 4 * u),
                "attn_norm": ("hbm", attn_norm_bytes(self.b * self.H, self.s, self.causal, False)),
                "attn_rowdot": ("hbm", 2.0 * self.T * self.h * 2 + rows * 4.0)}


class LayerBench:
    """One transformer layer, forward and backward (LayerNorm, QKV projection,
    causal attention core with attention dropout, output projection, dropout +
    residual, LayerNorm, MLP, dropout + residual).  The step's FLOPs: three
    times the forward's linear layers (8 T h^2 + 4 T h h') plus the attention
    core's 12 b H s^2 d times the causal fraction; the row kernels' work is
    counted in bytes per kernel."""
    kind = "layer"

    def __init__(self, name, tp, torch):
        self.name, self.tp, self.torch = name, tp, torch
        cfg = dict(SI.WORKLOADS[name])
        inp = SI.layer_inputs(cfg)
        self.T, self.h, self.hp, self.s = inp["T"], cfg["h"], cfg["hp"], cfg["s"]
        self.H, self.N = cfg["n_heads"], cfg["N"]
        self.b, self.d = self.T // self.s, self.h // self.H
        self.cfg = dict(cfg, T=self.T)
        d = lambda t: t.cuda().contiguous()
        self.params = dict(g1=d(inp["g1"]), b1=d(inp["b1"]), g2=d(inp["g2"]), b2=d(inp["b2"]),
                           Wqkv=[d(t) for t in inp["Wqkv"]], bqkv=[d(t) for t in inp["bqkv"]],
                           Wo=[d(t) for t in inp["Wo"]], bo=d(inp["bo"]), W=[d(t) for t in inp["W"]],
                           a=[d(t) for t in inp["a"]], U=[d(t) for t in inp["U"]], b=d(inp["b"]))
        bf, f32 = torch.bfloat16, torch.float32
        e = lambda *shape, dt=bf: torch.empty(*shape, dtype=dt, device="cuda")
        T, h, hp, H, s = self.T, self.h, self.hp, self.H, self.s
        self.saved = dict(ln1=e(T, h), mean1=e(T, dt=f32), rstd1=e(T, dt=f32), QKV=e(T, 3 * h),
                          P=e(self.b, H, s, s), Pd=e(self.b, H, s, s), C=e(T, h), h1=e(T, h),
                          ln2=e(T, h), mean2=e(T, dt=f32), rstd2=e(T, dt=f32), Z=e(T, hp), Y=e(T, hp),
                          attn_keep=e(self.b * H * s * ((s + 31) // 32), dt=torch.int32))
        N, d3, n = self.N, h // self.N, hp // self.N
        self.grads = dict(dg1=e(h, dt=f32), db1=e(h, dt=f32), dg2=e(h, dt=f32), db2=e(h, dt=f32),
                          dbo=e(h, dt=f32), db=e(h, dt=f32),
                          dWqkv=[e(3 * d3, h, dt=f32) for _ in range(N)],
                          dbqkv=[e(3 * d3, dt=f32) for _ in range(N)],
                          dWo=[e(h, d3, dt=f32) for _ in range(N)], dW=[e(n, h, dt=f32) for _ in range(N)],
                          da=[e(n, dt=f32) for _ in range(N)], dU=[e(h, n, dt=f32) for _ in range(N)])
        self.x, self.dout = d(inp["x"]), d(inp["dout"])
        self.out, self.dx = torch.empty_like(self.x), torch.empty_like(self.x)
        self.ws = torch.empty(tp.tp_transformer_layer_workspace_size(self.cfg), dtype=torch.uint8,
                              device="cuda")
        self.frac = (s + 1) / (2.0 * s) if cfg["causal"] else 1.0

    def step(self):
        tp = self.tp
        tp.tp_transformer_layer_fwd(self.cfg, self.params, self.x, self.out, self.saved, self.ws)
        tp.tp_transformer_layer_bwd(self.cfg, self.params, self.x, self.saved, self.dout, self.dx,
                                    self.grads, self.ws)

    def units(self):
        T, h, hp = self.T, self.h, self.hp
        core = 12.0 * self.b * self.H * self.s * self.s * self.d * self.frac
        return 3.0 * (8.0 * T * h * h + 4.0 * T * h * hp) + core, "TFLOP/s", 1e12

    def kernel_work(self):
        T, h, hp = self.T, self.h, self.hp
        u = 2.0 * self.b * self.H * self.s * self.s * self.d * self.frac
        rows = self.b * self.H * self.s
        th = T * h * 2.0
        return {"gemm_layer_qkv": ("tensor", 6.0 * T * h * h), "gemm_layer_oproj": ("tensor", 2.0 * T * h * h),
                "gemm_layer_oproj_bwd": ("tensor", 4.0 * T * h * h),
                "gemm_layer_qkv_bwd": ("tensor", 12.0 * T * h * h),
                "gemm_mlp_fwd": ("tensor", 4.0 * T * h * hp), "gemm_mlp_bwd": ("tensor", 8.0 * T * h * hp),
                "gemm_attn_scores": ("tensor", u), "gemm_attn_pv": ("tensor", u),
                "gemm_attn_bwd": ("tensor", 4 * u),
                "attn_norm": ("hbm", attn_norm_bytes(self.b * self.H, self.s, self.cfg["causal"],
                                                     self.cfg["p_attn"] > 0)),
                "attn_rowdot": ("hbm", 2.0 * th + rows * 4.0),
                "attn_keep": ("hbm", rows * ((self.s + 31) // 32) * 4.0),
                # per call: read x, write y (bf16) plus the row statistics
                "layer_ln": ("hbm", 2.0 * th + 8.0 * T),
                "layer_ln_bwd": ("hbm", 4.0 * th + 8.0 * T),
                # forward: read x and res, write out; backward: read dout, write dx (mean of both)
                "layer_dropout_add": ("hbm", 2.5 * th)}


class AdamBench:
    """Mixed-precision Adam step over fp32 flat groups: the norm pass reads the
    gradients (4 B per value); the update reads parameter, gradient and both
    moments and writes parameter, moments and the bf16 model copy (30 B)."""
    kind = "adam"

    def __init__(self, name, tp, torch):
        self.name, self.tp, self.torch = name, tp, torch
        inp = SI.adam_inputs(SI.WORKLOADS[name])
        self.hyper = inp["hyper"]
        self.groups = []
        for g in inp["groups"]:
            d = {k: g[k].cuda() for k in ("param", "grad", "m", "v")}
            d["model"] = torch.empty(g["param"].numel(), dtype=torch.bfloat16, device="cuda")
            d["weight_decay"] = g["weight_decay"]
            self.groups.append(d)
        self.n = sum(g["param"].numel() for g in self.groups)
        self.state = tp.make_optimizer_state(**inp["state"])
        self.ws = torch.empty(tp.tp_adam_step_workspace_size(), dtype=torch.uint8, device="cuda")

    def step(self):
        self.tp.tp_adam_step(self.groups, self.hyper, self.state, self.ws)

    def units(self):
        return 34.0 * self.n, "GB/s", 1e9

    def kernel_work(self):
        return {"adam_update": ("hbm", 30.0 * self.n), "adam_norm": ("hbm", 4.0 * self.n)}


BENCHES = {"mlp": MLPBench, "attn": AttnBench, "embed": EmbedBench, "ce": CEBench,
           "adam": AdamBench, "attn_core": AttnCoreBench, "layer": LayerBench}


def time_steps(torch, fn, steps, warmup, flush, tp=None):
    """W untimed steps, then K steps each bracketed by CUDA events on the
    current stream, with an L2 flush before every step outside the events.
    With `tp` given, each timed step is followed by one more step with the
    library's per-launch CUDA events on (they serialise the launches they
    bracket, so they stay out of the timed steps; alternating keeps both kinds
    of step at the same clocks and power).  Returns (per-step ms list of the
    timed steps, wall seconds of the loop, the profiled steps' per-kind record
    from tp_profile_read or None)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    if tp is not None:
        tp.tp_profile_reset()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for e0, e1 in ev:
        flush.fill_(1)
        e0.record()
        fn()
        e1.record()
        if tp is not None:
            flush.fill_(1)
            tp.tp_profile_enable(True)
            fn()
            tp.tp_profile_enable(False)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier()
    prof = tp.tp_profile_read() if tp is not None else None
    return [e0.elapsed_time(e1) for e0, e1 in ev], wall, prof


def roofline_for(tp, bench, prof, peaks, peak_src, sustained=True):
    """Dominant kernel (largest total device time) of the profiled region."""
    work = bench.kernel_work()
    rows = []
    for name, (calls, kernels, ms) in prof.items():
        if name not in work or calls == 0:
            continue
        bound, per_call = work[name]
        avg_s = ms / calls / 1e3
        rows.append((ms, name, bound, per_call, avg_s, calls, kernels))
    if not rows:
        return None, []
    rows.sort(reverse=True)
    out = []
    for ms, name, bound, per_call, avg_s, calls, kernels in rows:
        if bound == "tensor":
            ach, unit = per_call / avg_s / 1e12, "TFLOP/s"
            peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        else:
            ach, unit = per_call / avg_s / 1e9, "GB/s"
            peak = peaks["hbm_gbs"]
        out.append({"kernel": name, "bound": bound, "launches": calls,
                    "kernel_launches_per_call": kernels / calls, "avg_us": avg_s * 1e6,
                    "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
                    "share": ms / sum(r[0] for r in rows)})
    top = dict(out[0])
    top["traffic"] = load_traffic(top["kernel"], bench.name)
    top["peak_source"] = (f"{peak_src} {'bf16_tflops_sustained' if sustained else 'bf16_tflops'}"
                          if top["bound"] == "tensor" else f"{peak_src} hbm_gbs")
    return top, out


def workload_config(name: str, n_ranks: int) -> dict:
    """The `config` object of the JSON line: the workload's name and sizes
    (shared by both arms, so the two lines name the same workload)."""
    cfg = SI.WORKLOADS[name]
    out = {"workload": name, **{k: v for k, v in cfg.items() if k not in ("kind", "seed")},
           "parallelism": f"replicas{n_ranks}" if n_ranks > 1 else "single-gpu, N logical shards",
           "l2": "flushed before every timed step (256 MiB write)"}
    return out


def r4(x):
    """Four significant digits (keeps the printed line short)."""
    return None if x is None else float(f"{x:.4g}")


def compact_row(name, row):
    """One secondary row in the printed line: value, unit, ms per step and the
    fraction of peak of its two kernels with the most device time."""
    top = sorted(row["kernels"], key=lambda k: -k["share"])[:2]
    return {"value": r4(row["value"]), "unit": row["unit"], "ms": r4(row["ms_per_step"]),
            "frac": {k["kernel"]: r4(k["frac"]) for k in top}}


def write_detail(path, detail):
    """Full per-kernel lists of every row, written next to the run's outputs."""
    if not path:
        return None
    try:
        d = os.path.dirname(path)
        if d:
            os.makedirs(d, exist_ok=True)
        with open(path, "w") as f:
            json.dump(detail, f, indent=1)
        return path
    except OSError:
        return None


# ----------------------------------------------------------------------------
# the oracle as CPU baseline / reference arm
# ----------------------------------------------------------------------------
def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleMLP:
    """fp64 oracle forward + backward of the MLP block on the first tokens of a
    workload (same weights as the GPU arm); inputs widened once."""

    def __init__(self, workload: str, max_tokens: int):
        import torch

        import oracle.tp_oracle as O
        self.O = O
        cfg = SI.WORKLOADS[workload]
        inp = SI.mlp_inputs(cfg, M=max_tokens)
        f64 = lambda t: t.to(torch.float64).numpy()
        self.X, self.dOut = f64(inp["X"]), f64(inp["dOut"])
        self.W = [f64(t) for t in inp["W_shards"]]
        self.U = [f64(t) for t in inp["U_shards"]]
        self.a = [f64(t) for t in inp["a_shards"]]
        self.b = f64(inp["b"])
        self.h, self.hp, self.M_full = cfg["h"], cfg["hp"], cfg["b"] * cfg["s"]

    def flops(self, tokens):
        return 12.0 * tokens * self.h * self.hp

    def run(self, tokens):
        """One fwd+bwd on `tokens` tokens; returns seconds."""
        X, dO = self.X[:tokens], self.dOut[:tokens]
        t0 = time.perf_counter()
        self.O.mlp_fwd(X, self.W, self.a, self.U, self.b)
        self.O.mlp_bwd(dO, X, self.W, self.a, self.U)
        return time.perf_counter() - t0


def oracle_mlp_sample(workload: str, tokens: int, min_seconds: float, max_seconds: float):
    """The oracle repeated on `tokens` tokens for at least `min_seconds`
    (at most `max_seconds`).  Returns (TFLOP/s, seconds, repeats, tokens)."""
    orc = OracleMLP(workload, tokens)
    reps, el = 0, 0.0
    while el < min_seconds and el < max_seconds:
        el += orc.run(tokens)
        reps += 1
    return orc.flops(tokens) * reps / el / 1e12, el, reps, tokens


def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on the host cores.
    Every step is a bounded sample of the workload (the first `tokens` tokens,
    same weights), sized so the whole run stays within about two minutes."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    wl = args.workload
    cfg = SI.WORKLOADS[wl]
    if cfg["kind"] != "mlp":
        print(json.dumps({"impl": "reference", "unavailable":
                          "the reference arm times the MLP workloads only"}))
        return 0
    orc = OracleMLP(wl, 512)
    t64 = min(orc.run(64) for _ in range(2))
    budget = 120.0 / (args.steps + args.warmup)
    tokens = int(max(8, min(512, 64 * budget / max(t64, 1e-6))) // 8 * 8)
    times = []
    for i in range(args.warmup + args.steps):
        el = orc.run(tokens)
        if i >= args.warmup:
            times.append(el)
    ms = statistics.mean(times) * 1e3
    value = orc.flops(tokens) / (ms / 1e3) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded normals; no dataset)",
            "config": workload_config(wl, args.gpus),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"fp64 numpy oracle MLP fwd+bwd on {tokens} of "
                                       f"{orc.M_full} tokens per step, same weights"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------
# main arm
# ----------------------------------------------------------------------------
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # 20 timed steps (and as many profiled ones) of the headline take ~80 ms of
    # device time: short of the power cap, which longer loops of the
    # model-width MLP reach (the SM clock then drops from 2070 to ~1600 MHz)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-rows", action="store_true", help="skip the secondary rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--detail", default=DEFAULT_DETAIL,
                    help="file for every row's per-kernel list ('' to skip)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
    dist_init("nccl" if ws > 1 else "gloo")
    import megatron_tensor_transformer_tp_gb300 as tp
    tp.lib()
    peaks, peak_src = load_peaks()
    cfg = SI.WORKLOADS[args.workload]
    bench = BENCHES[cfg["kind"]](args.workload, tp, torch)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    # ---- headline: device-resident inputs ----------------------------------
    # The value: K steps, each bracketed by CUDA events, nothing between the
    # library's launches (they chain by programmatic dependent launch).  The
    # per-kernel times: K more steps, alternating with those, with the
    # library's per-launch events.
    tp.tp_profile_reset()
    for _ in range(args.warmup):
        bench.step()
    assert tp.tp_get_status() == tp.TP_OK
    sampler = ClockSampler(torch.cuda.current_device() if ws == 1 else local)
    sampler.start()
    time.sleep(0.3)
    step_ms, wall, prof = time_steps(torch, bench.step, args.steps, 0, flush, tp)
    clocks = sampler.stop()
    st = tp.tp_get_status()
    if st != tp.TP_OK:
        raise SystemExit(f"device status {tp.tp_status_string(st)}")
    units, unit, scale = bench.units()
    my_seconds = sum(step_ms) / 1e3
    max_seconds = reduce_max(my_seconds, device="cuda")
    total_units = reduce_sum(units * args.steps, device="cuda")
    value = aggregate_throughput(total_units, max_seconds) / scale
    ms_per_step = max_seconds / args.steps * 1e3
    launches = sum(k for _, k, _ in prof.values())
    # The sustained bf16 figure is for kernels timed inside a seconds-long loop
    # (the GPU then runs at its power cap); a shorter timed loop is a burst.
    sustained = max_seconds >= SUSTAINED_AFTER_S
    top, kernels = roofline_for(tp, bench, prof, peaks, peak_src, sustained=sustained)

    # ---- end to end through the C ABI with host buffers ---------------------
    e2e = None
    if hasattr(bench, "e2e_run"):
        n_e2e = max(args.steps // 4, 10)
        bench.e2e_run(3)  # warm-up
        barrier()
        e_sec = reduce_max(bench.e2e_run(n_e2e) / 1e3, device="cuda")
        e_units = reduce_sum(units * n_e2e, device="cuda")
        h2d, d2h = bench.e2e_bytes()
        e2e = {"value": aggregate_throughput(e_units, e_sec) / scale, "unit": unit,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_sec / n_e2e * 1e3,
               "how": "pinned host copies in and out every step"}

    # ---- secondary rows -----------------------------------------------------
    rows = {}
    if not args.no_rows and rank == 0:
        rows = secondary_rows(tp, torch, flush, peaks, peak_src, args.workload)

    # ---- CPU baseline: the oracle on a bounded sample ------------------------
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and cfg["kind"] == "mlp":
        tf, el, reps, tokens = oracle_mlp_sample(args.workload, 256, 10.0, 30.0)
        cpu = {"value": r4(tf), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"fp64 oracle fwd+bwd, {tokens} of {bench.M} tokens, same weights, "
                         f"{reps}x in {el:.1f} s"}

    if rank != 0:
        return 0
    gather = rows.pop("embed_gather", None) if rows else None
    detail = {"headline": {"workload": args.workload, "kernels": kernels},
              "embed_gather": gather, "rows": rows}
    detail_path = write_detail(args.detail, detail)
    line = {
        "metric": METRIC, "value": r4(value), "unit": unit, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r4(ms_per_step), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg.get("dtype", "bf16"),
        "data": "synthetic (seeded normals; no dataset)",
        "config": workload_config(args.workload, ws),
        "work_per_step": units,
        "roofline": None if top is None else {
            "bound": top["bound"], "achieved": r4(top["achieved"]), "peak": top["peak"],
            "unit": top["unit"], "frac": r4(top["frac"]), "traffic": top["traffic"],
            "kernel": top["kernel"], "peak_source": top["peak_source"],
            "avg_launch_us": r4(top["avg_us"]), "launches": top["launches"],
            "launches_per_call": r4(top["kernel_launches_per_call"])},
        "kernels_frac": {k["kernel"]: r4(k["frac"]) for k in kernels},
        "embed_gather": None if gather is None else {
            "value": r4(gather["value"]), "unit": "GB/s", "frac": r4(gather["frac"]),
            "peak": gather["peak"], "avg_launch_us": r4(gather["avg_launch_us"]),
            "traffic": gather["traffic"], "workload": gather["workload"]},
        "rows": {k: compact_row(k, v) for k, v in rows.items()},
        "cpu_baseline": cpu,
        "e2e": None if e2e is None else dict(e2e, value=r4(e2e["value"]),
                                             ms_per_step=r4(e2e["ms_per_step"])),
        "gpu_launches": launches,
        "clocks": clocks,
        "detail": detail_path,
    }
    print(json.dumps(line))
    return 0


def gather_row(tp, torch, b, name, peaks, peak_src, sets=4, per_graph=16, replays=20):
    """The vocab-parallel gather alone, HBM-bound.  A 19 us kernel is shorter
    than the host's per-call cost, so per-call events would time the host.
    Instead `per_graph` gathers are captured in one CUDA graph and replayed,
    with CUDA events on the replaying stream around each replay.  The gathers
    cycle through `sets` independent seeded id sets and output buffers: each
    set's unique rows (~62 MB) and output (67 MB) are reused only after the
    other sets have moved ~390 MB, more than the 129 MB L2, so no flush is
    needed between gathers."""
    ids = [b.ids] + [SI.uniform_ids(SI.WORKLOADS[name]["seed"], 100 + k, b.T, b.V).cuda()
                     for k in range(1, sets)]
    outs = [torch.empty_like(b.out) for _ in range(sets)]
    uniq = [int(torch.unique(x).numel()) for x in ids]
    bytes_per = statistics.mean(u * b.h * 2.0 + b.T * b.h * 2.0 + b.T * 8.0 for u in uniq)
    tp.tp_profile_enable(False)
    for k in range(sets):
        tp.vocab_parallel_embed(ids[k], b.E, b.rs, outs[k])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for j in range(per_graph):
            tp.vocab_parallel_embed(ids[j % sets], b.E, b.rs, outs[j % sets])
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(replays)]
    for e0, e1 in ev:
        e0.record()
        graph.replay()
        e1.record()
    torch.cuda.synchronize()
    avg = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) / per_graph / 1e3
    gbs = bytes_per / avg / 1e9
    return {"workload": name, "value": gbs, "unit": "GB/s", "bound": "hbm", "achieved": gbs,
            "peak": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"],
            "peak_source": f"{peak_src} hbm_gbs", "avg_launch_us": avg * 1e6,
            "bytes_per_launch": bytes_per, "unique_rows": statistics.mean(uniq),
            "timing": f"CUDA graph of {per_graph} gathers over {sets} rotating id/output sets, "
                      f"{replays} replays, events on the replaying stream",
            "traffic": load_traffic("embed_gather", name)}


def secondary_rows(tp, torch, flush, peaks, peak_src, main_workload):
    """The other rows of the block, each on its own workload, a few timed steps."""
    rows = {}
    for name in ("mlp_b4_s1024_h1024_hp4096_N4", "mlp_b2_s2048_h4096_hp16384_N2",
                 "embed_tied_V50257_h4096_T8192", "ce_V50257_h4096_T8192",
                 "attn_b1_s2048_h4096_heads8_N8",
                 "attn_core_b1_s2048_heads8_d512_causal", "layer_b1_s2048_h4096_heads8_hp16384_N8",
                 "adam_layer_H4096"):
        if name == main_workload:
            continue
        cfg = SI.WORKLOADS[name]
        b = BENCHES[cfg["kind"]](name, tp, torch)
        if cfg["kind"] == "embed":
            rows["embed_gather"] = gather_row(tp, torch, b, name, peaks, peak_src)
        s_ms, _, prof = time_steps(torch, b.step, 20, 5, flush, tp)
        units, unit, scale = b.units()
        top, kernels = roofline_for(tp, b, prof, peaks, peak_src,
                                    sustained=sum(s_ms) / 1e3 >= SUSTAINED_AFTER_S)
        rows[name] = {"value": units / (statistics.mean(s_ms) / 1e3) / scale, "unit": unit,
                      "ms_per_step": statistics.mean(s_ms), "kernels": kernels}
        del b
        torch.cuda.empty_cache()
    assert tp.tp_get_status() == tp.TP_OK
    return rows


if __name__ == "__main__":
    sys.exit(main())
