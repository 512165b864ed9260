#!/usr/bin/env python
"""Benchmark of the quantized linear layer's hot path on one Llama-shaped block.

One step = the whole path over the seven linears Q, K, V, O, Gate, Up, Down of
one block (SNIP, Figure 4) under a per-layer FP8/NVFP4 plan: for every linear
the forward quantizations (X, W along K, round-to-nearest) and GEMM Y = X W^T,
the backward quantizations (dY and W^T along N, dY^T and X^T along T,
stochastic rounding) and GEMMs dX = dY W, dW = dY^T X (SNIP, Figure 5), and the
statistics pass over X, W and dY.  value = 6*T*K*N summed over the linears per
step / step time (TFLOP/s), with all inputs resident in HBM.

Default workload: the Llama-7B block (T = 8192 tokens, hidden 4096,
intermediate 11008), the seeded plan closest to 80% FP4 FLOPs.  The inputs of
one step (1.5 GB bf16) exceed the 129 MB L2, so no flush is needed between
steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs its own replica (weak scaling, no collective on
the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "qlinear fwd+bwd TFLOP/s (NVFP4/FP8 mix) & quantizer GB/s, % of GB300 roofline"
UNIT = "TFLOP/s"
SCALES_BYTES_PER_ELEM = 2                        # amax pass: read
NVFP4_BYTES_PER_ELEM = 2 + 0.5 + 1 / 16          # read + codes + block scales
MXFP4_BYTES_PER_ELEM = 2 + 0.5 + 1 / 32          # read + codes + E8M0 block scales
FP8_BYTES_PER_ELEM = 2 + 1                       # read + codes
STATS_BYTES_PER_ELEM = 2                         # read
FP4_OVER_BF16, FP8_OVER_BF16 = 13.5 / 2.25, 4.5 / 2.25   # nominal dense ratios


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="llama-7b-block")
    ap.add_argument("--plan", default="mix",
                    choices=["mix", "nvfp4", "fp8", "mxfp4", "nvfp4-b32", "nvfp4-b64", "nvfp4-b128", "snip"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="issue the step's calls one by one instead of replaying them as a captured CUDA graph")
    ap.add_argument("--no-overlap", action="store_true",
                    help="run every call on one stream (no quantization beside the GEMMs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--vs-cublaslt", action="store_true",
                    help="instead of the step: the library's NVFP4 and FP8 GEMMs against cuBLASLt's on the "
                         "block's shapes (builds cublaslt_gemm.cu), one JSON line")
    ap.add_argument("--profile-run", action="store_true",
                    help="exactly --warmup untimed steps, no clock settle, e2e or CPU baseline (for ncu)")
    ap.add_argument("--scales-per-launch", type=int, default=5,
                    help="most tensors whose scales one launch computes, whole linears packed in order "
                         "(3 or less: one launch per linear)")
    ap.add_argument("--gemm-streams", type=int, default=3, choices=[1, 2, 3],
                    help="GEMM streams of the overlapped step: 1; 2, linears alternating; 3 (default), one per "
                         "GEMM kind")
    ap.add_argument("--no-scales-stream", action="store_true",
                    help="tensor-scale passes on the quantization stream (default: a stream of their own, "
                         "two linears ahead)")
    ap.add_argument("--scales-lead", type=int, default=2,
                    help="a linear's scale pass starts after the quantizations this many linears back")
    ap.add_argument("--order", default="",
                    help="comma-separated order in which the step runs its linears (default: the model's)")
    ap.add_argument("--layers", default="", help="comma-separated subset of Q,K,V,O,Gate,Up,Down (profiling)")
    ap.add_argument("--next4-only", action="store_true",
                    help="only the dW-level check (bf16 GEMM with fused norms) at the 7B Down shape, one JSON line")
    ap.add_argument("--cpu-sample-only", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-sample-seconds", type=float, default=10.0, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- workload description

# plan format names <-> the library's format codes (the same as inputs.FMT_*)
FORMAT_OF_NAME = {"fp8": 0, "nvfp4": 1, "mxfp4": 2, "nvfp4-b32": 5, "nvfp4-b64": 6, "nvfp4-b128": 7}
NAME_OF_FORMAT = {v: k for k, v in FORMAT_OF_NAME.items()}


def workload(args):
    from sub_byte_mixed_gb300 import inputs
    cfg = inputs.BLOCKS[args.config]
    if args.plan in ("mix", "snip"):
        # "snip" starts from the seeded plan; run_ours replaces it with SNIP's selection
        plan = inputs.seeded_plan(cfg, cfg.fp4_target, seed=0)
    else:
        plan = inputs.all_plan(FORMAT_OF_NAME[args.plan])
    return cfg, plan


def linear_order(args):
    return [n for n in args.order.split(",") if n] or None


def config_json(cfg, plan, args):
    from sub_byte_mixed_gb300 import inputs
    return {
        "workload": f"{cfg.name}: T={cfg.T} hidden={cfg.hidden} inter={cfg.inter} kv_out={cfg.kv_out}; "
                    f"7 linears fwd+dgrad+wgrad+stats",
        "plan": {n: NAME_OF_FORMAT[f] for n, f in zip(inputs.LAYER_NAMES, plan)},
        "fp4_flop_fraction": round(cfg.fp4_flop_fraction(plan), 4),
        "flop_per_step": cfg.flops_fwd_bwd(),
        "l2": "inputs larger than L2 (no flush)",
        "rounding": "RTN forward, SR (Philox4x32-10, 16 bits/elem) backward",
        "stats": "SNIP statistics of X, W (forward rounding) and dY (dgrad rounding) fused into their row-block quantizations",
        "schedule": ("one stream" if args.no_overlap else
                     "quantizations on one stream, GEMMs on others: a linear's quantizations run beside the "
                     "previous linear's GEMMs (events order every GEMM after its operands)")
                    + ("; the step captured once as a CUDA graph and replayed" if not args.no_graph else "")
                    + (f"; tensor scales of whole linears packed into launches of up to {args.scales_per_launch} "
                       "tensors (the first linear's alone)" if args.scales_per_launch > 3
                       else "; one tensor-scale launch per linear")
                    + (f"; linears run in the order {args.order}" if args.order else "")
                    + ("" if args.no_overlap else
                       f"; GEMMs on {args.gemm_streams} stream{'s' if args.gemm_streams > 1 else ''}"
                       + (" (forward, dgrad, wgrad each on its own)" if args.gemm_streams == 3 else "")
                       + ("" if args.no_scales_stream else
                          "; tensor-scale passes on a stream of their own, each after the quantizations two "
                          "linears back")),
        "plan_source": ("SNIP selection from one step's statistics (snip_plan_select, FP4-FLOP target "
                        f"{cfg.fp4_target})") if args.plan == "snip" else
                       ("seeded plan at the FP4-FLOP target" if args.plan == "mix" else "uniform"),
    }


# ----------------------------------------------------------------------------- CPU baseline (oracle)

# The bounded sample: the Q linear of the 7B block (K = N = 4096) restricted to 256 tokens and 512
# output features, forward + dgrad + wgrad in NVFP4 plus the statistics of X, W and dY.
SAMPLE_T, SAMPLE_K, SAMPLE_N = 256, 4096, 512
SAMPLE_FLOPS = 6 * SAMPLE_T * SAMPLE_K * SAMPLE_N
SAMPLE_TEXT = "Q linear of the 7B block cut to T=256, N=512 (K=4096), NVFP4 fwd+dgrad+wgrad+stats"
_worker = {}


def _oracle_worker_init():
    """Pool worker (spawned, one thread of BLAS): the oracle and the sample's inputs, once."""
    import oracle
    from sub_byte_mixed_gb300 import inputs
    oracle.build()
    _worker["linear"] = inputs.single_linear_inputs(SAMPLE_T, SAMPLE_K, SAMPLE_N, seed=0)


def _oracle_sample_rep(_=None) -> float:
    """One repetition of the bounded sample in this worker; returns its seconds."""
    import oracle
    X, W, dY = _worker["linear"]
    t0 = time.perf_counter()
    oracle.qlinear_fwd("nvfp4", X, W)
    oracle.qlinear_dgrad("nvfp4", dY, W)
    oracle.qlinear_wgrad("nvfp4", dY, X)
    for t, r in ((X, 0), (W, 0), (dY, 1)):
        oracle.quant_stats(t, rnd=r, seed=0, stream_id=2)
    return time.perf_counter() - t0


def _oracle_quant_rows(args) -> float:
    """NVFP4 row-block quantization (round to nearest) and SNIP's statistics of rows [r0, r1) of the
    7B block's Q-linear activation X (8192 x 4096) under the whole tensor's scales; returns seconds."""
    import oracle
    from sub_byte_mixed_gb300 import inputs
    r0, r1, g, s8 = args
    if "x" not in _worker:
        _worker["x"] = oracle._bits(inputs.linear_inputs(inputs.LLAMA7B, 0, seed=0)[0])
    part = _worker["x"][r0:r1]
    t0 = time.perf_counter()
    oracle.quantize_nvfp4(part, 0, 0, 0, 0, g_in=g)
    oracle.quant_stats(part, rnd=0, seed=0, stream_id=0, g_in=g, s_in=s8, index_base=r0 * part.shape[1])
    return time.perf_counter() - t0


def oracle_pool(n: int):
    """n spawned worker processes for the oracle (spawn: safe in a process that may hold a CUDA context)."""
    import multiprocessing as mp
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    os.environ["CUDA_VISIBLE_DEVICES"] = ""
    return mp.get_context("spawn").Pool(n, initializer=_oracle_worker_init)


def cpu_sample(seconds: float):
    """The oracle on every host core: one spawned worker per core, each repeating the bounded sample
    until `seconds` have passed, their flops summed over the wall time; then the quantizer and
    statistics on the full X of the same linear (8192 x 4096), its rows split over the workers."""
    import oracle
    from sub_byte_mixed_gb300 import inputs
    n = os.cpu_count() or 1
    with oracle_pool(n) as pool:
        pool.map(_oracle_sample_rep, range(n))            # first use: page in, build caches
        reps, t0 = 0, time.perf_counter()
        while True:
            pool.map(_oracle_sample_rep, range(n))
            reps += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
        # full-tensor quantizer + statistics, whole-tensor scales from the oracle's own amax
        oracle.build()
        X = inputs.linear_inputs(inputs.LLAMA7B, 0, seed=0)[0]
        am = oracle.amax(X)
        g, s8 = oracle.nvfp4_global_scale(am), oracle.fp8_tensor_scale(am)
        R, C = X.shape
        step = (R + n - 1) // n
        parts = [(r0, min(R, r0 + step), g, s8) for r0 in range(0, R, step)]
        pool.map(_oracle_quant_rows, [(0, 1, g, s8)] * n)  # each worker generates X once
        tq = time.perf_counter()
        pool.map(_oracle_quant_rows, parts)
        tq = time.perf_counter() - tq
    return {"value": SAMPLE_FLOPS * n * reps / el / 1e12, "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"{SAMPLE_TEXT}; {n} worker processes (one per host core, one BLAS thread each) "
                      f"repeating it, {n * reps} repetitions in {el:.1f} s",
            "quantizer": {"value": (2 + 0.5 + 1 / 16) * R * C / tq / 1e9, "unit": "GB/s",
                          "sample": f"NVFP4 row-block RTN quantization + SNIP statistics of the full 7B Q-linear X "
                                    f"({R}x{C} bf16), rows split over {n} workers, {tq:.2f} s; bytes counted "
                                    f"as the GPU quantizer's (read + codes + scales)"}}


def run_cpu_baseline_subprocess(seconds: float):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-sample-only",
                        "--cpu-sample-seconds", str(seconds)], capture_output=True, text=True, env=env)
    for line in r.stdout.splitlines()[::-1]:
        if line.startswith("{"):
            return json.loads(line)
    return {"value": None, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": "failed: " + r.stderr[-300:]}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []   # (host time, sm, max, power, reasons dict)
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, mx, pw = float(parts[0]), float(parts[1]), float(parts[2])
            except ValueError:
                continue
            names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
            reasons = [n for n, v in zip(names, parts[4:8]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, mx, pw, reasons))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        use = inside or [s for s in self.samples if s[0] >= t0 - 2.0] or self.samples
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sms = sorted(s[1] for s in use)
        reasons = sorted({r for s in use for r in s[4]})
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(s[2] for s in use), "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside),
                "power_w_max": max(s[3] for s in use)}


# ----------------------------------------------------------------------------- peaks and ncu traffic

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash(kind: str) -> str:
    """Hash of the code (comments and whitespace removed) of a kernel category's sources: a traffic
    figure measured on one build applies while that code is unchanged."""
    files = {"gemm": ["gemm.cu", "snip_device.cuh", "snip_kernels.cuh", "snip_quant.cuh"],
             "quant": ["quant.cu", "snip_device.cuh", "snip_kernels.cuh", "snip_quant.cuh"]}[kind]
    h = hashlib.sha256()
    for f in files:
        text = open(os.path.join(ROOT, "sub_byte_mixed_gb300", "csrc", f)).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(category: str):
    """DRAM bytes per unit of algorithmic work (per FLOP for a GEMM, per
    algorithmic byte for a quantizer) recorded in profiles/traffic.md for
    this kernel category, valid only while the kernel sources are unchanged
    since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    kind = "gemm" if category.startswith("gemm") else "quant"
    want = kernel_source_hash(kind)
    for line in open(path):
        m = re.match(r"\|\s*(\S+)\s*\|\s*(\S+)\s*\|\s*([0-9.eE+-]+)\s*\|", line)
        if m and m.group(1) == category and m.group(2) == want:
            return float(m.group(3))
    return None


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(ms: float, world: int, device: str) -> float:
    """The slowest rank's time per step (every rank gets it)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_tflops(world: int, flops_per_rank: float, ms: float) -> float:
    """Replicas: every rank runs the whole step on its own block, so the job
    does world x the flops of one step in the slowest rank's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------- our arm

class Step:
    """Pre-marshalled C-ABI calls of one step (ctypes function + fixed args)."""

    def __init__(self, cfg, plan, snip, device, layers=None, overlap=True, stats=True, own_stream=False,
                 share_x=True, scales_per_launch=5, order=None, gemm_streams=3, scales_stream=True,
                 scales_lead=2):
        import torch
        from sub_byte_mixed_gb300 import inputs
        self.cfg, self.plan, self.snip = cfg, plan, snip
        # overlap: quantizations on one stream, GEMMs on others, so that a linear's quantizations run
        # beside the previous linear's GEMMs; operand buffers alternate between two sets by position
        self.overlap = overlap
        # own_stream: the quantization stream is a stream of its own (a graph cannot be captured on
        # the default stream); run() then joins the caller's stream at both ends
        self.sQ = torch.cuda.Stream() if own_stream else torch.cuda.current_stream()
        # gemm_streams: 1, one GEMM stream; 2, the linears' GEMMs alternate between two streams; 3, the
        # forward, dgrad and wgrad GEMMs each on a stream of their own (a GEMM's last wave can then
        # overlap the next GEMM, which reads other operands and writes another output)
        self.gemm_streams = gemm_streams if overlap else 1
        self.sGs = [torch.cuda.Stream() for _ in range(self.gemm_streams)] if overlap else [self.sQ]
        # scales_stream: the tensor-scale passes on a stream of their own, each started once the
        # quantizations scales_lead positions back are done, so that it can run beside the GEMMs
        # (which leave registers and bandwidth to spare on their SMs) instead of on the quantization
        # stream
        self.sS = torch.cuda.Stream() if overlap and scales_stream else None
        self.scales_lead = scales_lead   # the pass of position p waits for the quantizations of p - scales_lead
        self.graph = None
        nsets = 2 if overlap else 1
        L = snip.load()
        self.inp = inputs.block_inputs(cfg, seed=0, device=device)
        T = cfg.T
        self.Y = [torch.empty((T, l.N), dtype=torch.float32, device=device) for l in cfg.linears]
        self.dX = [torch.empty((T, l.K), dtype=torch.float32, device=device) for l in cfg.linears]
        self.dW = [torch.empty((l.N, l.K), dtype=torch.float32, device=device) for l in cfg.linears]
        self.raw = torch.zeros((len(cfg.linears), 3, snip.STATS_NVALS), dtype=torch.float64, device=device)
        self.ws = snip.Workspace(snip.snip_quantize_workspace_size(0, 0), device)
        # {amax, NVFP4 g, FP8 s} of X, W and dY of every linear (16-byte slots)
        self.sc = torch.empty((len(cfg.linears), 3, 4), dtype=torch.float32, device=device)
        # operand roles: (source, orient, out_rows, out_cols) per linear; buffers sized for the largest
        roles = lambda l: [(l.x_id, 0, T, l.K), ("W", 0, l.N, l.K), ("dY", 0, T, l.N), ("W", 1, l.K, l.N),
                           ("dY", 1, l.N, T), (l.x_id, 1, l.K, T)]
        csz = [0] * 6
        ssz = [0] * 6
        for l, f in zip(cfg.linears, plan):
            for r, (_, _, orr, occ) in enumerate(roles(l)):
                c, s = snip.snip_quantized_bytes(f, snip.MMA, orr, occ)
                csz[r], ssz[r] = max(csz[r], c), max(ssz[r], s)
        codes_sets = [[torch.empty(c, dtype=torch.uint8, device=device) for c in csz] for _ in range(nsets)]
        scales_sets = [[torch.empty(max(s, 16), dtype=torch.uint8, device=device) for s in ssz] for _ in range(nsets)]
        ws, wsb, stream = self.ws.ptr, self.ws.nbytes, self.sQ.cuda_stream
        self.stream = stream
        calls = []   # (fn, args, category, units, stream kind 'q'/'g', position, GEMM index or -1)
        self.gsel = {}   # call index of a GEMM -> its GEMM stream
        self.gemm_wss = ([snip.Workspace(snip.WS_HEADER_BYTES, device) for _ in self.sGs] if overlap
                         else [self.ws])
        self.ws_s = snip.Workspace(snip.snip_quantize_workspace_size(0, 0), device) if self.sS is not None else None
        self.scale_call = {}   # call index of a scale pass -> its arguments on the scales stream
        self._keep = []   # ctypes arrays referenced by the calls
        # Activations read by several linears (Q/K/V, Gate/Up: SNIP, Figure 4): with share_x, their
        # tensor scales, statistics and round-to-nearest row-block quantization (forward operand) are
        # computed once -- the quantization once per format -- into a buffer of their own, read by
        # every sharer's forward GEMM.  The per-linear column-block (stochastic, own stream id)
        # quantizations of X are unchanged.
        active = [j for j, l in enumerate(cfg.linears) if not layers or l.name in layers]
        # the linears are independent here, so the step may run them in any order (order: their
        # names, first to last); buffer sets and stream waits go by position in that order, the
        # random streams and outputs by linear
        if order:
            rank = {n: i for i, n in enumerate(order)}
            missing = [cfg.linears[j].name for j in active if cfg.linears[j].name not in rank]
            if missing:
                raise ValueError(f"order leaves out {missing}")
            active.sort(key=lambda j: rank[cfg.linears[j].name])
        pos_of = {j: p for p, j in enumerate(active)}
        self.order = [cfg.linears[j].name for j in active]
        users = {}
        for j in active:
            users.setdefault(cfg.linears[j].x_id, []).append(j)
        self.share_x = share_x
        shared_ids = {k for k, v in users.items() if len(v) > 1} if share_x else set()
        self.first_user = {k: v[0] for k, v in users.items()}
        xq_owner = {}       # (x_id, format) -> (codes, scales) holding that row-block quantization
        xbuf = {}           # (activation, format) -> (codes, scales, position of its last user)
        # The tensor-scale passes: the first linear's alone (the first GEMM waits for it), then whole
        # linears packed in order into launches of at most scales_per_launch tensors (one launch per
        # linear when that is below 3).  An activation shared by several linears is read once, by
        # its first user.
        scale_items = {}
        for j in active:
            l = cfg.linears[j]
            src = {l.x_id: self.inp.X[l.x_id], "W": self.inp.W[j], "dY": self.inp.dY[j]}
            slot = {l.x_id: 0, "W": 1, "dY": 2}
            sharer = l.x_id in shared_ids and self.first_user[l.x_id] != j
            names = ("W", "dY") if sharer else (l.x_id, "W", "dY")
            scale_items[j] = [(src[nm], self.sc[j, slot[nm]].data_ptr()) for nm in names]
        scale_groups, cur_g = [], []
        for j in active:
            fits = sum(len(scale_items[i]) for i in cur_g) + len(scale_items[j]) <= max(scales_per_launch, 3)
            if cur_g and (not fits or cur_g[0] == active[0]):
                scale_groups.append(cur_g)
                cur_g = []
            cur_g.append(j)
        if cur_g:
            scale_groups.append(cur_g)
        group_of = {g[0]: g for g in scale_groups}
        self.scale_launches = len(scale_groups)
        self.wait_at = {}   # call index -> linear whose operand buffers that call (its first quantization) writes
        for j in active:
            p = pos_of[j]
            l, f = cfg.linears[j], plan[j]
            X = self.inp.X[l.x_id]
            W, dY = self.inp.W[j], self.inp.dY[j]
            self.codes, self.scales = codes_sets[p % nsets], scales_sets[p % nsets]
            src = {l.x_id: X, "W": W, "dY": dY}
            scp = {l.x_id: self.sc[j, 0].data_ptr(), "W": self.sc[j, 1].data_ptr(), "dY": self.sc[j, 2].data_ptr()}
            sid = 8 * j
            rnd = [0, 0, 1, 1, 1, 1]
            block = snip.NVFP4_BLOCK.get(f, 0)      # NVFP4 and its longer blocks: NVFP4's kernels
            fname = "nvfp4" if block else {snip.FP8: "fp8", snip.MXFP4: "mxfp4"}[f]
            qcat, gcat = "quant_" + fname, "gemm_" + fname
            bpe = NVFP4_BYTES_PER_ELEM if block else {snip.FP8: FP8_BYTES_PER_ELEM, snip.MXFP4: MXFP4_BYTES_PER_ELEM}[f]
            fo = 8 if f == snip.FP8 else 4            # byte offset of s (FP8) or g (NVFP4; MXFP4: unused) in a slot
            shared = l.x_id in shared_ids
            sharer = shared and self.first_user[l.x_id] != j
            if sharer:   # X's tensor scales are the first user's
                scp[l.x_id] = self.sc[self.first_user[l.x_id], 0].data_ptr()
            # the scales of this linear's group of linears in one launch
            if j in group_of:
                items = [it for i in group_of[j] for it in scale_items[i]]
                xs = (ctypes.c_void_p * len(items))(*[t.data_ptr() for t, _ in items])
                ns = (ctypes.c_int64 * len(items))(*[t.numel() for t, _ in items])
                outs = (ctypes.c_void_p * len(items))(*[o for _, o in items])
                self._keep.append((xs, ns, outs))
                if self.sS is not None:
                    self.scale_call[len(calls)] = (len(items), xs, ns, outs, self.ws_s.ptr, self.ws_s.nbytes,
                                                   self.sS.cuda_stream)
                calls.append((L.snip_tensor_scales_multi, (len(items), xs, ns, outs, ws, wsb, stream), "scales",
                              SCALES_BYTES_PER_ELEM * sum(t.numel() for t, _ in items), "q", p, -1))
            self.wait_at[len(calls)] = p
            xcodes = xscales = None      # forward operand of X when it comes from the shared buffers
            for r, (name, orient, orr, occ) in enumerate(roles(l)):
                t = src[name]
                rows, cols = t.shape
                g = scp[name] + fo
                if r == 0 and shared:
                    key = (l.x_id, f)
                    if key in xq_owner:          # another sharer already quantized X in this format
                        xcodes, xscales = xq_owner[key]
                        continue
                    c, sbytes = snip.snip_quantized_bytes(f, snip.MMA, orr, occ)
                    if key not in xbuf:
                        xbuf[key] = (torch.empty(c, dtype=torch.uint8, device=device),
                                     torch.empty(max(sbytes, 16), dtype=torch.uint8, device=device), None)
                    xc, xsb, last = xbuf[key]
                    # a previous content of the buffer is read by earlier forward GEMMs; this linear's
                    # quantizations wait for the GEMMs two positions back, which must cover them
                    if last is not None and last > p - 2:
                        raise RuntimeError("shared activations too close together for the two-set schedule")
                    xbuf[key] = (xc, xsb, max(pos_of[u] for u in users[l.x_id]))
                    xq_owner[key] = (xc, xsb)
                    xcodes, xscales = xc, xsb
                    dst_c, dst_s = xc.data_ptr(), xsb.data_ptr()
                    if stats and not sharer:
                        args = (f, t.data_ptr(), rows, cols, rnd[r], 0, sid + r, scp[name], snip.MMA, dst_c,
                                dst_s if f != snip.FP8 else None, self.raw[j, 0].data_ptr(), ws, wsb, stream)
                        calls.append((L.snip_quantize_stats, args, "quant_stats", (bpe + 0.0) * t.numel(), "q", p, -1))
                    else:
                        args = self._plain_quant(L, f, block, t, rows, cols, orient, rnd[r], sid + r, g, dst_c, dst_s,
                                                 ws, wsb, stream)
                        calls.append((args[0], args[1], qcat, bpe * t.numel(), "q", p, -1))
                    continue
                if r in (0, 1, 2) and stats:
                    # row-block quantization with SNIP's statistics of the same tensor in one pass
                    k = r
                    args = (f, t.data_ptr(), rows, cols, rnd[r], 0, sid + r, scp[name], snip.MMA,
                            self.codes[r].data_ptr(), self.scales[r].data_ptr() if f != snip.FP8 else None,
                            self.raw[j, k].data_ptr(), ws, wsb, stream)
                    calls.append((L.snip_quantize_stats, args, "quant_stats", (bpe + 0.0) * t.numel(), "q", p, -1))
                elif block > 16:
                    args = (t.data_ptr(), rows, cols, orient, rnd[r], 0, sid + r, g, block, snip.MMA,
                            self.codes[r].data_ptr(), self.scales[r].data_ptr(), g, ws, wsb, stream)
                    calls.append((L.snip_quantize_nvfp4_block, args, qcat, bpe * t.numel(), "q", p, -1))
                elif f == snip.NVFP4:
                    args = (t.data_ptr(), rows, cols, orient, rnd[r], 0, sid + r, g, snip.MMA,
                            self.codes[r].data_ptr(), self.scales[r].data_ptr(), g, None, ws, wsb, stream)
                    calls.append((L.snip_quantize_nvfp4, args, qcat, bpe * t.numel(), "q", p, -1))
                elif f == snip.MXFP4:
                    args = (t.data_ptr(), rows, cols, orient, rnd[r], 0, sid + r, snip.MMA,
                            self.codes[r].data_ptr(), self.scales[r].data_ptr(), ws, wsb, stream)
                    calls.append((L.snip_quantize_mxfp4, args, qcat, bpe * t.numel(), "q", p, -1))
                else:
                    args = (t.data_ptr(), rows, cols, orient, rnd[r], 0, sid + r, g, snip.MMA,
                            self.codes[r].data_ptr(), g, ws, wsb, stream)
                    calls.append((L.snip_quantize_fp8, args, qcat, bpe * t.numel(), "q", p, -1))
                if r in (1, 3, 5):   # both operands of a GEMM are ready
                    a, b = r - 1, r
                    M, N, K = {1: (T, l.N, l.K), 3: (T, l.K, l.N), 5: (l.N, l.K, T)}[r]
                    D = {1: self.Y[j], 3: self.dX[j], 5: self.dW[j]}[r]
                    ac, asc = self.codes[a], self.scales[a]
                    if r == 1 and xcodes is not None:
                        ac, asc = xcodes, xscales
                    sa = asc.data_ptr() if f != snip.FP8 else None
                    sb = self.scales[b].data_ptr() if f != snip.FP8 else None
                    ga = scp[roles(l)[a][0]] + fo if f != snip.MXFP4 else None
                    gb = scp[roles(l)[b][0]] + fo if f != snip.MXFP4 else None
                    k = (p if self.gemm_streams == 2 else r // 2) % self.gemm_streams
                    gw = self.gemm_wss[k]
                    args = (f, ac.data_ptr(), sa, ga, self.codes[b].data_ptr(), sb, gb, M, N, K,
                            D.data_ptr(), D.stride(0), gw.ptr, gw.nbytes, self.sGs[k].cuda_stream)
                    self.gsel[len(calls)] = k
                    calls.append((L.snip_gemm, args, gcat, 2.0 * M * N * K, "g", p, r // 2))
        self.calls = calls
        self.last_q = {}   # position -> index of its last quantization (tensor-scale passes excluded)
        for i, c in enumerate(calls):
            if c[4] == "q" and c[2] != "scales":
                self.last_q[c[5]] = i
        # the same calls with every launch on the quantization stream (kernels one after another)
        self.serial_args = [a if k == "q" else a[:-1] + (stream,) for (_, a, _, _, k, _, _) in calls]
        # one kernel per call (the scales are computed once per tensor and passed in; every plan
        # format here has its statistics fused into its row-block quantization)
        self.launches_per_step = len(calls)

    @staticmethod
    def _plain_quant(L, f, block, t, rows, cols, orient, rnd, sid, g, dst_c, dst_s, ws, wsb, stream):
        """(function, arguments) of a plain quantization of t in format f (MMA layout)."""
        import sub_byte_mixed_gb300.snip as snip
        if block > 16:
            return L.snip_quantize_nvfp4_block, (t.data_ptr(), rows, cols, orient, rnd, 0, sid, g, block, snip.MMA,
                                                 dst_c, dst_s, g, ws, wsb, stream)
        if f == snip.NVFP4:
            return L.snip_quantize_nvfp4, (t.data_ptr(), rows, cols, orient, rnd, 0, sid, g, snip.MMA, dst_c, dst_s, g,
                                           None, ws, wsb, stream)
        if f == snip.MXFP4:
            return L.snip_quantize_mxfp4, (t.data_ptr(), rows, cols, orient, rnd, 0, sid, snip.MMA, dst_c, dst_s, ws,
                                           wsb, stream)
        return L.snip_quantize_fp8, (t.data_ptr(), rows, cols, orient, rnd, 0, sid, g, snip.MMA, dst_c, g, ws, wsb,
                                     stream)

    def stats_host(self):
        """The step's statistics (linears x {X, W, dY} x raw values) on the host, the statistics of a
        shared activation repeated for every linear that reads it."""
        raw = self.raw.cpu().numpy().copy()
        for j, l in enumerate(self.cfg.linears):
            raw[j, 0] = raw[self.first_user[l.x_id], 0]
        return raw

    def run(self, events=None, serial=False):
        """One step.  With overlap, a GEMM waits for its two operands' quantizations, and the
        quantizations of the linear at position p wait until the GEMMs of the linear at p-2 (the
        last readers of the same operand buffers) are done; the step ends on the quantization
        stream after all GEMMs.
        serial: every kernel on the quantization stream, one after another (per-kernel timing)."""
        import torch
        ready, gdone = {}, {}
        last_g = {}
        qdone, sdone = {}, {}   # position -> event: its last quantization; its scale pass
        last_s = None
        overlap = self.overlap and not serial
        cur = torch.cuda.current_stream()
        if cur != self.sQ:
            ev = torch.cuda.Event()
            ev.record(cur)
            self.sQ.wait_event(ev)
        for i, (fn, args, _, _, kind, p, gi) in enumerate(self.calls):
            if serial:
                args = self.serial_args[i]
            stream = self.sQ if kind == "q" or serial else self.sGs[self.gsel[i]]
            on_s = overlap and i in self.scale_call
            if on_s:
                args, stream = self.scale_call[i], self.sS
                if (p - self.scales_lead) in qdone:
                    self.sS.wait_event(qdone[p - self.scales_lead])
                elif last_s is None:   # the first pass follows the caller's work
                    ev = torch.cuda.Event()
                    ev.record(self.sQ)
                    self.sS.wait_event(ev)
            if overlap:
                if i in self.wait_at:
                    for ev in gdone.get(p - 2, []):
                        self.sQ.wait_event(ev)
                    if p in sdone:
                        self.sQ.wait_event(sdone[p])
                if kind == "g":
                    stream.wait_event(ready[(p, gi)])
            if events is not None:
                events[i][0].record(stream)
            st = fn(*args)
            if st != 0:
                raise RuntimeError(f"{fn.__name__} failed with status {st}")
            if events is not None:
                events[i][1].record(stream)
            if on_s:
                ev = torch.cuda.Event()
                ev.record(self.sS)
                sdone[p] = ev
                last_s = ev
            if overlap:
                nxt = self.calls[i + 1] if i + 1 < len(self.calls) else None
                if self.scale_call and i == self.last_q.get(p):   # the last quantization of position p
                    ev = torch.cuda.Event()
                    ev.record(self.sQ)
                    qdone[p] = ev
                if kind == "q" and nxt is not None and nxt[4] == "g":   # both operands of the next GEMM written
                    ev = torch.cuda.Event()
                    ev.record(self.sQ)
                    ready[(nxt[5], nxt[6])] = ev
                if kind == "g":
                    ev = torch.cuda.Event()
                    ev.record(stream)
                    gdone.setdefault(p, []).append(ev)
                    last_g[self.gsel[i]] = ev
        if overlap:
            for ev in last_g.values():
                self.sQ.wait_event(ev)
            if last_s is not None:
                self.sQ.wait_event(last_s)
        if cur != self.sQ:
            ev = torch.cuda.Event()
            ev.record(self.sQ)
            cur.wait_event(ev)

    def capture(self):
        """Record one step (both streams, with their events) as a CUDA graph."""
        import torch
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.sQ):
            self.graph.capture_begin()
            self.run()
            self.graph.capture_end()
        torch.cuda.synchronize()

    def replay(self):
        """One step from the captured graph, on the caller's stream."""
        self.graph.replay()

    def status(self):
        for w in [self.ws] + self.gemm_wss + ([self.ws_s] if self.ws_s is not None else []):
            s = w.status()
            if s != self.snip.SNIP_OK:
                return s
        return self.snip.SNIP_OK


def quantizer_sweep(snip, hbm_gbs: float, reps: int = 10):
    """Standalone quantizers on the 8192 x 8192 tensor with 0.1% outliers (x100): each variant's
    algorithmic GB/s (bf16 read + codes + scales written; statistics and tensor scales read only)
    and its fraction of the measured HBM copy bandwidth.  Reading a 1.5 GB scratch buffer before
    each timed launch flushes L2 with clean lines (no write-back overlaps the launch) and keeps the
    GPU busy while the host queues the pre-marshalled C-ABI call, so no idle gap is timed."""
    import torch
    from sub_byte_mixed_gb300 import inputs
    L = snip.load()
    x = inputs.outlier_bf16(8192, 8192, seed=0, tensor_id=1, device="cuda")
    n, R, C = x.numel(), 8192, 8192
    ws = snip.Workspace(snip.snip_quantize_workspace_size(0, 0))
    st = torch.cuda.current_stream().cuda_stream
    sc = torch.empty(4, dtype=torch.float32, device="cuda")
    L.snip_tensor_scales(x.data_ptr(), n, sc.data_ptr(), ws.ptr, ws.nbytes, st)
    cb, sb = snip.snip_quantized_bytes(snip.NVFP4, snip.MMA, R, C)
    codes = torch.empty(max(cb, C * R), dtype=torch.uint8, device="cuda")
    scales = torch.empty(max(sb, 16), dtype=torch.uint8, device="cuda")
    s_out = torch.empty(1, dtype=torch.float32, device="cuda")
    raw = torch.empty(snip.STATS_NVALS, dtype=torch.float64, device="cuda")
    xp, cp, sp, w = x.data_ptr(), codes.data_ptr(), scales.data_ptr(), (ws.ptr, ws.nbytes, st)
    g, s8 = sc.data_ptr() + 4, sc.data_ptr() + 8
    variants = {   # name: (C-ABI function, arguments, algorithmic bytes per element)
        "scales": (L.snip_tensor_scales, (xp, n, sc.data_ptr(), *w), 2.0),
        "nvfp4_rtn_rows": (L.snip_quantize_nvfp4, (xp, R, C, 0, 0, 0, 1, g, snip.MMA, cp, sp, s_out.data_ptr(), None, *w),
                           2 + 0.5625),
        "nvfp4_sr_rows": (L.snip_quantize_nvfp4, (xp, R, C, 0, 1, 0, 2, g, snip.MMA, cp, sp, s_out.data_ptr(), None, *w),
                          2 + 0.5625),
        "nvfp4_sr_cols": (L.snip_quantize_nvfp4, (xp, R, C, 1, 1, 0, 3, g, snip.MMA, cp, sp, s_out.data_ptr(), None, *w),
                          2 + 0.5625),
        "mxfp4_sr_cols": (L.snip_quantize_mxfp4, (xp, R, C, 1, 1, 0, 4, snip.MMA, cp, sp, *w), 2 + 0.53125),
        "fp8_rtn_rows": (L.snip_quantize_fp8, (xp, R, C, 0, 0, 0, 5, s8, snip.MMA, cp, s_out.data_ptr(), *w), 3.0),
        "fp8_sr_cols": (L.snip_quantize_fp8, (xp, R, C, 1, 1, 0, 6, s8, snip.MMA, cp, s_out.data_ptr(), *w), 3.0),
        "stats_rtn": (L.snip_quant_stats, (xp, R, C, 0, 0, 7, sc.data_ptr(), raw.data_ptr(), None, None, *w), 2.0),
        "quant_stats_nvfp4_rtn": (L.snip_quantize_stats, (snip.NVFP4, xp, R, C, 0, 0, 8, sc.data_ptr(), snip.MMA, cp, sp,
                                                          raw.data_ptr(), *w), 2 + 0.5625),
        "quant_stats_nvfp4_sr": (L.snip_quantize_stats, (snip.NVFP4, xp, R, C, 1, 0, 9, sc.data_ptr(), snip.MMA, cp, sp,
                                                         raw.data_ptr(), *w), 2 + 0.5625),
    }
    flush = torch.ones(1536 << 20 >> 2, dtype=torch.int32, device="cuda")
    flush_out = torch.empty((), dtype=torch.int32, device="cuda")
    out = {}
    for name, (fn, args, bpe) in variants.items():
        if fn(*args) != 0:
            raise RuntimeError(f"{name} failed")
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(reps):
            torch.max(flush, out=flush_out)   # reads 1.5 GB
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn(*args)
            e1.record()
            torch.cuda.synchronize()
            tot += e0.elapsed_time(e1)
        ms = tot / reps
        gbs = bpe * n / (ms * 1e-3) / 1e9
        out[name] = {"us": round(ms * 1e3, 1), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm_gbs, 3)}
    if ws.status() != snip.SNIP_OK:
        raise RuntimeError("device status " + snip.status_string(ws.status()))
    return {"tensor": "8192x8192 bf16, N(0,1) with 0.1% of entries x100 (seeded)", "l2": "flushed before each launch",
            "variants": out}


def requant_compare(snip, reps: int = 10):
    """The Down linear's dgrad of the 7B block (dX = dY W: 8192 x 11008, contraction 4096), NVFP4:
    the product re-quantized in the GEMM epilogue for the preceding layer (snip_gemm_requant, no fp32
    output) against the unfused chain it replaces -- fp32 dX, a bf16 copy, then the row-block SR
    quantization of that copy."""
    import torch
    from sub_byte_mixed_gb300 import inputs
    M, N, K = 8192, 11008, 4096
    dY = inputs.normal_bf16((M, K), 1e-3, 0, 40, "cuda")
    Wt = inputs.normal_bf16((N, K), 0.02, 0, 41, "cuda")
    a = snip.quantize_nvfp4(dY, rnd=1, layout=snip.MMA)
    b = snip.quantize_nvfp4(Wt, rnd=1, layout=snip.MMA)
    g = torch.tensor([1e-5], dtype=torch.float32, device="cuda")
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    Db = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def fused():
        snip.gemm_requant(snip.NVFP4, a, b, M, N, K, g, rnd=1, seed=0, stream_id=2, want_d=False)

    def unfused():
        snip.gemm(snip.NVFP4, a, b, M, N, K, out=D)
        Db.copy_(D)
        snip.quantize_nvfp4(Db, rnd=1, seed=0, stream_id=2, g_in=g, layout=snip.MMA)

    # both orientations: the preceding layer's dgrad operand (row blocks) and its wgrad operand dY^T
    # (column blocks, along the tokens)
    def fused_both():
        snip.gemm_requant(snip.NVFP4, a, b, M, N, K, g, rnd=1, seed=0, stream_id=2, want_d=False, cols=True,
                          rnd_t=1, stream_id_t=4)

    def unfused_both():
        unfused()
        snip.quantize_nvfp4(Db, orient=snip.ALONG_ROWS, rnd=1, seed=0, stream_id=4, g_in=g, layout=snip.MMA)

    out = {}
    for name, fn in (("fused_ms", fused), ("unfused_ms", unfused), ("fused_both_ms", fused_both),
                     ("unfused_both_ms", unfused_both)):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        out[name] = round(e0.elapsed_time(e1) / reps, 4)
    out["shape"] = f"{M}x{N}x{K} NVFP4, SR re-quantization (row blocks; _both: row and column blocks)"
    return out


def chain_compare(snip, reps: int = 5):
    """NEXT-3 in the layer path on the 7B block: the backward of Down (K = 11008, N = 4096) and of the
    linear before it, Up (K = 4096, N = 11008), whose dY is Down's dX (T = 8192).  Unfused: Down's
    snip_qlinear_bwd writes fp32 dX, a bf16 copy of it is Up's dY, and Up's snip_qlinear_bwd quantizes
    it (just-in-time scale).  Fused: snip_qlinear_bwd_chain writes Up's two NVFP4 gradient operands in
    Down's dgrad epilogue (delayed scale), and snip_qlinear_bwd_q runs Up's backward from them."""
    import torch
    from sub_byte_mixed_gb300 import inputs
    cfg = inputs.LLAMA7B
    names = [l.name for l in cfg.linears]
    jd, ju = names.index("Down"), names.index("Up")
    Xd, Wd, dYd = inputs.linear_inputs(cfg, jd, seed=0, device="cuda")
    Xu, Wu, _ = inputs.linear_inputs(cfg, ju, seed=0, device="cuda")
    T = cfg.T
    plan = snip.Plan([1] * len(cfg.linears), seed=0)
    wsd = snip.qlinear_workspace(plan, jd, T, cfg.linears[jd].K, cfg.linears[jd].N)
    wsu = snip.qlinear_workspace(plan, ju, T, cfg.linears[ju].K, cfg.linears[ju].N)
    dX = torch.empty((T, cfg.linears[jd].K), dtype=torch.float32, device="cuda")
    dWd = torch.empty((cfg.linears[jd].N, cfg.linears[jd].K), dtype=torch.float32, device="cuda")
    dYu = torch.empty((T, cfg.linears[jd].K), dtype=torch.bfloat16, device="cuda")
    dXu = torch.empty((T, cfg.linears[ju].K), dtype=torch.float32, device="cuda")
    dWu = torch.empty((cfg.linears[ju].N, cfg.linears[ju].K), dtype=torch.float32, device="cuda")
    snip.qlinear_bwd(plan, jd, Xd, Wd, dYd, wsd, dX=dX, dW=dWd)
    g = (snip.tensor_scales(dX.to(torch.bfloat16))[1:2]).clone()   # the delayed scale: a previous step's

    def unfused():
        snip.qlinear_bwd(plan, jd, Xd, Wd, dYd, wsd, dX=dX, dW=dWd)
        dYu.copy_(dX)
        snip.qlinear_bwd(plan, ju, Xu, Wu, dYu, wsu, dX=dXu, dW=dWu)

    def fused():
        _, _, rows, cols, _ = snip.qlinear_bwd_chain(plan, jd, ju, Xd, Wd, dYd, g, wsd)
        snip.qlinear_bwd_q(plan, ju, Xu, Wu, rows, cols, wsu, dX=dXu, dW=dWu)

    out = {}
    for name, fn in (("unfused_ms", unfused), ("fused_ms", fused)):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        out[name] = round(e0.elapsed_time(e1) / reps, 4)
    if wsd.status() != snip.SNIP_OK or wsu.status() != snip.SNIP_OK:
        raise RuntimeError("device status")
    out["saved_ms"] = round(out["unfused_ms"] - out["fused_ms"], 4)
    out["what"] = ("backward of the 7B block's Down and Up linears (T = 8192), Up's dY = Down's dX: fused "
                   "(chain + backward from quantized operands) vs unfused (fp32 dX, bf16 copy, quantize)")
    return out


def dw_noise_time(snip, bf16_peak: float, reps: int = 10):
    """NEXT-4 at the 7B block's Down linear (T = 8192, K = 11008, N = 4096): snip_dw_noise, the bf16
    tensor-core GEMM dW = dY^T X with ||dW||^2 and ||dW_q - dW||^2 in its epilogue, against the
    measured bf16 burst peak (the kernel is timed alone, back to back, operands from HBM: 247 MB of
    bf16 inputs and 180 MB of dW_q)."""
    import torch
    from sub_byte_mixed_gb300 import inputs
    cfg = inputs.LLAMA7B
    j = [l.name for l in cfg.linears].index("Down")
    X, W, dY = inputs.linear_inputs(cfg, j, seed=0, device="cuda")
    T, K, N = cfg.T, cfg.linears[j].K, cfg.linears[j].N
    dwq = torch.randn((N, K), dtype=torch.float32, device="cuda")
    ws = snip.Workspace(snip.snip_dw_noise_workspace_size(K, N))
    out = torch.empty(2, dtype=torch.float64, device="cuda")
    L = snip.load()
    args = (X.data_ptr(), dY.data_ptr(), T, K, N, dwq.data_ptr(), out.data_ptr(), ws.ptr, ws.nbytes,
            torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        if L.snip_dw_noise(*args) != 0:
            raise RuntimeError("snip_dw_noise failed")
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        L.snip_dw_noise(*args)
    e1.record()
    torch.cuda.synchronize()
    if ws.status() != snip.SNIP_OK:
        raise RuntimeError("device status " + snip.status_string(ws.status()))
    ms = e0.elapsed_time(e1) / reps
    tf = 2.0 * T * K * N / (ms * 1e-3) / 1e12
    return {"shape": f"T={T} K={K} N={N} (7B Down)", "ms": round(ms, 4), "TFLOP/s": round(tf, 1),
            "frac_bf16_burst": round(tf / bf16_peak, 3),
            "what": "bf16 tcgen05 GEMM dW = dY^T X, norms of dW and dW_q - dW in its epilogue; dW never stored"}


def e2e_run(cfg, plan, snip, step: Step, nsteps: int, rounds_n: int = 5, with_outputs: bool = False):
    """The same step through the layer API (snip_qlinear_fwd / _bwd, statistics fused into their
    quantizations) with host buffers: every step copies all inputs (X, W, dY, bf16) in from pinned host
    memory and reads the step's metric -- SNIP's statistics of every operand tensor -- back to the host,
    inside the timed region.  Y, dX and dW stay on the device, where the next layer, the previous layer
    and the optimizer consume them; with_outputs: they are copied back to pinned host memory too, every
    step (host to host)."""
    import torch
    inp = step.inp
    hX = {k: v.cpu().pin_memory() for k, v in inp.X.items()}
    hW = [w.cpu().pin_memory() for w in inp.W]
    hdY = [d.cpu().pin_memory() for d in inp.dY]
    hraw = torch.empty(step.raw.shape, dtype=step.raw.dtype).pin_memory()
    p = snip.Plan(plan, seed=0)
    wsb = max(snip.snip_qlinear_workspace_size(p.handle, j, cfg.T, l.K, l.N) for j, l in enumerate(cfg.linears))
    # two layer-call streams, linears alternating between them with a workspace each: a linear's
    # quantizations run beside the previous linear's GEMMs
    wss = [snip.Workspace(wsb), snip.Workspace(wsb)]
    h2d = sum(t.numel() * t.element_size() for t in list(hX.values()) + hW + hdY)
    d2h = hraw.numel() * 8
    if with_outputs:
        hout = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (step.Y[j], step.dX[j], step.dW[j])]
                for j in range(len(cfg.linears))]
        d2h += sum(t.numel() * t.element_size() for ts in hout for t in ts)

    # Three streams: host->device copies (H), the layer calls (C), device->host copies (D).  Linear j's
    # inputs are copied while earlier linears compute, and its statistics read back while later ones do;
    # events keep each device buffer from being overwritten before its last reader is done.
    sC, sH, sD = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sCs = [sC, torch.cuda.Stream()]
    n = len(cfg.linears)
    ev = lambda: torch.cuda.Event()
    last_user = {}   # x_id -> last linear reading that activation
    for j, l in enumerate(cfg.linears):
        last_user[l.x_id] = j
    first_user = {}
    for j, l in enumerate(cfg.linears):
        first_user.setdefault(l.x_id, j)
    state = {"computed": [None] * n, "drained": [None] * n}

    def one():
        loaded = [None] * n
        for j, l in enumerate(cfg.linears):
            with torch.cuda.stream(sH):
                prev = state["computed"][j]
                if prev is not None:
                    sH.wait_event(prev)                 # the previous step's linear j has read its inputs
                if first_user[l.x_id] == j:
                    lu = state["computed"][last_user[l.x_id]]
                    if lu is not None:
                        sH.wait_event(lu)               # ... and every reader of the shared activation
                    inp.X[l.x_id].copy_(hX[l.x_id], non_blocking=True)
                inp.W[j].copy_(hW[j], non_blocking=True)
                inp.dY[j].copy_(hdY[j], non_blocking=True)
                loaded[j] = ev()
                loaded[j].record(sH)
        for j, l in enumerate(cfg.linears):
            sc, ws = sCs[j % 2], wss[j % 2]
            sc.wait_event(loaded[j])
            if first_user[l.x_id] != j:
                sc.wait_event(loaded[first_user[l.x_id]])
            if state["drained"][j] is not None:
                sc.wait_event(state["drained"][j])      # the previous step's statistics copied out
            X = inp.X[l.x_id]
            # statistics of X, W (forward) and dY (dgrad) come out of the quantization passes
            with torch.cuda.stream(sc):
                snip.qlinear_fwd(p, j, X, inp.W[j], ws, Y=step.Y[j], stats=step.raw[j, 0:2])
                snip.qlinear_bwd(p, j, X, inp.W[j], inp.dY[j], ws, dX=step.dX[j], dW=step.dW[j],
                                 stats=step.raw[j, 2])
            done = ev()
            done.record(sc)
            state["computed"][j] = done
            with torch.cuda.stream(sD):
                sD.wait_event(done)
                hraw[j].copy_(step.raw[j], non_blocking=True)
                if with_outputs:
                    for h, d in zip(hout[j], (step.Y[j], step.dX[j], step.dW[j])):
                        h.copy_(d, non_blocking=True)
                dr = ev()
                dr.record(sD)
                state["drained"][j] = dr

    for _ in range(2):   # warm-up: first-use costs of the layer calls and the pinned buffers
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # several rounds of nsteps, the median reported: a round now and then runs about twice as long
    # (the host-driven step leaves the GPU waiting on copies); the clocks are sampled meanwhile
    sampler = ClockSampler(torch.cuda.current_device())
    t_start = time.time()
    rounds = []
    for _ in range(rounds_n):
        e0.record(sC)
        sH.wait_event(e0)
        sD.wait_event(e0)
        sCs[1].wait_event(e0)
        for _ in range(nsteps):
            one()
        for j in range(n):
            sC.wait_event(state["drained"][j])
        e1.record(sC)
        torch.cuda.synchronize()
        rounds.append(e0.elapsed_time(e1) / nsteps)
    clocks = sampler.summary(t_start, time.time())
    sampler.stop()
    for ws in wss:
        if ws.status() != snip.SNIP_OK:
            raise RuntimeError("device status " + snip.status_string(ws.status()))
    ms = sorted(rounds)[len(rounds) // 2]
    # the host->device copies of one step alone, for the bound they put on the step (median of as many
    # rounds as the step itself: one slow round of the host link must not set it)
    h2d_rounds = []
    for _ in range(rounds_n):
        torch.cuda.synchronize()
        e0.record(sH)
        for _ in range(nsteps):
            with torch.cuda.stream(sH):
                for k in hX:
                    inp.X[k].copy_(hX[k], non_blocking=True)
                for j in range(n):
                    inp.W[j].copy_(hW[j], non_blocking=True)
                    inp.dY[j].copy_(hdY[j], non_blocking=True)
        e1.record(sH)
        torch.cuda.synchronize()
        h2d_rounds.append(e0.elapsed_time(e1) / nsteps)
    ms_h2d = sorted(h2d_rounds)[len(h2d_rounds) // 2]
    return {"value": cfg.flops_fwd_bwd() / (ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "h2d_only_ms_per_step": ms_h2d,
            "h2d_gbs": h2d / (ms_h2d * 1e-3) / 1e9,
            "rounds_ms_per_step": [round(r, 3) for r in rounds], "timing": f"median of {rounds_n} rounds of {nsteps} steps",
            "h2d_only_rounds_ms_per_step": [round(r, 3) for r in h2d_rounds],
            "clocks": clocks,
            "path": "snip_qlinear_fwd/bwd with fused statistics; all inputs copied in from pinned host memory "
                    "and the step's SNIP statistics read back every step, overlapping other linears' calls "
                    "(copy-in, two layer-call and copy-out streams); "
                    + ("Y, dX, dW (fp32) copied back to pinned host memory every step as well"
                       if with_outputs else "Y, dX, dW stay on the device")}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from sub_byte_mixed_gb300 import build, snip
    torch.cuda.set_device(local_rank)
    build.build()
    snip.load()
    snip.snip_device_check()
    cfg, plan = workload(args)
    layers = [x for x in args.layers.split(",") if x]
    graph = not args.no_graph
    step = Step(cfg, plan, snip, "cuda", layers, overlap=not args.no_overlap, own_stream=graph,
                scales_per_launch=args.scales_per_launch, order=linear_order(args),
                gemm_streams=args.gemm_streams, scales_stream=not args.no_scales_stream,
                scales_lead=args.scales_lead)
    if args.plan == "snip" and layers:
        raise SystemExit("--plan snip selects formats for the whole block; it cannot be combined with --layers")
    if args.plan == "snip":
        # SNIP's loop: statistics of one step feed the layer-wise selection (C ABI, host code)
        step.run()
        torch.cuda.synchronize()
        c8, c4 = snip.snip_plan_costs(step.stats_host())
        flops = [6.0 * cfg.T * l.K * l.N for l in cfg.linears]
        plan, _, _ = snip.snip_plan_select(flops, c8, c4, cfg.fp4_target)
        del step
        step = Step(cfg, plan, snip, "cuda", layers, overlap=not args.no_overlap, own_stream=graph,
                scales_per_launch=args.scales_per_launch, order=linear_order(args),
                gemm_streams=args.gemm_streams, scales_stream=not args.no_scales_stream,
                scales_lead=args.scales_lead)
    torch.cuda.synchronize()
    ncalls = len(step.calls)
    sampler = ClockSampler(local_rank) if rank == 0 and not args.profile_run else None
    for _ in range(args.warmup if args.profile_run else max(args.warmup, 3)):
        step.run()
    if not args.profile_run:
        # keep the GPU loaded for ~1 s so the clock sampler sees load before timing
        t_settle = time.time()
        while time.time() - t_settle < 1.0:
            step.run()
            torch.cuda.synchronize()
    if graph:
        step.capture()   # the whole step, both streams, as one CUDA graph
        for _ in range(2):
            step.replay()
    events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(ncalls)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record()
    for s in range(args.steps):
        if graph:
            step.replay()
        else:
            step.run()
    stop.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    ms = start.elapsed_time(stop) / args.steps
    status = step.status()
    if status != snip.SNIP_OK:
        raise RuntimeError("device status " + snip.status_string(status))
    # per-kernel durations: kernels that share the SMs stretch each other's event times, and a
    # replayed graph has no per-launch events, so the breakdown and the roofline come from the
    # same calls issued one at a time on one stream, K more steps in a row
    for _ in range(3):
        step.run(serial=True)
    torch.cuda.synchronize()
    start.record()
    for s in range(args.steps):
        step.run(events[s], serial=True)
    stop.record()
    torch.cuda.synchronize()
    ms_serial = start.elapsed_time(stop) / args.steps
    status = step.status()
    if status != snip.SNIP_OK:
        raise RuntimeError("device status " + snip.status_string(status))
    # per-category kernel time
    cat_ms, cat_units, cat_n = {}, {}, {}
    for s in range(args.steps):
        for i, (_, _, cat, units, _, _, _) in enumerate(step.calls):
            t = events[s][i][0].elapsed_time(events[s][i][1])
            cat_ms[cat] = cat_ms.get(cat, 0.0) + t
            cat_units[cat] = cat_units.get(cat, 0.0) + units
            cat_n[cat] = cat_n.get(cat, 0) + 1
    flops_step = cfg.flops_fwd_bwd() if not layers else sum(6 * cfg.T * l.K * l.N for l in cfg.linears
                                                             if l.name in layers)

    def time_variant(plan_v, stats_v):
        """Another step of the same block, timed as the headline (K steps after 3 warm-up steps)."""
        sv = Step(cfg, plan_v, snip, "cuda", layers, overlap=not args.no_overlap, stats=stats_v, own_stream=graph,
                  scales_per_launch=args.scales_per_launch, order=linear_order(args),
                gemm_streams=args.gemm_streams, scales_stream=not args.no_scales_stream,
                scales_lead=args.scales_lead)
        for _ in range(3):
            sv.run()
        if graph:
            sv.capture()
            sv.replay()
        torch.cuda.synchronize()
        start.record()
        for _ in range(args.steps):
            if graph:
                sv.replay()
            else:
                sv.run()
        stop.record()
        torch.cuda.synchronize()
        if sv.status() != snip.SNIP_OK:
            raise RuntimeError("device status " + snip.status_string(sv.status()))
        msv = start.elapsed_time(stop) / args.steps
        return {"value": flops_step / (msv * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": msv,
                "launches_per_step": sv.launches_per_step, "fp4_flop_fraction": round(cfg.fp4_flop_fraction(plan_v), 4)}

    # the same step without SNIP's statistics (SNIP collects them periodically; the steps in between
    # only quantize and multiply), for the statistics' share of the step; and the block's uniform plans
    no_stats = other_plans = None
    if not args.profile_run and rank == 0:
        no_stats = time_variant(plan, False)
        no_stats["what"] = "the same step with plain row-block quantizations in place of the statistics-fused ones"
        if args.plan in ("mix", "snip") and not layers:
            from sub_byte_mixed_gb300 import inputs as inp_mod
            other_plans = {name: time_variant(inp_mod.all_plan(FORMAT_OF_NAME[name]), True)
                           for name in ("fp8", "nvfp4")}
    t2 = time.time()
    ms = max_over_ranks(ms, world, "cuda")
    clocks = sampler.summary(t0, t2) if sampler else None
    if sampler:
        sampler.stop()
    qsweep = rqcmp = dwn = chn = None
    if not args.profile_run and not layers and rank == 0:
        qsweep = quantizer_sweep(snip, measured_peaks()["hbm_gbs"])
        rqcmp = requant_compare(snip)
        dwn = dw_noise_time(snip, measured_peaks()["bf16"])
        chn = chain_compare(snip)
    e2e = e2e_out = None
    if not args.no_e2e and not args.profile_run and not layers and rank == 0:
        e2e = e2e_run(cfg, plan, snip, step, args.e2e_steps)
        e2e_out = e2e_run(cfg, plan, snip, step, max(2, args.e2e_steps // 2), rounds_n=3, with_outputs=True)
    if rank != 0:
        return
    flops = cfg.flops_fwd_bwd() if not layers else sum(
        6 * cfg.T * l.K * l.N for l in cfg.linears if l.name in layers)
    value = whole_job_tflops(world, flops, ms)
    peaks = measured_peaks()
    breakdown = {}
    for cat in cat_ms:
        t = cat_ms[cat] / 1e3
        if cat.startswith("gemm"):
            # each launch is timed alone on the GPU (serial pass): the burst bf16 figure x the nominal
            # dense ratio is its peak; the sustained-derived fraction is kept beside it
            ratio = FP8_OVER_BF16 if cat == "gemm_fp8" else FP4_OVER_BF16
            ach = cat_units[cat] / t / 1e12
            pk = peaks["bf16"] * ratio
            pks = peaks["bf16_sustained"] * ratio
            breakdown[cat] = {"ms_per_step": cat_ms[cat] / args.steps, "launches_per_step": cat_n[cat] // args.steps,
                              "achieved": ach, "unit": "TFLOP/s", "peak": pk, "frac": ach / pk,
                              "peak_sustained": pks, "frac_sustained": ach / pks}
        else:
            ach = cat_units[cat] / t / 1e9
            breakdown[cat] = {"ms_per_step": cat_ms[cat] / args.steps, "launches_per_step": cat_n[cat] // args.steps,
                              "achieved": ach, "unit": "GB/s", "peak": peaks["hbm_gbs"],
                              "frac": ach / peaks["hbm_gbs"]}
    dom = max(breakdown, key=lambda c: breakdown[c]["ms_per_step"])
    d = breakdown[dom]
    tr = ncu_traffic(dom)
    traffic = None
    if tr is not None:
        # DRAM bytes of one average launch = recorded bytes per unit x units per launch
        traffic = tr * cat_units[dom] / cat_n[dom]
    roofline = {"bound": "tensor" if dom.startswith("gemm") else "hbm", "kernel": dom,
                "achieved": d["achieved"], "peak": d["peak"], "unit": d["unit"], "frac": d["frac"],
                "traffic": traffic,
                "timed": "CUDA events around each launch in K steps issued one call at a time on one stream, "
                         "right after the timed region (kernels alone on the GPU)",
                "peak_source": f"{peaks['source']} ("
                + ("bf16 burst x nominal FP4/FP8 dense ratio: the kernel is timed alone"
                   if dom.startswith("gemm") else "HBM copy") + ")"}
    qcats = [c for c in breakdown if not c.startswith("gemm")]
    q_bytes = sum(cat_units[c] for c in qcats) / args.steps
    q_ms = sum(cat_ms[c] for c in qcats) / args.steps
    quant = {"value": q_bytes / (q_ms * 1e-3) / 1e9, "unit": "GB/s",
             "frac": q_bytes / (q_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], "of": "measured HBM copy bandwidth"}
    gemm_fl = sum(cat_units[c] for c in breakdown if c.startswith("gemm")) / args.steps
    gemm_ms = sum(cat_ms[c] for c in breakdown if c.startswith("gemm")) / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4/fp8 (fp32 accumulate)", "data": "synthetic (seeded N(0,s^2) bf16)",
        "config": config_json(cfg, plan, args),
        "roofline": roofline,
        "quantizer": quant,
        "gemm_only": {"value": gemm_fl / (gemm_ms * 1e-3) / 1e12, "unit": UNIT},
        "quantizer_sweep": qsweep,
        "next3_requant": rqcmp,
        "next4_dw_noise": dwn,
        "next3_chain": chn,
        "breakdown": breakdown,
        "clocks": clocks,
        "e2e": e2e,
        "e2e_with_outputs": e2e_out,
        "gpu_launches": step.launches_per_step * args.steps,
        "ms_per_step_one_stream": ms_serial,
        "without_stats": no_stats,
        "uniform_plans": other_plans,
    }
    if layers:
        line["config"]["layers"] = layers
    if not args.no_cpu_baseline and not args.profile_run:
        line["cpu_baseline"] = run_cpu_baseline_subprocess(args.cpu_sample_seconds)
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- reference arm (the oracle)

def run_reference(args, rank):
    """The oracle, as it stands, on every host core: each step is one repetition of the bounded sample
    in each of n worker processes at once; value = n x the sample's flops / the step's wall time."""
    if rank != 0:
        return
    cfg, plan = workload(args)
    n = os.cpu_count() or 1
    times = []
    with oracle_pool(n) as pool:
        pool.map(_oracle_sample_rep, range(n))            # first use, untimed
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            pool.map(_oracle_sample_rep, range(n))
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = n * SAMPLE_FLOPS / (ms * 1e-3) / 1e12
    sample = f"{SAMPLE_TEXT}; one per worker per step, {n} worker processes (one per host core)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded N(0,s^2) bf16)",
            "config": config_json(cfg, plan, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": n, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


GEMM_SHAPES = [  # (M, N, K): the 7B block's Down fwd / dgrad / wgrad and Q fwd, the 70B block's Down fwd
    ("llama7b Down fwd", 8192, 4096, 11008), ("llama7b Down dgrad", 8192, 11008, 4096),
    ("llama7b Down wgrad", 4096, 11008, 8192), ("llama7b Q fwd", 8192, 4096, 4096),
    ("llama70b Down fwd", 16384, 8192, 28672)]


def vs_cublaslt(reps: int = 20):
    """Both GEMMs timed the same way (best of back-to-back launches on one set of buffers, L2-warm,
    CUDA events), on constant operands: fp32 output, NVFP4 with E4M3 block scales and FP8 E4M3."""
    import torch
    from sub_byte_mixed_gb300 import build, snip
    build.build()
    snip.load()
    here = os.path.dirname(os.path.abspath(__file__))
    exe = os.path.join(here, "sub_byte_mixed_gb300", "_build", "cublaslt_gemm")
    os.makedirs(os.path.dirname(exe), exist_ok=True)
    subprocess.check_call([build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-o", exe,
                           os.path.join(here, "cublaslt_gemm.cu"), "-lcublasLt"])
    rows = []
    for name, M, N, K in GEMM_SHAPES:
        for fmt, fname in ((snip.NVFP4, "nvfp4"), (snip.FP8, "fp8")):
            ops = []
            for r in (M, N):
                cb, sb = snip.snip_quantized_bytes(fmt, snip.MMA, r, K)
                codes = torch.full((cb,), 0x22 if fmt == snip.NVFP4 else 0x38, dtype=torch.uint8, device="cuda")
                one = torch.ones(1, dtype=torch.float32, device="cuda")
                if fmt == snip.NVFP4:
                    scales = torch.full((sb,), 0x38, dtype=torch.uint8, device="cuda")
                    ops.append(snip.QuantNVFP4(codes, scales, one, r, K, snip.MMA))
                else:
                    ops.append(snip.QuantFP8(codes, one, r, K, snip.MMA))
            D = torch.empty((M, N), dtype=torch.float32, device="cuda")
            ws = snip.small_workspace()
            best = None
            for _ in range(3):
                snip.gemm(fmt, ops[0], ops[1], M, N, K, out=D, ws=ws)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(reps):
                    snip.gemm(fmt, ops[0], ops[1], M, N, K, out=D, ws=ws)
                e1.record()
                torch.cuda.synchronize()
                t = e0.elapsed_time(e1) / reps
                best = t if best is None else min(best, t)
            if ws.status() != snip.SNIP_OK:
                raise RuntimeError("device status " + snip.status_string(ws.status()))
            del ops, D
            torch.cuda.empty_cache()
            out = subprocess.run([exe, fname, str(M), str(N), str(K), str(reps)], capture_output=True, text=True)
            lt = json.loads(out.stdout.strip().splitlines()[-1])
            fl = 2.0 * M * N * K
            ours = fl / (best * 1e-3) / 1e12
            rows.append({"gemm": name, "fmt": fname, "M": M, "N": N, "K": K, "ours_ms": round(best, 5),
                         "ours_tflops": round(ours, 1), "cublaslt_ms": lt.get("ms"),
                         "cublaslt_tflops": lt.get("tflops"),
                         "ratio": round(ours / lt["tflops"], 3) if "tflops" in lt else None})
    print(json.dumps({"metric": "GEMM TFLOP/s, this library vs cuBLASLt (fp32 output)", "unit": "TFLOP/s",
                      "timing": f"best of 3 x {reps} back-to-back launches, same buffers (L2-warm), CUDA events",
                      "operands": "constant codes (1.0), unit scales", "rows": rows}), flush=True)


def main():
    args = parse_args()
    if args.vs_cublaslt:
        vs_cublaslt()
        return
    if args.next4_only:
        import torch
        from sub_byte_mixed_gb300 import build, snip
        build.build()
        snip.load()
        snip.snip_device_check()
        print(json.dumps(dw_noise_time(snip, measured_peaks()["bf16"])), flush=True)
        return
    if args.cpu_sample_only:
        print(json.dumps(cpu_sample(args.cpu_sample_seconds)), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if world > 1:
            os.environ.setdefault("OMP_NUM_THREADS", "1")
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    if "--impl" in sys.argv and "reference" in sys.argv:
        os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
        os.environ.setdefault("OMP_NUM_THREADS", "1")
    main()
