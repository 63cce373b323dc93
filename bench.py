#!/usr/bin/env python
"""Benchmark of the block-quantized routed MoE layer on GB300.

One step = one pass of the whole layer (q8_K quantize, router top-k,
bucketing, expert gate/up + SwiGLU + down, combine into the residual) over
every layer of the workload, for that workload's tokens per layer.  The
default workload is the Qwen3.6-35B-A3B-shaped decode stack: 40 layers,
H=2048, 256 routed experts (softmax top-8) + 1 shared expert, I=512,
Q4_K-style weights (18.2 GB resident), one token per layer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--T T]
  python bench.py --impl reference ...   (the CPU oracle, as the reference arm)

Prints one JSON line (rank 0).  With torchrun (N > 1) each rank runs an
independent replica of the workload on its own GPU (the layer has no data-path
exchange on one GPU); value = tokens of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth.workloads import DEFAULT_BENCH, WORKLOADS  # noqa: E402

METRIC = "MoE-layer decode tokens/s; active-expert HBM GB/s as fraction of GB300 peak"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: about 3 s of work)")
    ap.add_argument("--warmup", type=int, default=None, help="untimed warm-up steps (default 20, at least 3)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_BENCH, choices=sorted(WORKLOADS))
    ap.add_argument("--T", type=int, default=None, help="tokens per layer (overrides the workload's)")
    ap.add_argument("--fmt", default=None, choices=sorted(synth.layout.NAMES.values()),
                    help="weight format (overrides the workload's, e.g. iq2_g for the grid format)")
    ap.add_argument("--layers", type=int, default=None,
                    help="layers (overrides the workload's; smaller cases for profiling captures)")
    ap.add_argument("--rotations", type=int, default=16, help="distinct input sets cycled through the steps")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying a CUDA graph")
    ap.add_argument("--chained", action="store_true",
                    help="the chained order of a decode step: layers 1, L/2 and L-1 read the previous layer's "
                         "output, which makes the kernel run every layer after the one before it")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=100.0,
                    help="oracle seconds the reference arm spends in its timed steps")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_barrier():
    """Barrier across the ranks of an initialised process group (no-op for one process)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(value, device=None):
    """The largest `value` of all ranks (every rank gets it); `value` itself for one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return type(value)(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense fp16/bf16 tensor peak (TFLOP/s): the sustained cuBLAS bf16 figure (the GEMMs run inside
    seconds of back-to-back steps); fp16 and bf16 share one rate on tcgen05 kind::f16."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured (cuBLAS bf16, sustained)"
    except (OSError, KeyError, ValueError):
        return 1700.0, "fallback (sustained)"


# the files defining each profiled kernel (plus the shared headers)
KERNEL_SOURCES = {"decode_fused_kernel": ["moe_decode_kernels.cuh"], "decode_stack_kernel": ["moe_decode_kernels.cuh"],
                  "prefill_gemm_kernel": ["moe_prefill.cu"], "router_gemm_kernel": ["moe_route.cu"],
                  "gateup_kernel": ["moe_ffn.cu"]}


def code_only(src):
    """C/C++/CUDA source with its comments removed (string and character
    literals kept as they are), so that an edit of a comment does not count
    as a change of the code."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).split("\n"))


def kernel_source_hash(kernel):
    """Hash of the code (comments removed) of the sources a kernel is built
    from, to tell whether a profile still applies."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantized_routed_gb300", "csrc")
    paths = [os.path.join(csrc, f) for f in KERNEL_SOURCES[kernel] + ["moe_device.cuh", "moe_internal.h"]]
    for path in paths + [os.path.join(ROOT, "include", "moe_q8k.h")]:
        h.update(code_only(open(path, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name, kernel):
    """dram bytes per launch of `kernel` from a committed ncu summary, if its
    kernel-source hash matches the current sources (else None)."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    want = kernel_source_hash(kernel)
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md"):
            continue
        txt = open(os.path.join(pdir, f)).read()
        for m in re.finditer(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)\s+kernel:\s*(\S+)\s+workload:\s*(\S+)"
                             r"\s+source_hash:\s*(\w+)", txt, flags=re.M):
            if m.group(2) == kernel and m.group(3) == workload_name and m.group(4) == want:
                return float(m.group(1))
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def host_inputs(wl, T, R):
    """x [R, L, T, H] fp32 (rotation r, layer l)."""
    return np.stack([np.stack([synth.activations(T, wl.H, wl.seed, l, r) for l in range(wl.layers)])
                     for r in range(R)])


def chain_links(L):
    """Layers that read the previous layer's output in the chained order.

    Any one such link makes the stack kernel run every layer after the one
    before it (the order of a decode step through the stack), so the timing
    is that of a full chain.  The links are few because these synthetic
    weights have a non-zero mean: with residual = x, a deeper chain of real
    data grows past fp32 within about four layers, after which the routing
    of NaN logits degenerates to experts 0..k-1 (an unrealistic workload)."""
    return sorted({1, L // 2, L - 1}) if L > 1 else []


# ----------------------------------------------------------------------------- CPU oracle

# Tokens are independent through a layer (routing, expert FFNs and combine
# are per token), so the oracle may run a subset of a chunk's tokens and the
# result rows are exactly the chunk's rows for those tokens.
ORACLE_MAX_TOKENS = 64


def token_sample(T):
    """All tokens of small chunks; for large ones 64 tokens spread over the chunk (first and last included)."""
    if T <= ORACLE_MAX_TOKENS:
        return np.arange(T)
    return np.unique(np.linspace(0, T - 1, ORACLE_MAX_TOKENS).round().astype(np.int64))


def oracle_layers(wl, T, x_rl, layers, nthreads, tokens=None):
    """Run the oracle on the given layers of one rotation (x_rl [L, T, H]),
    on the rows `tokens` (default all); experts are generated on the host
    for the routed ones only.  Returns (outputs {layer: fp64 [len(tokens), H]},
    seconds spent in the oracle)."""
    import oracle
    outs, spent = {}, 0.0
    for l in layers:
        wr = synth.router_weight(wl.E, wl.H, wl.seed, l)
        bias = synth.router_bias(wl.E, wl.bias_std, wl.seed, l) if wl.bias_std > 0 else None
        x = x_rl[l] if tokens is None else np.ascontiguousarray(x_rl[l][tokens])
        _, ids, _, _ = oracle.route(x, wr, bias, wl.k, wl.route)
        need = sorted(set(ids.reshape(-1).tolist()) | set(range(wl.E, wl.E + wl.S)))
        experts = [None] * (wl.E + wl.S)
        for e in need:
            experts[e] = (synth.gen_matrix(wl.fmt, wl.I, wl.H, wl.seed, l, e, 0),
                          synth.gen_matrix(wl.fmt, wl.I, wl.H, wl.seed, l, e, 1),
                          synth.gen_matrix(wl.fmt, wl.H, wl.I, wl.seed, l, e, 2))
        t0 = time.perf_counter()
        out, _, _, _ = oracle.layer_forward(wl.fmt, wl.H, wl.I, wl.E, wl.k, wl.S, wl.route, experts, wr, bias, x,
                                            residual=x, nthreads=nthreads)
        spent += time.perf_counter() - t0
        outs[l] = out
    return outs, spent


def cpu_baseline(args, wl, T, budget_s):
    """The oracle timed the way the reference arm times it, in a fresh process
    (no CUDA context, no GPU-side threads), so both report one measurement."""
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--workload", args.workload,
           "--steps", "3", "--warmup", "1", "--ref-budget-s", str(budget_s)]
    if args.T:
        cmd += ["--T", str(args.T)]
    if args.layers:
        cmd += ["--layers", str(args.layers)]
    env = {k_: v for k_, v in os.environ.items() if k_ not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=max(120.0, 6 * budget_s))
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    if r.returncode != 0 or not lines:
        return {"value": None, "unit": "tokens/s", "kind": "oracle", "error": (r.stderr or "")[-300:]}
    ref = json.loads(lines[-1])
    cb = dict(ref["cpu_baseline"])
    cb["value"] = ref["value"]
    cb["how"] = "bench.py --impl reference in a child process (" + " ".join(cmd[2:]) + ")"
    return cb


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, wl, T):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    K = args.steps if args.steps is not None else 3
    W = max(args.warmup if args.warmup is not None else 1, 0)
    x_host = host_inputs(wl, T, 1)
    nthreads = oracle.default_threads()
    tokens = token_sample(T)
    # size each step's sample so that the timed steps take about --ref-budget-s
    _, t_layer = oracle_layers(wl, T, x_host[0], [0], nthreads, tokens)
    per_step = max(1, min(wl.layers * 16, int(args.ref_budget_s / max(K, 1) / max(t_layer, 1e-3))))
    for i in range(W):
        oracle_layers(wl, T, x_host[0], [(i * per_step + j) % wl.layers for j in range(per_step)], nthreads, tokens)
    spent = 0.0
    for i in range(K):
        _, s = oracle_layers(wl, T, x_host[0], [(i * per_step + j) % wl.layers for j in range(per_step)], nthreads,
                             tokens)
        spent += s
    tok_s = (K * per_step / wl.layers) * len(tokens) / spent
    line = {
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": 1e3 * spent / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (int64 sub-block sums)", "data": "synthetic",
        "config": {"workload": wl.name, "layers": wl.layers, "T": T, "sample_layers_per_step": per_step},
        "cpu_baseline": {"kind": "oracle", "cores": nthreads, "value": tok_s, "unit": "tokens/s",
                         "threads": f"{nthreads} std::thread workers per parallel loop (rows or tokens), "
                                    f"not pinned; host cores {os.cpu_count()}",
                         "sample": f"{per_step} layer evaluations per step (layers cycled over the {wl.layers} of "
                                   f"the workload), {len(tokens)} of {T} token(s) per layer, rotation 0; "
                                   f"tokens/s = evaluations / layers per step * tokens / oracle seconds"},
        "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- parity spot check

def snapshot_layers(moe, wl, T, desc, L, stacked, ws, layers, check_layers, xin, out, ids_buf):
    """Host copies of what the oracle comparison reads, for the checked layers
    of the run just made: the layer's input, its q8_K codes, routing, bucket
    order, and the h / y rows of the sampled tokens' slots."""
    import torch
    tokens = token_sample(T)
    P = T * (wl.k + wl.S)
    snap = {"tokens": tokens, "layers": {}}
    # the dataflow stack kernel keeps every layer's buffers; the pipelined one
    # (short stacks of heavy layers) keeps a single layer's in the layer
    # workspace at the start of the stack workspace
    per_layer = stacked and moe.moe_stack_kernel(desc, L, T) == moe.STACK_DATAFLOW
    if stacked and not per_layer:
        if L > 1:
            return None
        layout = moe.moe_workspace_layout(desc)

        class _One:
            def ws_view(self, name, dt, shape):
                return moe.MoeLayer.ws_view_of(ws, layout, name, dt, shape)
        layers = [_One()]
    for l in check_layers:
        if per_layer:
            lay = moe.moe_stack_layer_layout(desc, L, T, l)
            v = lambda off, dt, shape: moe.ws_view(ws, off, dt, shape)
            xq, ids, gates = v(lay.xq, torch.int8, (T, wl.H)), v(lay.ids, torch.int32, (T, wl.k)), \
                v(lay.gates, torch.float32, (T, wl.k))
            logits = v(lay.logits, torch.float32, (T, wl.E))
            perm, h, y = v(lay.slot, torch.int32, (P,)), v(lay.h, torch.float32, (P, wl.I)), \
                v(lay.y, torch.float32, (P, wl.H))
        else:
            ly = layers[l]
            xq, gates = ly.ws_view("xq", torch.int8, (T, wl.H)), ly.ws_view("gates", torch.float32, (T, wl.k))
            logits = ly.ws_view("logits", torch.float32, (T, wl.E))
            ids = ids_buf[l]
            perm, h, y = ly.ws_view("perm", torch.int32, (P,)), ly.ws_view("h", torch.float32, (P, wl.I)), \
                ly.ws_view("y", torch.float32, (P, wl.H))
        perm_h = perm.cpu().numpy()
        inv = np.empty(P, np.int64)
        inv[perm_h] = np.arange(P)
        slots = sorted({int(t) * wl.k + s_ for t in tokens for s_ in range(wl.k)} |
                       {T * wl.k + sh * T + int(t) for t in tokens for sh in range(wl.S)})
        sl = torch.as_tensor(slots, device=h.device, dtype=torch.int64)
        hrows = h.index_select(0, torch.as_tensor(inv[slots], device=h.device)).cpu().numpy()
        yrows = y.index_select(0, sl).cpu().numpy()
        snap["layers"][l] = dict(x=xin(l).cpu().numpy(), xq=xq.cpu().numpy(), ids=ids.cpu().numpy(),
                                 gates=gates.cpu().numpy(), logits=logits.cpu().numpy(), perm=perm_h,
                                 out=out[l].cpu().numpy(),
                                 h={int(inv[p]): hrows[i] for i, p in enumerate(slots)},
                                 y={p: yrows[i] for i, p in enumerate(slots)})
    return snap


def spot_check(wl, T, snap):
    """The oracle comparison rule of the parity tests (oracle.parity) on the
    snapshot: codes, ids, bucketing exact; near-ties and h-code flips counted;
    y and out within the fp32 forward-error bound; out within 1e-3 of the
    row's L2 norm of the oracle's own layer."""
    from oracle import parity
    if snap is None:
        return {"skipped": "the pipelined kernel of a multi-layer stack keeps no per-layer buffers"}
    t0 = time.perf_counter()
    metrics, fails = [], []
    for l, d in snap["layers"].items():
        wr = synth.router_weight(wl.E, wl.H, wl.seed, l)
        bias = synth.router_bias(wl.E, wl.bias_std, wl.seed, l) if wl.bias_std > 0 else None
        tokens = snap["tokens"]
        need = sorted(set(d["ids"][tokens].reshape(-1).tolist()) | set(range(wl.E, wl.E + wl.S)))
        experts = [None] * (wl.E + wl.S)
        for e in need:
            experts[e] = (synth.gen_matrix(wl.fmt, wl.I, wl.H, wl.seed, l, e, 0),
                          synth.gen_matrix(wl.fmt, wl.I, wl.H, wl.seed, l, e, 1),
                          synth.gen_matrix(wl.fmt, wl.H, wl.I, wl.seed, l, e, 2))
        m, f = parity.check_layer(wl.fmt, wl.H, wl.I, wl.E, wl.k, wl.S, wl.route, experts, wr, bias, d["x"],
                                  d["x"], d, tokens)
        metrics.append(m)
        fails += [f"layer {l}: {x}" for x in f]
    out = parity.merge(metrics)
    out.update({"layers": sorted(snap["layers"]), "failures": len(fails), "first_failures": fails[:3],
                "seconds": round(time.perf_counter() - t0, 1),
                "rule": "oracle/parity.py: exact codes/ids/bucketing; y, out within the fp32 forward-error bound; "
                        "out within 1e-3 of the row L2 norm"})
    return out


# ----------------------------------------------------------------------------- our arm

def run_ours(args, wl, T):
    import torch

    import block_quantized_routed_gb300 as moe
    import synth.gpu

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    moe.load()
    L, H, R = wl.layers, wl.H, args.rotations
    bank = synth.gpu.ExpertBank(wl.fmt, wl.H, wl.I, wl.E + wl.S, L, wl.seed, device=dev)
    routers = [torch.from_numpy(synth.router_weight(wl.E, H, wl.seed, l)).to(dev) for l in range(L)]
    biases = [torch.from_numpy(synth.router_bias(wl.E, wl.bias_std, wl.seed, l)).to(dev) if wl.bias_std > 0 else None
              for l in range(L)]
    tables = [bank.table(l) for l in range(L)]
    x_host = host_inputs(wl, T, R)
    xs = torch.from_numpy(x_host).to(dev)                      # [R, L, T, H]
    x_static = torch.empty((L, T, H), dtype=torch.float32, device=dev)
    out = torch.empty((L, T, H), dtype=torch.float32, device=dev)
    ids_buf = torch.empty((L, T, wl.k), dtype=torch.int32, device=dev)
    desc = wl.desc(T)
    ws = torch.zeros(max(moe.moe_layer_workspace_size(desc), moe.moe_stack_workspace_size(desc, L)),
                     dtype=torch.uint8, device=dev)
    links = chain_links(L) if args.chained else []

    def xin(l):  # layer l's input (and residual)
        return out[l - 1] if l in links else x_static[l]

    rows = [dict(table=tables[l], w_router=routers[l], router_bias=biases[l], x=xin(l), residual=xin(l),
                 out=out[l], ids_out=ids_buf[l]) for l in range(L)]
    stack = moe.stack_pointer_table(rows, device=dev)
    # the single-launch stack serves decode shapes; other shapes run layer by layer
    try:
        x_static.copy_(xs[0])
        moe.moe_stack_forward(desc, stack, T, ws)
        stacked = True
    except moe.MoeError as err:
        if err.status != moe.MOE_ERR_UNSUPPORTED:
            raise
        stacked = False
        layers = [moe.MoeLayer(desc, tables[l], routers[l], biases[l], device=dev) for l in range(L)]
    torch.cuda.synchronize()
    path = moe.moe_layer_path(desc, T)

    def body():
        if stacked:
            moe.moe_stack_forward(desc, stack, T, ws)
        else:
            for l in range(L):
                layers[l].forward(xin(l), residual=xin(l), out=out[l], ids_out=ids_buf[l])

    # unique active experts per layer for every rotation (counted from the routing)
    union = np.zeros((R, L), np.int64)
    for r in range(R):
        x_static.copy_(xs[r])
        body()
        ids = ids_buf.cpu().numpy()
        for l in range(L):
            union[r, l] = len(set(ids[l].reshape(-1).tolist())) + wl.S
    for w_ in ([ws] if stacked else [ly.ws for ly in layers]):
        st = moe.moe_get_status(w_)
        if st != 0:
            raise RuntimeError(f"device status {moe.moe_status_string(st)}")
    x_static.copy_(xs[0])
    body()
    torch.cuda.synchronize()
    # device results of rotation 0 on the layers the parity spot check compares
    check_layers = sorted({0, L // 2, L - 1} | ({1} if links else set()))
    snap = snapshot_layers(moe, wl, T, desc, L, stacked, ws if stacked else None,
                           None if stacked else layers, check_layers, xin, out, ids_buf)

    # CUDA graphs of one step, one per input rotation: each reads its rotation's
    # inputs where they already sit in HBM (no copy inside the timed steps),
    # with trace events around the expert launches
    def body_rot(r):
        def xin_r(l):
            return out[l - 1] if l in links else xs[r][l]
        if stacked:
            rows_r = [dict(table=tables[l], w_router=routers[l], router_bias=biases[l], x=xin_r(l),
                           residual=xin_r(l), out=out[l], ids_out=ids_buf[l]) for l in range(L)]
            tab = moe.stack_pointer_table(rows_r, device=dev)
            return lambda: moe.moe_stack_forward(desc, tab, T, ws)

        def run_layers():
            for l in range(L):
                layers[l].forward(xin_r(l), residual=xin_r(l), out=out[l], ids_out=ids_buf[l])
        return run_layers

    events = [torch.cuda.Event(enable_timing=True) for _ in range(4 * L)]
    use_graph = not args.no_graph
    graphs = []
    rot_bodies = []                      # keep each rotation's pointer table alive with its graph
    launches_per_step = n_traced = 0
    if use_graph:
        for r in range(R):
            body_r = body_rot(r)
            rot_bodies.append(body_r)
            moe.moe_trace_events(events)
            n_launch0 = moe.moe_kernel_launch_count()
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_):
                body_r()
            if r == 0:
                launches_per_step = moe.moe_kernel_launch_count() - n_launch0   # this library's kernels in one step
                n_traced = moe.moe_trace_used()
            moe.moe_trace_events(None)
            graphs.append(g_)
    else:
        moe.moe_trace_events(events)
        n_launch0 = moe.moe_kernel_launch_count()
        body()
        launches_per_step = moe.moe_kernel_launch_count() - n_launch0
        n_traced = moe.moe_trace_used()
        moe.moe_trace_events(None)

    stream = torch.cuda.current_stream()

    eager_traced = [n_traced]

    def step(i):
        if use_graph:
            graphs[i % R].replay()
        else:
            x_static.copy_(xs[i % R], non_blocking=True)
            moe.moe_trace_events(events)
            body()
            eager_traced[0] = moe.moe_trace_used()
            moe.moe_trace_events(None)

    W = max(3, args.warmup if args.warmup is not None else 20)
    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(5):
        step(i)
    torch.cuda.synchronize()
    t_step = (time.perf_counter() - t0) / 5
    K = args.steps if args.steps is not None else int(min(20000, max(20, 3.0 / max(t_step, 1e-6))))
    K = max_over_ranks(K, dev)          # every rank times the same number of steps

    clocks = ClockSampler(local)
    rank_barrier()
    torch.cuda.synchronize()
    clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(K):
        step(W + i)
    ev1.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    rank_barrier()
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), dev)
    ms_step = ms_total / K

    # phase stamps (SM cycles of CTA 0) of the single-launch kernel's last layer
    phases = None
    phase_ws = ws if stacked else layers[-1].ws
    st = moe.MoeLayer.ws_view_of(phase_ws, moe.moe_workspace_layout(desc), "phase_ns", torch.int64, (16,)).cpu().numpy()
    ran = int(st[15])  # which single-launch kernel ran a stack: 3/4 dataflow, 1/2 pipelined
    if path == moe.PATH_TENSOR_PREFILL:
        # wait statistics of the GEMMs' CTA 0 (SM cycles): per role, then the CTA's total
        mhz = clock_info.get("sm_mhz") or 2070.0
        names = ["producer_wait_raw_slot", "producer_wait_act_slot", "expander_wait_raw", "expander_wait_slot",
                 "mma_wait_accum", "mma_wait_operands", "epilogue_wait_accum", "cta_total"]
        phases = {"schedule": "prefill_gemm_waits",
                  "gate_up": {n: round(float(v) / mhz, 1) for n, v in zip(names, st[0:8])},
                  "down": {n: round(float(v) / mhz, 1) for n, v in zip(names, st[8:16])}}
        st = np.zeros(16, np.int64)
    if stacked and st[15] in (3, 4):
        # per item kind of the stack kernel, summed over CTAs: work and wait cycles, items
        mhz = clock_info.get("sm_mhz") or 2070.0
        kinds = ["router", "routing", "gate_up", "down", "combine"]
        G_ = int(st[14])  # CTAs of the launch
        us = lambda v: round(float(v) / mhz, 1)
        phases = {"schedule": "stack_items_" + ("overlapped" if st[15] == 3 else "chained"),
                  "cta_us_summed_over_ctas": {**{f"work_{n}": us(st[k_]) for k_, n in enumerate(kinds)},
                                              **{f"wait_{n}": us(st[5 + k_]) for k_, n in enumerate(kinds)},
                                              "prologue": us(st[10]), "before_first_item": us(st[11]),
                                              "between_items": us(st[12])},
                  "items": int(st[13]), "ctas": G_}
        st = np.zeros(16, np.int64)
    if st[15] == 2:   # pipelined schedule: one stage
        order = [0, 3, 4, 6, 1, 8, 12]
        names = ["stage_x", "gate_up", "down_prev", "router_next2", "combine_prev2", "wait_route_next+prefetch"]
    else:
        order = [0, 1, 2, 9, 10, 11, 3, 4, 5, 6, 7, 8]
        names = ["router+quant", "barrier1", "topk+stage", "counts+scan", "positions", "tile_plan", "gate_up",
                 "barrier2", "down", "barrier3", "combine"]
    seq = st[order].astype(np.float64)
    if seq[0] > 0 and (np.diff(seq) >= 0).all():
        mhz = clock_info.get("sm_mhz") or 2070.0
        phases = {n: round(float(v) / mhz, 3) for n, v in zip(names, np.diff(seq))}
        phases["schedule"] = "pipelined" if st[15] == 2 else "sequential"

    # bytes
    gu_bytes = synth.layout.matrix_bytes(wl.fmt, wl.I, wl.H)
    dn_bytes = synth.layout.matrix_bytes(wl.fmt, wl.H, wl.I)
    exp_bytes = 2 * gu_bytes + dn_bytes
    steps_rot = [(W + i) % R for i in range(K)]
    active_bytes_total = float(sum(union[r].sum() for r in steps_rot)) * exp_bytes
    active_gbs = active_bytes_total / (ms_total * 1e-3) / 1e9
    last_r = (W + K - 1) % R
    peak, peak_src = measured_peaks()
    router_bytes = wl.E * wl.H * 4
    traced = n_traced if use_graph else eager_traced[0]
    if traced < (2 if stacked else 2 * L) or (not stacked and traced not in (2 * L, 4 * L)):
        raise RuntimeError(f"the launch trace recorded {traced} events; the roofline needs every launch bracketed")
    if stacked:
        # one launch per step moves every layer's router weights and active experts' 3 matrices
        launch_ms = events[0].elapsed_time(events[1])
        alg = float(union[last_r].sum() * exp_bytes + L * router_bytes)
        gbs = alg / (launch_ms * 1e-3) / 1e9
        kname = "decode_stack_kernel" if ran in (3, 4) else "decode_fused_kernel"
        roofline = {"bound": "hbm", "kernel": f"{kname} (all layers of a step, one cooperative launch)",
                    "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak, "peak_source": peak_src,
                    "traffic": profiled_traffic(wl.name, kname),
                    "algorithmic_bytes_per_launch": alg, "avg_launch_us": 1e3 * launch_ms}
    elif path == moe.PATH_TENSOR_PREFILL:
        # the tcgen05 gate/up GEMM (+ SwiGLU) is the dominant kernel; a contraction: tensor-bound
        gu_ms = [events[4 * l].elapsed_time(events[4 * l + 1]) for l in range(L)]
        dn_ms = [events[4 * l + 2].elapsed_time(events[4 * l + 3]) for l in range(L)]
        rows = T * (wl.k + wl.S)                      # bucket rows: every expert is present
        gu_flop = 2.0 * rows * 2 * wl.I * wl.H
        dn_flop = 2.0 * rows * wl.H * wl.I
        tpeak, tpeak_src = measured_tensor_peak()
        gu_tf = gu_flop / (float(np.mean(gu_ms)) * 1e-3) / 1e12
        dn_tf = dn_flop / (float(np.mean(dn_ms)) * 1e-3) / 1e12
        roofline = {"bound": "tensor",
                    "kernel": "prefill_gemm_kernel<gate/up> (tcgen05 kind::f16 grouped GEMM + SwiGLU)",
                    "achieved": gu_tf, "peak": tpeak, "unit": "TFLOP/s", "frac": gu_tf / tpeak,
                    "peak_source": tpeak_src, "traffic": profiled_traffic(wl.name, "prefill_gemm_kernel"),
                    "algorithmic_flops_per_launch": gu_flop, "avg_launch_us": 1e3 * float(np.mean(gu_ms)),
                    "down_kernel_tflops": dn_tf, "down_avg_launch_us": 1e3 * float(np.mean(dn_ms)),
                    "down_frac": dn_tf / tpeak}
    else:
        per_layer = traced // L
        if per_layer == 2:
            fz_ms = [events[2 * l].elapsed_time(events[2 * l + 1]) for l in range(L)]
            alg = union[last_r] * exp_bytes + router_bytes
            gbs = float(np.sum(alg) / (np.sum(fz_ms) * 1e-3) / 1e9)
            roofline = {"bound": "hbm", "kernel": "decode_fused_kernel (one layer, one cooperative launch)",
                        "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak, "peak_source": peak_src,
                        "traffic": profiled_traffic(wl.name, "decode_fused_kernel"),
                        "algorithmic_bytes_per_launch": float(np.mean(alg)), "avg_launch_us": 1e3 * float(np.mean(fz_ms))}
        else:
            gu_ms = [events[4 * l].elapsed_time(events[4 * l + 1]) for l in range(L)]
            dn_ms = [events[4 * l + 2].elapsed_time(events[4 * l + 3]) for l in range(L)]
            gu_alg = union[last_r] * 2 * gu_bytes
            dn_alg = union[last_r] * dn_bytes
            gu_gbs = float(np.sum(gu_alg) / (np.sum(gu_ms) * 1e-3) / 1e9)
            dn_gbs = float(np.sum(dn_alg) / (np.sum(dn_ms) * 1e-3) / 1e9)
            roofline = {"bound": "hbm", "kernel": "gateup_kernel (expert gate/up GEMV + SwiGLU + q8_K requant)",
                        "achieved": gu_gbs, "peak": peak, "unit": "GB/s", "frac": gu_gbs / peak,
                        "peak_source": peak_src, "traffic": profiled_traffic(wl.name, "gateup_kernel"),
                        "algorithmic_bytes_per_launch": float(np.mean(gu_alg)),
                        "avg_launch_us": 1e3 * float(np.mean(gu_ms)),
                        "down_kernel_gbs": dn_gbs, "down_avg_launch_us": 1e3 * float(np.mean(dn_ms))}

    # end to end through the public call with host buffers, every step: a
    # pinned H2D copy of the step's inputs, the C-ABI call(s) themselves
    # (argument checks and launches on the host, no graph replay), and a D2H
    # copy of the outputs.  Two input and two output buffers: a step's H2D
    # copy (one copy stream) and the previous step's D2H copy (another) run
    # while the step before computes; the steps themselves run in order on
    # the compute stream, sharing one workspace.
    x_pinned = torch.from_numpy(x_host).pin_memory()
    out_pinned = [torch.empty((L, T, H), dtype=torch.float32).pin_memory() for _ in range(2)]
    xb = [x_static, torch.empty_like(x_static)]
    ob = [out, torch.empty_like(out)]
    ib = [ids_buf, torch.empty_like(ids_buf)]

    def make_body(j):
        def xin_j(l):
            return ob[j][l - 1] if l in links else xb[j][l]
        if stacked:
            if j == 0:
                tab = stack
            else:
                rows_j = [dict(table=tables[l], w_router=routers[l], router_bias=biases[l], x=xin_j(l),
                               residual=xin_j(l), out=ob[j][l], ids_out=ib[j][l]) for l in range(L)]
                tab = moe.stack_pointer_table(rows_j, device=dev)
            return lambda: moe.moe_stack_forward(desc, tab, T, ws)

        def run_layers():
            for l in range(L):
                layers[l].forward(xin_j(l), residual=xin_j(l), out=ob[j][l], ids_out=ib[j][l])
        return run_layers

    bodies = [make_body(0), make_body(1)]
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    Ke = max(10, min(K, 2000))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    h2d_s.wait_event(e0)
    for i in range(Ke):
        j = i % 2
        with torch.cuda.stream(h2d_s):
            if i >= 2:
                h2d_s.wait_event(comp_done[j])        # step i - 2 has read xb[j]
            xb[j].copy_(x_pinned[i % R], non_blocking=True)
            h2d_done[j].record(h2d_s)
        stream.wait_event(h2d_done[j])
        if i >= 2:
            stream.wait_event(d2h_done[j])            # the D2H of step i - 2 has read ob[j]
        bodies[j]()
        comp_done[j].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(comp_done[j])
            out_pinned[j].copy_(ob[j], non_blocking=True)
            d2h_done[j].record(d2h_s)
    stream.wait_event(d2h_done[(Ke - 1) % 2])
    stream.wait_event(d2h_done[Ke % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / Ke
    h2d = L * T * H * 4
    d2h = L * T * H * 4

    tokens_per_step = T * world
    value = tokens_per_step / (ms_step * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("int8 codes x (scale*code) as exact fp16 integers on tcgen05 kind::f16 -> fp32"
                  if path == moe.PATH_TENSOR_PREFILL else "int8 x int4/int2 -> int32 (dp4a) + fp32"),
        "data": "synthetic",
        "config": {"workload": wl.name, "layers": L, "T": T, "H": wl.H, "I": wl.I, "E": wl.E, "top_k": wl.k,
                   "n_shared": wl.S, "route": ["softmax", "sigmoid"][wl.route], "fmt": synth.layout.NAMES[wl.fmt],
                   "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2: each step streams %.0f MB of distinct expert weights "
                         "plus %.0f MB of router weights (L2 129 MB)" % (
                             np.mean(union.sum(axis=1)) * exp_bytes / 1e6, L * wl.E * wl.H * 4 / 1e6),
                   "graph": use_graph, "rotations": R, "single_launch_stack": stacked,
                   "timed_step": ("replay of one CUDA graph per input rotation; each graph reads its rotation's "
                                  "inputs where they sit in HBM" if use_graph else
                                  "device copy of the rotation's inputs, then the eager launches"),
                   "layer_inputs": (f"chained order (layers {links} read the previous layer's output)"
                                    if links else "independent"),
                   "path": ["decode_fused", "gemv", "tensor_prefill"][path]},
        "clocks": clock_info,
        "us_per_layer": 1e3 * ms_step / L,
        "active_expert_bytes_per_step": active_bytes_total / K,
        "active_expert_gbs": active_gbs,
        "active_frac_of_8tbs": active_gbs / NOMINAL_HBM_GBS,
        "active_frac_of_measured": active_gbs / peak,
        "roofline": roofline,
        "decode_phases_us": phases,
        "e2e": {"value": tokens_per_step / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "how": "per step: pinned H2D of x, the C-ABI call through the binding (no graph), D2H of out; "
                       "two buffers each way, copies on two copy streams overlapping the previous step"},
        "gpu_launches": launches_per_step * K,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, wl, T, args.cpu_budget_s)
        # parity spot check of the bench's own launch (rotation 0) on layers 0, L/2, L-1
        line["parity"] = spot_check(wl, T, snap)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    wl = WORKLOADS[args.workload]
    T = args.T or wl.T
    if args.T:
        wl = wl.with_T(T)
    if args.fmt:
        import dataclasses
        fmt = {v: k for k, v in synth.layout.NAMES.items()}[args.fmt]
        old = synth.layout.NAMES[wl.fmt].replace("_", "")
        wl = dataclasses.replace(wl, fmt=fmt, name=wl.name.replace(old, args.fmt.replace("_", "")))
    if args.layers:
        import dataclasses
        wl = dataclasses.replace(wl, layers=args.layers, name=f"{wl.name}_l{args.layers}")
    if args.impl == "reference":
        run_reference(args, wl, T)
    else:
        run_ours(args, wl, T)


if __name__ == "__main__":
    main()
