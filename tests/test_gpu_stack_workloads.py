"""Parity of the decode stack in the launch configuration bench.py times: ONE
moe_stack_forward over every layer of a workload, with the dataflow stack
kernel, for

  the decode workload  40 layers, H 2048, 256 experts top-8 softmax + 1 shared,
                       I 512, Q4_K-style, 1 token per layer;
  the verify workload  48 layers, H 4096, 512 experts top-10 sigmoid + 1 shared,
                       I 1024, Q2_K-style, 4 tokens per layer,

each with independent layer inputs (the bench's default; the kernel overlaps
neighbouring layers) and in the chained order (some layer reads the previous
layer's output, so the kernel runs every layer after the one before it).
Layers 0, L/2 and L-1 (and 1 when chained) are compared with the oracle by
oracle.parity.check_layer, each on the input the device actually gave it:
codes, ids, bucketing bit for bit; near-ties and h-code flips counted; per-slot
y and the output within the fp32 forward-error bound; the output within 1e-3 of
the row's L2 norm of the oracle's own fp64 layer.

Chained order with real data: these synthetic weights have a non-zero mean,
so a 40-deep chain of layers with residual = x grows past fp32 within about
four layers.  The chain links are therefore the checked layers' own: layer 1
reads layer 0's output, L/2 reads L/2-1's, L-1 reads L-2's; any such link
makes the kernel take the layer-by-layer order for the whole stack."""
import gc

import numpy as np
import pytest

import synth
from oracle import parity
from synth.workloads import WORKLOADS

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DECODE = "decode_h2048_e256k8s1_i512_q4k_l40_t1"
VERIFY = "verify_h4096_e512k10s1_i1024_q2k_l48_t4"


@pytest.fixture(scope="module")
def moe():
    import block_quantized_routed_gb300 as m
    m.load()
    return m


def chain_links(L):
    """Layers whose input is the previous layer's output in the chained order."""
    return sorted({1, L // 2, L - 1})


def run_stack(moe, wl, bank, links, rotation=0):
    """One moe_stack_forward of all layers; returns (device tensors, workspace, inputs)."""
    import synth.gpu  # noqa: F401
    dev = bank.buf.device
    L, T, H = wl.layers, wl.T, wl.H
    x_host = np.stack([synth.activations(T, H, wl.seed, l, rotation) for l in range(L)])
    xs = torch.from_numpy(x_host).to(dev)
    out = torch.empty((L, T, H), dtype=torch.float32, device=dev)
    routers = [torch.from_numpy(synth.router_weight(wl.E, H, wl.seed, l)).to(dev) for l in range(L)]
    biases = [torch.from_numpy(synth.router_bias(wl.E, wl.bias_std, wl.seed, l)).to(dev) if wl.bias_std > 0
              else None for l in range(L)]
    xin = [out[l - 1] if l in links else xs[l] for l in range(L)]
    rows = [dict(table=bank.table(l), w_router=routers[l], router_bias=biases[l], x=xin[l], residual=xin[l],
                 out=out[l]) for l in range(L)]
    stack = moe.stack_pointer_table(rows, device=dev)
    desc = wl.desc(T)
    assert moe.moe_stack_kernel(desc, L, T) == moe.STACK_DATAFLOW
    ws = torch.zeros(moe.moe_stack_workspace_size(desc, L), dtype=torch.uint8, device=dev)
    moe.moe_stack_forward(desc, stack, T, ws)
    assert moe.moe_get_status(ws) == 0
    phase = moe.MoeLayer.ws_view_of(ws, moe.moe_workspace_layout(desc), "phase_ns", torch.int64, (16,))
    order = int(phase[15].item())
    assert order == (4 if links else 3), order     # 4: layer by layer, 3: neighbouring layers overlapped
    return dict(out=out, xin=xin, routers=routers, biases=biases, ws=ws, desc=desc)


class Rows:
    """Row access to a device tensor (copies one row to the host per access)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, i):
        return self.t[int(i)].cpu().numpy()


def check_stack_layer(moe, wl, run, l):
    T, H, I, k, S = wl.T, wl.H, wl.I, wl.k, wl.S
    P = T * (k + S)
    lay = moe.moe_stack_layer_layout(run["desc"], wl.layers, T, l)
    v = lambda off, dt, shape: moe.ws_view(run["ws"], off, dt, shape)
    dev = dict(xq=v(lay.xq, torch.int8, (T, H)).cpu().numpy(),
               logits=v(lay.logits, torch.float32, (T, wl.E)).cpu().numpy(),
               ids=v(lay.ids, torch.int32, (T, k)).cpu().numpy(),
               gates=v(lay.gates, torch.float32, (T, k)).cpu().numpy(),
               perm=v(lay.slot, torch.int32, (P,)).cpu().numpy(),
               h=Rows(v(lay.h, torch.float32, (P, I))), y=Rows(v(lay.y, torch.float32, (P, H))),
               out=run["out"][l].cpu().numpy())
    tok = v(lay.tok, torch.int32, (P,)).cpu().numpy()
    np.testing.assert_array_equal(tok, np.where(dev["perm"] < T * k, dev["perm"] // k, (dev["perm"] - T * k) % T))
    x = run["xin"][l].cpu().numpy()
    wr = run["routers"][l].cpu().numpy()
    bias = None if run["biases"][l] is None else run["biases"][l].cpu().numpy()
    need = sorted(set(dev["ids"].reshape(-1).tolist()) | set(range(wl.E, wl.E + wl.S)))
    experts = [None] * (wl.E + wl.S)
    for e in need:
        experts[e] = (synth.gen_matrix(wl.fmt, I, H, wl.seed, l, e, 0), synth.gen_matrix(wl.fmt, I, H, wl.seed, l, e, 1),
                      synth.gen_matrix(wl.fmt, H, I, wl.seed, l, e, 2))
    metrics, fails = parity.check_layer(wl.fmt, H, I, wl.E, k, S, wl.route, experts, wr, bias, x, x, dev,
                                        np.arange(T))
    assert not fails, f"layer {l}: " + "; ".join(fails[:5])
    return metrics


@pytest.mark.parametrize("fmt", [synth.FMT_Q5K, synth.FMT_Q3K, synth.FMT_Q6K, synth.FMT_IQ2G],
                         ids=["q5k", "q3k", "q6k", "iq2g"])
def test_decode_stack_other_formats(moe, fmt):
    """The decode workload's shape (40 layers, H 2048, 256 experts top-8 + shared, I 512, 1 token) with
    Q5_K/Q3_K/Q6_K-style or IQ2-style grid weights made on the device, as one moe_stack_forward."""
    import dataclasses

    import synth.gpu
    wl = dataclasses.replace(WORKLOADS[DECODE], fmt=fmt)
    bank = synth.gpu.ExpertBank(wl.fmt, wl.H, wl.I, wl.E + wl.S, wl.layers, wl.seed)
    run = run_stack(moe, wl, bank, [])
    L = wl.layers
    summary = parity.merge([check_stack_layer(moe, wl, run, l) for l in sorted({0, L // 2, L - 1})])
    print(f"\n{synth.layout.NAMES[fmt]} decode stack: {summary}")
    assert summary["bucket_exact"]
    del run, bank
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("chained", [False, True], ids=["independent", "chained"])
@pytest.mark.parametrize("name", [DECODE, VERIFY])
def test_stack_at_bench_shape(moe, name, chained):
    import synth.gpu
    wl = WORKLOADS[name]
    bank = synth.gpu.ExpertBank(wl.fmt, wl.H, wl.I, wl.E + wl.S, wl.layers, wl.seed)
    L = wl.layers
    links = chain_links(L) if chained else []
    run = run_stack(moe, wl, bank, links)
    layers = sorted({0, L // 2, L - 1} | ({1} if chained else set()))
    metrics = [check_stack_layer(moe, wl, run, l) for l in layers]
    summary = parity.merge(metrics)
    print(f"\n{name} {'chained' if chained else 'independent'}: {summary}")
    assert summary["bucket_exact"]
    del run, bank
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
