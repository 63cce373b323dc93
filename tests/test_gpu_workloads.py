"""Parity at the full sizes of the five workloads through moe_layer_forward
(one layer per call, all experts resident on the device, weights made by
the device generator): the single-launch decode kernel for the decode,
verify and wide workloads, the tcgen05 grouped GEMMs for the prefill chunk.
(bench.py times the decode and verify workloads as one moe_stack_forward per
step; tests/test_gpu_stack_workloads.py checks that launch.)  The oracle
recomputes sampled layers and tokens one by one from host-generated copies
of the routed experts, with the rule of oracle.parity.check_layer; bucketing
is checked bit for bit on every token."""
import gc

import numpy as np
import pytest

import oracle
import synth
from oracle import parity
from synth.workloads import WORKLOADS

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import block_quantized_routed_gb300 as m
    m.load()
    return m


def _free():
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _host_experts(wl, layer, need):
    experts = [None] * (wl.E + wl.S)
    for e in need:
        experts[e] = (synth.gen_matrix(wl.fmt, wl.I, wl.H, wl.seed, layer, e, 0),
                      synth.gen_matrix(wl.fmt, wl.I, wl.H, wl.seed, layer, e, 1),
                      synth.gen_matrix(wl.fmt, wl.H, wl.I, wl.seed, layer, e, 2))
    return experts


class Rows:
    """Row access to a device tensor (one row copied to the host per access)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, i):
        return self.t[int(i)].cpu().numpy()


def _check_layer(moe, wl, bank, layer, T, tokens=None, rep=0, tile_rows=False):
    """Run one layer on the device and compare it with the oracle on `tokens`
    (all if None); with tile_rows, also on the first and last rows of every
    token tile of some experts (the tensor-core path's tile edges)."""
    import synth.gpu  # noqa: F401
    dev = bank.buf.device
    wr = synth.router_weight(wl.E, wl.H, wl.seed, layer)
    bias = synth.router_bias(wl.E, wl.bias_std, wl.seed, layer) if wl.bias_std > 0 else None
    x = synth.activations(T, wl.H, wl.seed, layer, rep)
    lay = moe.MoeLayer(wl.desc(T), bank.table(layer), torch.from_numpy(wr).to(dev),
                       None if bias is None else torch.from_numpy(bias).to(dev), device=dev)
    xd = torch.from_numpy(x).to(dev)
    ids = torch.empty((T, wl.k), dtype=torch.int32, device=dev)
    gates = torch.empty((T, wl.k), dtype=torch.float32, device=dev)
    out = lay.forward(xd, residual=xd, ids_out=ids, gates_out=gates)
    assert moe.moe_get_status(lay.ws) == 0
    P = T * (wl.k + wl.S)
    gids = ids.cpu().numpy()
    rc, ro, _ = oracle.bucket(gids, wl.E, wl.S)
    np.testing.assert_array_equal(lay.ws_view("counts", torch.int32, (wl.E + wl.S,)).cpu().numpy(), rc)
    np.testing.assert_array_equal(lay.ws_view("offsets", torch.int32, (wl.E + wl.S + 1,)).cpu().numpy(), ro)
    perm = lay.ws_view("perm", torch.int32, (P,)).cpu().numpy()
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    if tile_rows:
        # first and last rows of the token tiles of the experts with the most tokens (and of the shared
        # expert's first tiles): c tokens form ceil(c / n) tiles of ceil(c / tiles) rows
        n = moe.moe_prefill_tile_tokens()
        edge = []
        for e in list(np.argsort(-rc[:wl.E], kind="stable")[:6]) + list(range(wl.E, wl.E + wl.S)):
            c = int(rc[e])
            per = -(-c // -(-c // n)) if c else 1
            for t0 in range(0, min(c, 3 * per), per):
                for pos in (ro[e] + t0, ro[e] + min(t0 + per, c) - 1):
                    p_ = int(perm[pos])
                    edge.append(p_ // wl.k if p_ < T * wl.k else (p_ - T * wl.k) % T)
        sel = np.unique(np.concatenate([sel, np.asarray(edge, np.int64)]))
    need = sorted(set(gids[sel].reshape(-1).tolist()) | set(range(wl.E, wl.E + wl.S)))
    experts = _host_experts(wl, layer, need)
    devd = dict(xq=lay.ws_view("xq", torch.int8, (T, wl.H)).cpu().numpy(), ids=gids, gates=gates.cpu().numpy(),
                logits=lay.ws_view("logits", torch.float32, (T, wl.E)).cpu().numpy(),
                perm=perm, h=Rows(lay.ws_view("h", torch.float32, (P, wl.I))),
                y=Rows(lay.ws_view("y", torch.float32, (P, wl.H))), out=out.cpu().numpy())
    metrics, fails = parity.check_layer(wl.fmt, wl.H, wl.I, wl.E, wl.k, wl.S, wl.route, experts, wr, bias, x, x,
                                        devd, sel)
    assert not fails, f"layer {layer}: " + "; ".join(fails[:5])
    return metrics


def test_device_generator_matches_host_generator(moe):
    import dataclasses

    import synth.gpu
    base = WORKLOADS["decode_h2048_e256k8s1_i512_q4k_l40_t1"]
    for wl in [base, WORKLOADS["verify_h4096_e512k10s1_i1024_q2k_l48_t4"]] + \
            [dataclasses.replace(base, fmt=f) for f in (synth.FMT_Q5K, synth.FMT_Q3K, synth.FMT_Q6K, synth.FMT_IQ2G)]:
        bank = synth.gpu.ExpertBank(wl.fmt, wl.H, wl.I, 3, 2, wl.seed)
        for layer, e, m in [(0, 0, 0), (1, 2, 1), (1, 1, 2)]:
            want = _host_experts(wl, layer, [e])[e][m]
            np.testing.assert_array_equal(bank.view(layer, e, m).cpu().numpy(), want)
        del bank
        _free()


def test_tiny_workload(moe):
    import synth.gpu
    wl = WORKLOADS["tiny_h512_e16k2_i256_t4"]
    bank = synth.gpu.ExpertBank(wl.fmt, wl.H, wl.I, wl.E + wl.S, wl.layers, wl.seed)
    for rep in range(4):
        _check_layer(moe, wl, bank, 0, wl.T, rep=rep)
    del bank
    _free()


def test_decode_stack_40_layers(moe):
    import synth.gpu
    wl = WORKLOADS["decode_h2048_e256k8s1_i512_q4k_l40_t1"]
    bank = synth.gpu.ExpertBank(wl.fmt, wl.H, wl.I, wl.E + wl.S, wl.layers, wl.seed)
    for layer in [0, 17, 39]:
        _check_layer(moe, wl, bank, layer, wl.T)
    del bank
    _free()


def test_verify_window_q2k_48_layers(moe):
    import synth.gpu
    wl = WORKLOADS["verify_h4096_e512k10s1_i1024_q2k_l48_t4"]
    bank = synth.gpu.ExpertBank(wl.fmt, wl.H, wl.I, wl.E + wl.S, wl.layers, wl.seed)
    for layer in [0, 47]:
        _check_layer(moe, wl, bank, layer, wl.T)
    del bank
    _free()


@pytest.mark.parametrize("T", [1, 2, 4, 8, 16])
def test_wide_experts_token_sweep(moe, T):
    import synth.gpu
    wl = WORKLOADS["wide_h6144_e192k8_i2048_q4k_t16"].with_T(T)
    bank = synth.gpu.ExpertBank(wl.fmt, wl.H, wl.I, wl.E + wl.S, wl.layers, wl.seed)
    _check_layer(moe, wl, bank, 0, T, tokens=None if T <= 4 else [0, T // 2, T - 1])
    del bank
    _free()


def test_prefill_chunk_8192(moe):
    import synth.gpu
    wl = WORKLOADS["prefill_h4096_e512k10s1_i1024_q4k_t8192"]
    bank = synth.gpu.ExpertBank(wl.fmt, wl.H, wl.I, wl.E + wl.S, wl.layers, wl.seed)
    tokens = np.unique(np.linspace(0, wl.T - 1, 64).round().astype(np.int64))
    m = _check_layer(moe, wl, bank, 0, wl.T, tokens=tokens, tile_rows=True)
    assert m["tokens"] >= 64
    print(f"\nprefill: {m}")
    del bank
    _free()
