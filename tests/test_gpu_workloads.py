"""Parity at the full sizes of the five workloads, in the launch configuration
bench.py times (one MoeLayer per layer, all experts resident on the device,
weights made by the device generator).  The oracle recomputes sampled layers
and sampled tokens one by one from host-generated copies of the routed
experts; bucketing is checked bit for bit on every token."""
import gc

import numpy as np
import pytest

import oracle
import synth
from synth.workloads import WORKLOADS
from tests.gpu_util import assert_close_rows, routing_ok

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


def _check_layer(moe, wl, bank, layer, T, tokens=None, rep=0):
    """Run one layer on the device, compare ids/gates/bucketing (all tokens) and
    outputs of `tokens` (all if None) with the oracle."""
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
    gids = ids.cpu().numpy()
    # bucketing of every token, bit for bit, from the device's own ids
    P = T * (wl.k + wl.S)
    rc, ro, rp = oracle.bucket(gids, wl.E, wl.S)
    np.testing.assert_array_equal(lay.ws_view("counts", torch.int32, (wl.E + wl.S,)).cpu().numpy(), rc)
    np.testing.assert_array_equal(lay.ws_view("offsets", torch.int32, (wl.E + wl.S + 1,)).cpu().numpy(), ro)
    np.testing.assert_array_equal(lay.ws_view("perm", torch.int32, (P,)).cpu().numpy(), rp)
    # q8_K codes of every token, bit for bit
    xq = lay.ws_view("xq", torch.int8, (T, wl.H)).cpu().numpy()
    rq, rd, _ = oracle.q8k_quantize(x)
    np.testing.assert_array_equal(xq, rq)
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    rl, rids, _, rgap = oracle.route(x[sel], wr, bias, wl.k, wl.route)
    near = routing_ok(gids[sel], rids, rgap, rl)
    need = sorted(set(gids[sel].reshape(-1).tolist()) | set(range(wl.E, wl.E + wl.S)))
    experts = _host_experts(wl, layer, need)
    ref, _, rg, _ = oracle.layer_forward(wl.fmt, wl.H, wl.I, wl.E, wl.k, wl.S, wl.route, experts, wr, bias, x[sel],
                                         residual=x[sel], forced_ids=gids[sel])
    np.testing.assert_allclose(gates.cpu().numpy()[sel], rg, rtol=1e-5, atol=1e-6)
    assert_close_rows(out.cpu().numpy()[sel], ref, f"layer {layer}")
    return near


def test_device_generator_matches_host_generator(moe):
    import synth.gpu
    for wl_name in ["decode_h2048_e256k8s1_i512_q4k_l40_t1", "verify_h4096_e512k10s1_i1024_q2k_l48_t4"]:
        wl = WORKLOADS[wl_name]
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
    _check_layer(moe, wl, bank, 0, wl.T, tokens=[0, 1, 4095, 8191])
    del bank
    _free()
