"""The comparison rule of the parity tests (oracle/parity.py), on the CPU.

A "device" result is assembled from the oracle's own pieces (fp32 gates, h,
per-slot y and the layer output rounded to fp32, as a device would store
them), and must pass with no h-code flip; then single planted mistakes of the
kinds a kernel could make (a dropped min term in one slot, a swapped expert
id, a wrong bucket position, a wrong gate, an output off by a few units in
its last place beyond the fp32 bound) must each be reported."""
import numpy as np
import pytest

import oracle
import synth
from oracle import parity
from synth.layout import FMT_Q4K, FMT_Q2K


def _layer(fmt, H, I, E, k, S, T, seed, route_kind=0, scale=1.0):
    experts = [(synth.gen_matrix(fmt, I, H, seed, 0, e, 0), synth.gen_matrix(fmt, I, H, seed, 0, e, 1),
                synth.gen_matrix(fmt, H, I, seed, 0, e, 2)) for e in range(E + S)]
    wr = synth.router_weight(E, H, seed)
    x = (synth.activations(T, H, seed) * np.float32(scale)).astype(np.float32)
    return experts, wr, x


def _device_like(fmt, H, I, E, k, S, route_kind, experts, wr, x):
    """What a correct device would hold: fp32 results of the oracle's steps."""
    T = x.shape[0]
    _, ids, gates, _ = oracle.route(x, wr, None, k, route_kind)
    _, _, perm = oracle.bucket(ids, E, S)
    P = T * (k + S)
    xq, xd, _ = oracle.q8k_quantize(x)
    h = np.zeros((P, I), np.float32)
    y = np.zeros((P, H), np.float32)
    inv = np.empty(P, np.int64)
    inv[perm] = np.arange(P)
    for t in range(T):
        pairs = [(t * k + s, ids[t, s]) for s in range(k)] + [(T * k + sh * T + t, E + sh) for sh in range(S)]
        for p, e in pairs:
            yy, hh, _, _ = oracle.expert_ffn(*experts[e], fmt, H, I, xq[t:t + 1], xd[t:t + 1], return_h=True)
            h[inv[p]] = hh[0]
            y[p] = yy[0].astype(np.float32)
    out, _, _, _ = oracle.layer_forward(fmt, H, I, E, k, S, route_kind, experts, wr, None, x, residual=x)
    return dict(xq=xq, ids=ids, gates=gates.astype(np.float32), perm=perm.astype(np.int32), h=h, y=y,
                out=out.astype(np.float32))


CASES = [(FMT_Q4K, 512, 256, 16, 2, 0, 4, 0), (FMT_Q2K, 512, 256, 16, 4, 1, 3, 1)]


@pytest.mark.parametrize("fmt,H,I,E,k,S,T,route_kind", CASES)
def test_oracle_made_result_passes(fmt, H, I, E, k, S, T, route_kind):
    experts, wr, x = _layer(fmt, H, I, E, k, S, T, 7, route_kind)
    dev = _device_like(fmt, H, I, E, k, S, route_kind, experts, wr, x)
    m, fails = parity.check_layer(fmt, H, I, E, k, S, route_kind, experts, wr, None, x, x, dev, np.arange(T))
    assert fails == []
    assert m["h_code_flips"] == 0 and m["h_scale_flips"] == 0 and m["near_ties"] == 0 and m["bucket_exact"]
    assert m["h_codes"] == T * (k + S) * I
    assert m["max_rel_l2_err"] < 1e-7


def _fails_after(mutate, case=CASES[1]):
    fmt, H, I, E, k, S, T, route_kind = case
    experts, wr, x = _layer(fmt, H, I, E, k, S, T, 7, route_kind)
    dev = _device_like(fmt, H, I, E, k, S, route_kind, experts, wr, x)
    mutate(dev, dict(experts=experts, wr=wr, x=x, fmt=fmt, H=H, I=I, E=E, k=k, S=S, T=T))
    _, fails = parity.check_layer(fmt, H, I, E, k, S, route_kind, experts, wr, None, x, x, dev, np.arange(T))
    return fails


def test_dropped_min_term_in_one_slot_is_reported():
    def mutate(dev, c):
        # row 0 of slot 1 (token 0) computed without the dmin * min term of its first super-block
        fmt, H, I = c["fmt"], c["H"], c["I"]
        gate, up, down = c["experts"][int(dev["ids"][0, 1])]
        xq, xd, _ = oracle.q8k_quantize(c["x"][:1])
        _, _, hq, hd = oracle.expert_ffn(gate, up, down, fmt, H, I, xq, xd, return_h=True)
        _, _, mn, _, dmin = oracle.unpack_sb(down, fmt, H, I, 0, 0)
        bsum = hq[0, :256].astype(np.int64).reshape(len(mn), -1).sum(axis=1)
        term = float(hd[0, 0]) * dmin * float((mn * bsum).sum())
        assert term != 0.0
        dev["y"][1, 0] += np.float32(term)
    fails = _fails_after(mutate)
    assert any(f.startswith("y of token 0 slot 1") for f in fails)


def test_swapped_expert_id_is_reported():
    def mutate(dev, c):
        dev["ids"][0, [0, 1]] = dev["ids"][0, [1, 0]]
    fails = _fails_after(mutate)
    assert any("routing differs" in f for f in fails)


def test_wrong_bucket_position_is_reported():
    def mutate(dev, c):
        dev["perm"][[0, 1]] = dev["perm"][[1, 0]]
    fails = _fails_after(mutate)
    assert any("bucket order" in f for f in fails)


def test_wrong_gate_is_reported():
    def mutate(dev, c):
        dev["gates"][1, 0] *= np.float32(1.001)
    fails = _fails_after(mutate)
    assert any(f.startswith("gate of token 1 slot 0") for f in fails)


def test_output_beyond_fp32_bound_is_reported():
    def mutate(dev, c):
        i = int(np.argmax(np.abs(dev["out"][2])))
        dev["out"][2, i] += np.float32(64 * np.spacing(np.abs(dev["out"][2, i])) * 64)
    fails = _fails_after(mutate)
    assert any(f.startswith("out of token 2") for f in fails)


def test_bound_is_below_1e4_for_small_outputs():
    """With x scaled down the outputs are small, and the fp32 bound is far tighter than 1e-4."""
    fmt, H, I, E, k, S, T, route_kind = CASES[1]
    experts, wr, x = _layer(fmt, H, I, E, k, S, T, 7, route_kind, scale=1e-2)
    dev = _device_like(fmt, H, I, E, k, S, route_kind, experts, wr, x)
    dev["out"][0, 5] += np.float32(5e-5)
    _, fails = parity.check_layer(fmt, H, I, E, k, S, route_kind, experts, wr, None, x, x, dev, np.arange(T))
    assert any(f.startswith("out of token 0 elt 5") for f in fails)
