"""Layer-level pins of the oracle (CPU only): brute-force dense evaluation,
shared-expert and residual linearity, NULL experts, and SwiGLU on weights
constructed so that every matmul has a closed form."""
import numpy as np
import pytest

import oracle
import synth
from synth.layout import FMT_Q4K, FMT_Q2K
from tests import fieldpack


def _experts(fmt, E, H, I, seed, layer=0):
    return [(synth.gen_matrix(fmt, I, H, seed, layer, e, 0), synth.gen_matrix(fmt, I, H, seed, layer, e, 1),
             synth.gen_matrix(fmt, H, I, seed, layer, e, 2)) for e in range(E)]


@pytest.mark.parametrize("fmt,route_kind,S", [(FMT_Q4K, 0, 0), (FMT_Q2K, 1, 1), (FMT_Q4K, 1, 1)])
def test_sparse_equals_dense_with_unselected_gates_zeroed(fmt, route_kind, S):
    E, H, I, k, T = 8, 256, 256, 3, 3
    ex = _experts(fmt, E + S, H, I, seed=7)
    wr = synth.router_weight(E, H, 7)
    x = synth.activations(T, H, 7)
    out, ids, gates, _ = oracle.layer_forward(fmt, H, I, E, k, S, route_kind, ex, wr, None, x)
    xq, xd, _ = oracle.q8k_quantize(x)
    dense = np.zeros((T, H))
    for e in range(E + S):
        y = oracle.expert_ffn(*ex[e], fmt, H, I, xq, xd)
        if e < E:
            g = np.zeros(T)
            for t in range(T):
                hit = np.nonzero(ids[t] == e)[0]
                if hit.size:
                    g[t] = gates[t, hit[0]]
        else:
            g = np.ones(T)
        dense += g[:, None] * y
    np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-12 * np.abs(dense).max())


def test_shared_expert_and_residual_linearity():
    fmt, E, H, I, k, T = FMT_Q4K, 6, 512, 256, 2, 2
    ex = _experts(fmt, E + 1, H, I, seed=9)
    wr = synth.router_weight(E, H, 9)
    x = synth.activations(T, H, 9)
    res = synth.normal_f32((T, H), 1.0, 9, synth.TAG_RESIDUAL)
    out1, ids1, g1, _ = oracle.layer_forward(fmt, H, I, E, k, 1, 0, ex, wr, None, x, residual=res)
    out0, ids0, g0, _ = oracle.layer_forward(fmt, H, I, E, k, 0, 0, ex[:E], wr, None, x)
    np.testing.assert_array_equal(ids0, ids1)
    xq, xd, _ = oracle.q8k_quantize(x)
    ysh = oracle.expert_ffn(*ex[E], fmt, H, I, xq, xd)
    np.testing.assert_allclose(out1 - out0, ysh + res, rtol=1e-11, atol=1e-11 * np.abs(out1).max())


def test_null_expert_contributes_nothing():
    fmt, E, H, I, k, T = FMT_Q4K, 4, 256, 256, 2, 4
    ex = _experts(fmt, E, H, I, seed=13)
    wr = synth.router_weight(E, H, 13)
    x = synth.activations(T, H, 13)
    full, ids, gates, _ = oracle.layer_forward(fmt, H, I, E, k, 0, 0, ex, wr, None, x)
    dead = int(ids[0, 0])
    part_ex = list(ex)
    part_ex[dead] = None
    part, ids2, gates2, _ = oracle.layer_forward(fmt, H, I, E, k, 0, 0, part_ex, wr, None, x)
    np.testing.assert_array_equal(ids, ids2)
    xq, xd, _ = oracle.q8k_quantize(x)
    ydead = oracle.expert_ffn(*ex[dead], fmt, H, I, xq, xd)
    g = np.where(ids == dead, gates, 0.0).sum(axis=1)
    np.testing.assert_allclose(full - part, g[:, None] * ydead, rtol=1e-11, atol=1e-11 * np.abs(full).max())


def test_swiglu_on_constructed_weights():
    """Diagonal weights with w = 1/64 make G = U = x_q exactly (up to 1/64 * d_a),
    so h = silu(G) * U and the down projection returns h/64 to within q8_K rounding."""
    fmt, H, I, E, k = FMT_Q4K, 256, 256, 1, 1
    N = 256
    q = np.zeros((N, 1, 256), np.int64)
    q[np.arange(N), 0, np.arange(N)] = 1                  # identity pattern of codes
    sc = np.ones((N, 1, 8), np.int64)
    mn = np.zeros((N, 1, 8), np.int64)
    d = np.full((N, 1), 1.0 / 64, np.float16)             # exact in fp16
    dmin = np.zeros((N, 1), np.float16)
    eye = fieldpack.pack_fields(fmt, N, N, q, sc, mn, d, dmin)
    # up = 2 * identity/64: scale 2
    up = fieldpack.pack_fields(fmt, N, N, q, 2 * sc, mn, d, dmin)
    rng = np.random.default_rng(17)
    x = (rng.standard_normal((2, H)) * 100).astype(np.float32)
    wr = np.ones((1, H), np.float32)
    out, ids, gates, _ = oracle.layer_forward(fmt, H, I, E, k, 0, 0, [(eye, up, eye)], wr, None, x)
    assert (ids == 0).all() and (gates == 1.0).all()
    xq, xd, _ = oracle.q8k_quantize(x)
    a = xq.astype(np.float64) * xd.astype(np.float64)     # dequantized activation (one block)
    G = a / 64
    U = 2 * a / 64
    h = G / (1 + np.exp(-G)) * U
    dh = np.abs(h).max(axis=1, keepdims=True) / 127
    # down = identity/64 applied to q8_K(h): |y - h/64| <= (d_h/2)/64 (+ fp32 rounding of h)
    bound = (dh * 0.5 + 1e-6 * np.abs(h)) / 64 + 1e-12
    assert (np.abs(out - h / 64) <= bound).all()
    # the same bound rejects the other ways of gating: silu(U) * G, G * U, silu(G + U)
    for alt in [(U / (1 + np.exp(-U))) * G, G * U, (G + U) / (1 + np.exp(-(G + U)))]:
        assert not (np.abs(out - alt / 64) <= bound).all()
