"""Pins of the oracle to facts outside itself (CPU only).

Each test checks one oracle function against something the oracle does not
compute itself: hand-derived golden values (tests/golden), closed forms,
brute force on small inputs, library routines (sorting, dense matmul), or
invariants of the definition.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth
from synth.layout import FMT_Q4K, FMT_Q2K, FMT_Q5K, FMT_Q3K, FMT_Q6K, FMT_IQ2G, FORMATS
from tests import fieldpack

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _sparse(d, n=256, dtype=np.float32):
    v = np.zeros(n, dtype)
    for k, x in d.items():
        v[int(k)] = x
    return v


# ---------------------------------------------------------------- q8_K

@pytest.mark.parametrize("case", _load("q8k_blocks.json")["cases"], ids=lambda c: c["name"][:40])
def test_q8k_golden(case):
    x = _sparse(case["x"])
    q, d, bs = oracle.q8k_quantize(x[None, :])
    assert d[0, 0] == np.float32(case["d"])
    np.testing.assert_array_equal(q[0], _sparse(case["q"], dtype=np.int8))
    np.testing.assert_array_equal(bs[0], np.array(case["bsum16"], np.int16))


def test_q8k_roundtrip_bounds():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 1024)) * rng.uniform(1e-3, 1e3, (64, 1))).astype(np.float32)
    x[3, 256:512] = 0.0                                            # one all-zero block
    x[4, :256] = np.float32(1e-40) * rng.standard_normal(256)       # subnormal inputs
    q, d, bs = oracle.q8k_quantize(x)
    xb = x.reshape(64, 4, 256).astype(np.float64)
    qb = q.reshape(64, 4, 256).astype(np.float64)
    amax = np.abs(xb).max(axis=2)
    np.testing.assert_array_equal(d, (amax.astype(np.float32) / np.float32(127)))
    assert np.abs(q).max() <= 127
    # |x - d q| <= d/2 (plus a few fp32 ulps of x/d)
    err = np.abs(xb - d[..., None].astype(np.float64) * qb)
    bound = d[..., None].astype(np.float64) * (0.5 + 1e-5) + 1e-45
    assert (err <= bound).all()
    # the largest magnitude maps to +-127 (where d > 0)
    nz = d > 0
    imax = np.abs(xb).argmax(axis=2)
    qmax = np.take_along_axis(qb, imax[..., None], axis=2)[..., 0]
    assert (np.abs(qmax[nz]) == 127).all()
    assert (q.reshape(64, 4, 256)[3, 1] == 0).all() and d[3, 1] == 0
    # sign is preserved
    assert ((np.sign(qb) * np.sign(xb)) >= 0).all()
    # bsum16 = sums of 16 consecutive codes
    np.testing.assert_array_equal(bs, q.reshape(64, 64, 16).astype(np.int32).sum(axis=2))


# --------------------------------------------------------- format decode

@pytest.mark.parametrize("bits,value", [(0x3C00, 1.0), (0x3800, 0.5), (0xC000, -2.0), (0x0001, 2.0 ** -24),
                                        (0x03FF, 1023 * 2.0 ** -24), (0x0400, 2.0 ** -14),
                                        (0x7BFF, 65504.0), (0x1E1B, 1563 * 2.0 ** -18)])
def test_half_decode(bits, value):
    assert oracle.half_to_double(bits) == pytest.approx(value, rel=0, abs=1e-16)


@pytest.mark.parametrize("fmt", FORMATS)
def test_unpack_recovers_encoded_fields(fmt):
    rng = np.random.default_rng(11 + fmt)
    N, K = 256, 512
    q, sc, mn, d, dmin = fieldpack.random_fields(fmt, N, K, rng)
    w = fieldpack.pack_fields(fmt, N, K, q, sc, mn, d, dmin)
    assert w.size == synth.matrix_bytes(fmt, N, K)
    for n, b in [(0, 0), (1, 1), (31, 0), (32, 1), (77, 0), (255, 1)]:
        uq, usc, umn, ud, udmin = oracle.unpack_sb(w, fmt, N, K, n, b)
        np.testing.assert_array_equal(uq, q[n, b])
        np.testing.assert_array_equal(usc, sc[n, b])
        np.testing.assert_array_equal(umn, mn[n, b])
        assert ud == float(d[n, b]) and udmin == float(dmin[n, b])
    np.testing.assert_array_equal(oracle.dequant_matrix(w, fmt, N, K),
                                  fieldpack.dequant_fields(fmt, q, sc, mn, d, dmin))


@pytest.mark.parametrize("fmt", FORMATS)
def test_one_hot_activation_reads_one_weight(fmt):
    """x = c * e_i  ->  q8_K gives d = c/127, q_i = 127, so y[n] = fp32(c/127) * 127 * w[n, i]."""
    rng = np.random.default_rng(21 + fmt)
    N, K = 256, 768
    q, sc, mn, d, dmin = fieldpack.random_fields(fmt, N, K, rng)
    w = fieldpack.pack_fields(fmt, N, K, q, sc, mn, d, dmin)
    W = fieldpack.dequant_fields(fmt, q, sc, mn, d, dmin)
    for i, c in [(0, 3.0), (17, -1.5), (300, 0.75), (511, 2.0), (767, -5.0)]:
        x = np.zeros((1, K), np.float32)
        x[0, i] = c
        xq, xd, _ = oracle.q8k_quantize(x)
        y = oracle.qmatvec(w, fmt, N, K, xq, xd)[0]
        scale = float(np.float32(abs(c)) / np.float32(127)) * 127 * np.sign(c)
        np.testing.assert_allclose(y, scale * W[:, i], rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("fmt", FORMATS)
def test_integer_subblock_dot_equals_dense_dequantized_dot(fmt):
    """Brute force: sum_k w[n,k] * (d_a q_a[k]) in fp64 equals the sub-block integer form."""
    rng = np.random.default_rng(31 + fmt)
    N, K, T = 256, 1024, 3
    q, sc, mn, d, dmin = fieldpack.random_fields(fmt, N, K, rng)
    w = fieldpack.pack_fields(fmt, N, K, q, sc, mn, d, dmin)
    W = fieldpack.dequant_fields(fmt, q, sc, mn, d, dmin)
    x = rng.standard_normal((T, K)).astype(np.float32)
    xq, xd, _ = oracle.q8k_quantize(x)
    a = xq.astype(np.float64) * np.repeat(xd.astype(np.float64), 256, axis=1)
    y_dense = a @ W.T
    y = oracle.qmatvec(w, fmt, N, K, xq, xd)
    np.testing.assert_allclose(y, y_dense, rtol=1e-11, atol=1e-11 * np.abs(y_dense).max())
    # the integer sums themselves, against their definition on the fields
    isum, bsum = oracle.subblock_dots(w, fmt, N, K, xq)
    sl = synth.layout.SUB_LEN[fmt]
    ns = 256 // sl
    qa = xq.reshape(T, K // 256, ns, sl).astype(np.int64)
    np.testing.assert_array_equal(bsum, qa.sum(axis=3))
    qw = q.reshape(N, K // 256, ns, sl).astype(np.int64)
    np.testing.assert_array_equal(isum, np.einsum("nbjs,tbjs->tnbj", qw, qa))


@pytest.mark.parametrize("fmt", [f for f in FORMATS if f != FMT_IQ2G])   # its scales 2t + 1 are never 0
def test_zero_scale_and_min_give_zero(fmt):
    rng = np.random.default_rng(41)
    N, K = 256, 256
    q, sc, mn, d, dmin = fieldpack.random_fields(fmt, N, K, rng)
    sc[:] = 0
    mn[:] = 0
    w = fieldpack.pack_fields(fmt, N, K, q, sc, mn, d, dmin)
    x = rng.standard_normal((2, K)).astype(np.float32)
    xq, xd, _ = oracle.q8k_quantize(x)
    assert (oracle.qmatvec(w, fmt, N, K, xq, xd) == 0).all()


def test_extreme_codes_stay_exact():
    """Largest |isum|: q_w = 15, scale 63, q_a = +-127 everywhere; int64 sums are exact."""
    fmt, N, K = FMT_Q4K, 256, 256
    q = np.full((N, 1, 256), 15)
    sc = np.full((N, 1, 8), 63)
    mn = np.full((N, 1, 8), 63)
    d = np.full((N, 1), 1.0, np.float16)
    dmin = np.full((N, 1), 0.5, np.float16)
    w = fieldpack.pack_fields(fmt, N, K, q, sc, mn, d, dmin)
    x = np.full((1, K), -127.0, np.float32)      # d_a = 1, q_a = -127
    xq, xd, _ = oracle.q8k_quantize(x)
    y = oracle.qmatvec(w, fmt, N, K, xq, xd)
    # S = 8 * 63 * (32 * 15 * -127), M = 8 * 63 * (32 * -127)
    S = 8 * 63 * 32 * 15 * -127
    M = 8 * 63 * 32 * -127
    assert (y == 1.0 * (1.0 * S - 0.5 * M)).all()


@pytest.mark.parametrize("fmt", FORMATS)
def test_superblock_sums_from_fields(fmt):
    """S = sum_j sc_j isum_j and M = sum_j mn_j bsum_j, recomputed with numpy from the encoded fields;
    and y = sum_b d_a (d S - dmin M) reproduces qmatvec."""
    rng = np.random.default_rng(71 + fmt)
    N, K, T = 256, 512, 3
    q, sc, mn, d, dmin = fieldpack.random_fields(fmt, N, K, rng)
    w = fieldpack.pack_fields(fmt, N, K, q, sc, mn, d, dmin)
    x = rng.standard_normal((T, K)).astype(np.float32)
    xq, xd, _ = oracle.q8k_quantize(x)
    S, M = oracle.superblock_sums(w, fmt, N, K, xq)
    sl = synth.layout.SUB_LEN[fmt]
    ns = 256 // sl
    qa = xq.reshape(T, K // 256, ns, sl).astype(np.int64)
    qw = np.asarray(q, np.int64).reshape(N, K // 256, ns, sl)
    isum = np.einsum("nbjs,tbjs->tnbj", qw, qa)
    bsum = qa.sum(axis=3)
    # the min term: mn_j (scale dmin), or offset * scale_j (scale d) for the symmetric formats
    sym = fmt in fieldpack.SYMMETRIC
    m = fieldpack.OFFSET[fmt] * np.asarray(sc, np.int64) if sym else np.asarray(mn, np.int64)
    mscale = d if sym else dmin
    np.testing.assert_array_equal(S, np.einsum("nbj,tnbj->tnb", np.asarray(sc, np.int64), isum))
    np.testing.assert_array_equal(M, np.einsum("nbj,tbj->tnb", m, bsum))
    y = (xd.astype(np.float64)[:, None, :] * (d.astype(np.float64)[None] * S - mscale.astype(np.float64)[None] * M)).sum(axis=2)
    np.testing.assert_allclose(oracle.qmatvec(w, fmt, N, K, xq, xd), y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_superblock_sums_extreme_block():
    """q = 15, scale 63, min 63, activation codes all +127: S = 63 * 15 * 127 * 256 (above 2^24), M = 63 * 127 * 256."""
    fmt, N, K = FMT_Q4K, 256, 256
    w = fieldpack.pack_fields(fmt, N, K, np.full((N, 1, 256), 15), np.full((N, 1, 8), 63), np.full((N, 1, 8), 63),
                              np.full((N, 1), 1.0, np.float16), np.full((N, 1), 0.5, np.float16))
    S, M = oracle.superblock_sums(w, fmt, N, K, np.full((2, K), 127, np.int8))
    assert (S == 63 * 15 * 127 * 256).all() and S[0, 0, 0] > 2 ** 24
    assert (M == 63 * 127 * 256).all()


@pytest.mark.parametrize("fmt", FORMATS)
def test_absterms_from_fields_brute_force(fmt):
    """qmatvec_absterms = sum over super-blocks of |d_a| (|d| |S_b| + |dmin| |M_b|), with S_b and M_b
    recomputed here from the encoded fields by plain loops; and it bounds |qmatvec| (triangle inequality)."""
    rng = np.random.default_rng(51 + fmt)
    N, K, T = 256, 768, 2
    q, sc, mn, d, dmin = fieldpack.random_fields(fmt, N, K, rng)
    w = fieldpack.pack_fields(fmt, N, K, q, sc, mn, d, dmin)
    x = rng.standard_normal((T, K)).astype(np.float32)
    xq, xd, _ = oracle.q8k_quantize(x)
    a = oracle.qmatvec_absterms(w, fmt, N, K, xq, xd)
    sl = synth.layout.SUB_LEN[fmt]
    ns = 256 // sl
    sym = fmt in fieldpack.SYMMETRIC
    want = np.zeros((T, N))
    for t in range(T):
        for n in range(N):
            for b in range(K // 256):
                qa = xq[t, 256 * b:256 * b + 256].astype(np.int64).reshape(ns, sl)
                qw = np.asarray(q[n, b], np.int64).reshape(ns, sl)
                scb = np.asarray(sc[n, b], np.int64)
                S = int((scb * (qw * qa).sum(axis=1)).sum())
                m = fieldpack.OFFSET[fmt] * scb if sym else np.asarray(mn[n, b], np.int64)
                M = int((m * qa.sum(axis=1)).sum())
                mscale = float(d[n, b]) if sym else float(dmin[n, b])
                want[t, n] += abs(float(xd[t, b])) * (abs(float(d[n, b])) * abs(S) + abs(mscale) * abs(M))
    np.testing.assert_allclose(a, want, rtol=1e-13)
    y = oracle.qmatvec(w, fmt, N, K, xq, xd)
    assert (np.abs(y) <= a * (1 + 1e-12)).all()
    assert (a > np.abs(y)).any()                          # random signs do cancel somewhere


def test_absterms_equal_output_when_nothing_cancels():
    """dmin = 0 and non-negative activations: every term is >= 0, so the magnitude sum is the output."""
    fmt = FMT_Q4K
    rng = np.random.default_rng(61)
    N, K = 256, 512
    q, sc, mn, d, dmin = fieldpack.random_fields(fmt, N, K, rng)
    dmin[:] = 0
    w = fieldpack.pack_fields(fmt, N, K, q, sc, mn, d, dmin)
    x = np.abs(rng.standard_normal((3, K))).astype(np.float32)
    xq, xd, _ = oracle.q8k_quantize(x)
    np.testing.assert_array_equal(oracle.qmatvec_absterms(w, fmt, N, K, xq, xd), oracle.qmatvec(w, fmt, N, K, xq, xd))


@pytest.mark.parametrize("fmt", [FMT_Q5K, FMT_Q3K, FMT_Q6K])
def test_extreme_fields_closed_form(fmt):
    """Every code at its largest value, the scale at its extreme, activation codes all -127 (d_a = 1):
    y = -127 * 256 * d * scale * (qmax - o) + 127 * 256 * dmin * min, computed here from the definition."""
    N, K = 256, 256
    qmax = fieldpack.QMAX[fmt]
    scale = fieldpack.SCALE_RANGE[fmt][0] if fmt in fieldpack.SYMMETRIC else fieldpack.SCALE_RANGE[fmt][1]
    mn = fieldpack.MIN_RANGE[fmt][1]
    ns = synth.layout.N_SUB[fmt]
    w = fieldpack.pack_fields(fmt, N, K, np.full((N, 1, 256), qmax), np.full((N, 1, ns), scale),
                              np.full((N, 1, ns), mn), np.full((N, 1), 0.5, np.float16), np.full((N, 1), 0.25, np.float16))
    x = np.full((1, K), -127.0, np.float32)
    xq, xd, _ = oracle.q8k_quantize(x)
    off = fieldpack.OFFSET.get(fmt, 0)
    dmin = 0.25 if fmt not in fieldpack.SYMMETRIC else 0.0
    want = -127 * 256 * 0.5 * scale * (qmax - off) + 127 * 256 * dmin * mn
    assert (oracle.qmatvec(w, fmt, N, K, xq, xd) == want).all()
    q, sc, m, dd, dm = oracle.unpack_sb(w, fmt, N, K, 5, 0)
    assert (q == qmax).all() and (sc == scale).all() and dd == 0.5


# ------------------------------------------------------- IQ2-style grid format

def test_iq2g_grid_class_sizes_closed_form():
    """A vector of {1, 3, 5}^8 with a threes and b fives has sum of squares 8 + 8a + 24b, and there are
    C(8, a) C(8 - a, b) of them.  The grid takes every vector with a sum below 48 (1 + 8 + 28 + 64 + 126 =
    227 of them) and the first 29 of sum 48."""
    from math import comb
    g = oracle.iq2g_grid()
    assert g.shape == (256, 8) and set(np.unique(g)) <= {1, 3, 5}
    ss = (g.astype(np.int64) ** 2).sum(axis=1)
    want = {}
    for a in range(9):
        for b in range(9 - a):
            n = 8 + 8 * a + 24 * b
            want[n] = want.get(n, 0) + comb(8, a) * comb(8 - a, b)
    got = {int(k): int(v) for k, v in zip(*np.unique(ss, return_counts=True))}
    assert got == {8: want[8], 16: want[16], 24: want[24], 32: want[32], 40: want[40], 48: 29}
    assert (want[8], want[16], want[24], want[32], want[40]) == (1, 8, 28, 64, 126)
    assert (np.diff(ss) >= 0).all()                               # ordered by the sum of squares
    assert len({tuple(r) for r in g.tolist()}) == 256              # distinct


def test_iq2g_grid_entries_by_hand():
    """Entries worked out from the rule: 0 is all ones; 1..8 put one 3 at element 7, 6, .., 0 (smallest
    base-3 number first, element 0 most significant); 9 is the first sum-24 vector, threes at 6 and 7; 37 is
    the first sum-32 vector: one 5 at element 7 (digit 2 = base-3 number 2, below three 3s = 13)."""
    g = oracle.iq2g_grid()
    assert (g[0] == 1).all()
    for u in range(1, 9):
        want = np.ones(8, np.int32)
        want[8 - u] = 3
        np.testing.assert_array_equal(g[u], want)
    np.testing.assert_array_equal(g[9], [1, 1, 1, 1, 1, 1, 3, 3])
    np.testing.assert_array_equal(g[37], [1, 1, 1, 1, 1, 1, 1, 5])


def test_iq2g_grid_brute_force():
    """The rule by brute force over all 3^8 vectors (itertools order is increasing base-3 order)."""
    import itertools
    allv = [(sum(v * v for v in vec), n, vec) for n, vec in enumerate(itertools.product((1, 3, 5), repeat=8))]
    allv.sort()
    np.testing.assert_array_equal(oracle.iq2g_grid(), np.array([vec for _, _, vec in allv[:256]]))


def test_iq2g_closed_form_groups():
    """Hand-derived outputs (activation codes all -127, d_a = 1, d = 0.5):
    grid entry 0, no signs, t = 15 (scale 31): y = -127 * 256 * 0.5 * 31;
    grid entry 1 (element 7 = 3) with sign bit 0 set: the 8th sign is then minus too, so each group sums
    -1 + 6 * 1 - 3 = 2 and y = -127 * 32 * 2 * 0.5 * scale, with scales 1, 3, .., 15 over the sub-blocks."""
    fmt, N, K = FMT_IQ2G, 256, 256
    ones = np.ones(256, np.int64)
    w = fieldpack.pack_fields(fmt, N, K, np.tile(ones, (N, 1, 1)), np.full((N, 1, 8), 31), np.zeros((N, 1, 8)),
                              np.full((N, 1), 0.5, np.float16), np.zeros((N, 1), np.float16))
    xq, xd, _ = oracle.q8k_quantize(np.full((1, K), -127.0, np.float32))
    assert (oracle.qmatvec(w, fmt, N, K, xq, xd) == -127 * 256 * 0.5 * 31).all()
    grp = np.array([-1, 1, 1, 1, 1, 1, 1, -3])
    scales = np.arange(1, 17, 2)
    w = fieldpack.pack_fields(fmt, N, K, np.tile(np.tile(grp, 32), (N, 1, 1)), np.tile(scales, (N, 1, 1)),
                              np.zeros((N, 1, 8)), np.full((N, 1), 0.5, np.float16), np.zeros((N, 1), np.float16))
    y = oracle.qmatvec(w, fmt, N, K, xq, xd)
    assert (y == sum(-127 * 4 * 2 * 0.5 * s for s in scales)).all()
    # the stored bytes of one row: index byte 1 per group, sign byte 0b0000001 per group, scale nibbles t = 0..7
    slab = w[:synth.layout.SLAB_BYTES[fmt]]
    codes = slab[synth.layout.CODE_OFFSET[fmt]:].reshape(4, 32, 16)
    assert (codes[0:2, 3] == 1).all() and (codes[2:4, 3] == 1).all()
    sm = slab[synth.layout.SM_OFFSET[fmt]:synth.layout.CODE_OFFSET[fmt]].reshape(32, 4)
    np.testing.assert_array_equal(sm[3], [0x10, 0x32, 0x54, 0x76])


# ---------------------------------------------------------------- routing

@pytest.mark.parametrize("case", _load("route_cases.json")["cases"], ids=lambda c: c["name"][:40])
def test_route_golden(case):
    x = np.array([case["x"]], np.float32)
    wr = np.array(case["w_r"], np.float32)[:, None]
    _, ids, gates, gap = oracle.route(x, wr, None, case["k"], case["route"])
    np.testing.assert_array_equal(ids[0], case["ids"])
    np.testing.assert_allclose(gates[0], case["gates"], rtol=1e-15, atol=1e-16)
    want_gap = math.inf if case["gap"] == "inf" else case["gap"]
    assert gap[0] == want_gap


@pytest.mark.parametrize("route_kind", [0, 1])
@pytest.mark.parametrize("E,k", [(16, 2), (64, 8), (512, 10)])
def test_route_matches_full_sort(route_kind, E, k):
    rng = np.random.default_rng(E + k + route_kind)
    T, H = 5, 256
    x = rng.standard_normal((T, H)).astype(np.float32)
    wr = (rng.standard_normal((E, H)) / np.sqrt(H)).astype(np.float32)
    bias = rng.normal(0, 2, E).astype(np.float32)
    logits, ids, gates, gap = oracle.route(x, wr, bias, k, route_kind)
    ref = x.astype(np.float64) @ wr.astype(np.float64).T + bias.astype(np.float64)
    np.testing.assert_allclose(logits, ref, rtol=1e-12, atol=1e-12)
    order = np.argsort(-logits, axis=1, kind="stable")
    np.testing.assert_array_equal(ids, order[:, :k])
    srt = np.take_along_axis(logits, order, axis=1)
    np.testing.assert_array_equal(gap, srt[:, k - 1] - srt[:, k])
    np.testing.assert_allclose(gates.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    sel = np.take_along_axis(logits, ids, axis=1)
    if route_kind == 0:
        full = np.exp(logits - logits.max(axis=1, keepdims=True))
        full /= full.sum(axis=1, keepdims=True)            # full softmax, then renormalise over k
        want = np.take_along_axis(full, ids, axis=1)
        want /= want.sum(axis=1, keepdims=True)
    else:
        s = 1.0 / (1.0 + np.exp(-sel))
        want = s / s.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(gates, want, rtol=1e-12)
    assert (np.diff(gates, axis=1) <= 1e-15).all()          # gates follow the logit order


def test_route_forced_ids():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 256)).astype(np.float32)
    wr = rng.standard_normal((8, 256)).astype(np.float32)
    forced = np.array([[5, 1], [0, 7]], np.int32)
    logits, ids, gates, _ = oracle.route(x, wr, None, 2, 0, forced_ids=forced)
    np.testing.assert_array_equal(ids, forced)
    sel = np.take_along_axis(logits, forced, axis=1)
    e = np.exp(sel - sel.max(axis=1, keepdims=True))
    np.testing.assert_allclose(gates, e / e.sum(axis=1, keepdims=True), rtol=1e-13)


# ---------------------------------------------------------------- bucketing

def test_bucket_golden():
    c = _load("bucket_case.json")
    counts, offsets, perm = oracle.bucket(np.array(c["ids"]), c["E"], c["S"])
    np.testing.assert_array_equal(counts, c["counts"])
    np.testing.assert_array_equal(offsets, c["offsets"])
    np.testing.assert_array_equal(perm, c["perm"])


@pytest.mark.parametrize("T,k,E,S", [(1, 8, 256, 1), (16, 8, 192, 0), (64, 10, 512, 1), (7, 1, 4, 0)])
def test_bucket_invariants(T, k, E, S):
    rng = np.random.default_rng(T * 1000 + E)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm = oracle.bucket(ids, E, S)
    assert counts.sum() == T * k + S * T
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    np.testing.assert_array_equal(np.sort(perm), np.arange(T * k + S * T))   # a permutation
    flat = ids.reshape(-1)
    for e in range(E):
        p = perm[offsets[e]:offsets[e + 1]]
        assert (flat[p] == e).all()
        assert (np.diff(p // k) > 0).all()                 # stable by token, one slot per token
    for sh in range(S):
        p = perm[offsets[E + sh]:offsets[E + sh + 1]]
        np.testing.assert_array_equal(p, T * k + sh * T + np.arange(T))
