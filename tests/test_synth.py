"""The seeded input generators (CPU): determinism, field ranges and
distributions, independence of streams."""
import numpy as np
import pytest

import oracle
import synth
from synth.layout import FMT_Q4K, FMT_Q2K, FORMATS
from tests import fieldpack


@pytest.mark.parametrize("fmt", FORMATS)
def test_matrix_generator_is_deterministic_and_keyed(fmt):
    a = synth.gen_matrix(fmt, 256, 512, 1, 0, 3, 0)
    b = synth.gen_matrix(fmt, 256, 512, 1, 0, 3, 0)
    c = synth.gen_matrix(fmt, 256, 512, 1, 0, 3, 1)
    d = synth.gen_matrix(fmt, 256, 512, 2, 0, 3, 0)
    assert a.size == synth.matrix_bytes(fmt, 256, 512)
    np.testing.assert_array_equal(a, b)
    assert (a != c).mean() > 0.9 and (a != d).mean() > 0.9


@pytest.mark.parametrize("fmt", FORMATS)
def test_generated_fields_follow_the_workload_distributions(fmt):
    """Codes, scales and mins uniform over their ranges (signed scales for the symmetric formats),
    d ~ U(1e-4, 1e-3), dmin ~ U(0, 5e-4) where the format has one."""
    N, K = 512, 1024
    w = synth.gen_matrix(fmt, N, K, 0, 0, 0, 0)
    qmax = fieldpack.QMAX[fmt]
    slo, shi = fieldpack.SCALE_RANGE[fmt]
    qs, scs, mns, ds, dms = [], [], [], [], []
    for n in range(0, N, 7):
        for b in range(K // 256):
            q, sc, mn, d, dmin = oracle.unpack_sb(w, fmt, N, K, n, b)
            qs.append(q); scs.append(sc); mns.append(mn); ds.append(d); dms.append(dmin)
    q = np.concatenate(qs); sc = np.concatenate(scs); mn = np.concatenate(mns)
    ds = np.array(ds); dms = np.array(dms)
    checks = [(q, 0, qmax), (sc, slo, shi)]
    if fmt == synth.FMT_IQ2G:
        # grid indices U{0..255}, scales 2t + 1 with t ~ U{0..15}, each sign a fair coin (bit 7: parity)
        gi = fieldpack._grid_index()
        grp = q.reshape(-1, 8)
        idx = np.array([gi[tuple(int(x) for x in np.abs(r))] for r in grp])
        checks = [(idx, 0, 255), ((sc - 1) // 2, 0, 15), ((grp[:, :7] < 0).astype(np.int64).reshape(-1), 0, 1)]
        assert ((grp < 0).sum(axis=1) % 2 == 0).all()
    elif fmt not in fieldpack.SYMMETRIC:
        checks.append((mn, 0, fieldpack.MIN_RANGE[fmt][1]))
    else:
        assert (mn == 0).all() and (dms == 0).all()
    for v, lo, top in checks:
        hist = np.bincount(v - lo, minlength=top - lo + 1)
        assert hist.size == top - lo + 1
        expect = v.size / (top - lo + 1)
        assert np.abs(hist - expect).max() < 6 * np.sqrt(expect) + 3
    assert ds.min() >= 1e-4 * 0.999 and ds.max() <= 1e-3 * 1.001
    assert abs(ds.mean() - 5.5e-4) < 3e-5
    if synth.layout.HAS_DMIN[fmt]:
        assert dms.min() >= 0 and dms.max() <= 5e-4 * 1.001
        assert abs(dms.mean() - 2.5e-4) < 2e-5


def test_float_streams():
    x = synth.activations(4, 512, 0)
    assert x.dtype == np.float32 and x.shape == (4, 512)
    np.testing.assert_array_equal(x, synth.activations(4, 512, 0))
    assert not np.array_equal(x, synth.activations(4, 512, 0, layer=1))
    wr = synth.router_weight(256, 2048, 1)
    assert abs(wr.std() * np.sqrt(2048) - 1) < 0.01
    b = synth.router_bias(192, 2.0, 3)
    assert abs(b.std() - 2) < 0.4
