"""Test-side encoder: super-block FIELDS -> bytes in the documented layout.

Independent of the oracle's decoder (oracle/moe_oracle.cpp) and of the CUDA
kernels: it encodes chosen codes/scales/mins/d/dmin by the layout rules
(synth/layout.py docstring) so that a decoder can be checked against known
fields.  The slab placement reuses synth.layout.pack (which only moves bytes).
Scales are passed signed where the format's scale is signed (Q3_K-style:
-32..31, Q6_K-style: -128..127); the symmetric formats have no min and no
dmin (zeros are passed and ignored).  For the IQ2-style grid format the
"codes" are the signed weight values s * C[u][i] and the scale is 2t + 1;
encoding finds each group's grid index in the grid the oracle exports (the
grid itself is pinned by its own tests) and checks the sign parity rule.
"""
from __future__ import annotations

import numpy as np

from synth import layout
from synth.layout import FMT_Q4K, FMT_Q2K, FMT_Q5K, FMT_Q3K, FMT_Q6K, FMT_IQ2G

QMAX = {FMT_Q4K: 15, FMT_Q2K: 3, FMT_Q5K: 31, FMT_Q3K: 7, FMT_Q6K: 63, FMT_IQ2G: 5}
SCALE_RANGE = {FMT_Q4K: (0, 63), FMT_Q2K: (0, 15), FMT_Q5K: (0, 63), FMT_Q3K: (-32, 31), FMT_Q6K: (-128, 127),
               FMT_IQ2G: (1, 31)}
MIN_RANGE = {FMT_Q4K: (0, 63), FMT_Q2K: (0, 15), FMT_Q5K: (0, 63), FMT_Q3K: (0, 0), FMT_Q6K: (0, 0),
             FMT_IQ2G: (0, 0)}
OFFSET = {FMT_Q3K: 4, FMT_Q6K: 32}          # symmetric formats: weight = d * scale * (q - offset)
SYMMETRIC = (FMT_Q3K, FMT_Q6K)


def _q4k_lines(q):
    """codes [..., 256] (< 16) -> 128 bytes: line j, byte i = code i | code i+16 << 4 of sub-block j."""
    lead = q.shape[:-1]
    sub = q.reshape(*lead, 8, 32)
    return (sub[..., :16] | (sub[..., 16:] << 4)).reshape(*lead, 128).astype(np.uint8)


def _q2k_lines(q):
    """codes [..., 256] (< 4) -> 64 bytes: sub-block j, bits 2p..2p+1 of byte m = code 4p + m."""
    lead = q.shape[:-1]
    sub = q.reshape(*lead, 16, 4, 4)                  # sub-block j, p, m  (code 4p + m)
    byte = np.zeros((*lead, 16, 4), np.uint8)
    for p in range(4):
        byte |= (sub[..., p, :] << (2 * p)).astype(np.uint8)
    return byte.reshape(*lead, 64)


_GRID_INDEX = None


def _grid_index():
    """{tuple of 8 magnitudes: grid index} of the oracle's IQ2-style grid."""
    global _GRID_INDEX
    if _GRID_INDEX is None:
        import oracle
        _GRID_INDEX = {tuple(int(v) for v in row): u for u, row in enumerate(oracle.iq2g_grid())}
    return _GRID_INDEX


def _iq2g_planes(q):
    """signed values [..., 256] -> 64 bytes: 32 grid indices, then 32 sign bytes (bits 0-6)."""
    lead = q.shape[:-1]
    grp = q.reshape(-1, 32, 8)
    idx = np.zeros((grp.shape[0], 32), np.uint8)
    sgn = np.zeros((grp.shape[0], 32), np.uint8)
    gi = _grid_index()
    for r in range(grp.shape[0]):
        for g in range(32):
            v = grp[r, g]
            neg = (v < 0).astype(np.int64)
            assert neg.sum() % 2 == 0, "an IQ2-style group has an even number of negative weights"
            idx[r, g] = gi[tuple(int(x) for x in np.abs(v))]
            sgn[r, g] = int((neg[:7] << np.arange(7)).sum())
    return np.concatenate([idx, sgn], axis=1).reshape(*lead, 64)


def encode_codes(fmt: int, q: np.ndarray) -> np.ndarray:
    """codes [..., 256] -> logical code bytes [..., CODE_BYTES] (the planes in order)."""
    q = np.asarray(q).astype(np.int64)
    if fmt == FMT_IQ2G:
        return _iq2g_planes(q)
    assert q.min() >= 0 and q.max() <= QMAX[fmt]
    lead = q.shape[:-1]
    if fmt == FMT_Q4K:
        return _q4k_lines(q)
    if fmt == FMT_Q2K:
        return _q2k_lines(q)
    if fmt == FMT_Q5K:
        hi = np.zeros((*lead, 32), np.uint8)          # line m, byte i -> index 16 m + i
        for m in range(2):
            for i in range(16):
                v = np.zeros(lead, np.int64)
                for jj in range(4):
                    for h in range(2):
                        v |= ((q[..., 32 * (4 * m + jj) + i + 16 * h] >> 4) & 1) << (2 * jj + h)
                hi[..., 16 * m + i] = v
        return np.concatenate([_q4k_lines(q & 15), hi], axis=-1)
    if fmt == FMT_Q3K:
        hi = np.zeros((*lead, 32), np.uint8)
        for j in range(16):
            for p in range(4):
                for m in range(4):
                    idx = 16 * (j // 8) + 4 * ((j // 2) % 4) + m
                    hi[..., idx] |= (((q[..., 16 * j + 4 * p + m] >> 2) & 1) << (p + 4 * (j % 2))).astype(np.uint8)
        return np.concatenate([_q2k_lines(q & 3), hi], axis=-1)
    # Q6_K
    lo = np.zeros((*lead, 128), np.uint8)
    for l_ in range(8):
        for i in range(16):
            lo[..., 16 * l_ + i] = ((q[..., 16 * (2 * l_) + i] & 15) | ((q[..., 16 * (2 * l_ + 1) + i] & 15) << 4))
    hi = np.zeros((*lead, 64), np.uint8)
    for m in range(4):
        for i in range(16):
            v = np.zeros(lead, np.int64)
            for jj in range(4):
                v |= ((q[..., 16 * (4 * m + jj) + i] >> 4) & 3) << (2 * jj)
            hi[..., 16 * m + i] = v
    return np.concatenate([lo, hi], axis=-1)


def _bits96(fields, width=6):
    """[..., nf] small ints -> [..., 12] bytes of a little-endian bit string (field f at bits width*f)."""
    lead = fields.shape[:-1]
    flat = fields.reshape(-1, fields.shape[-1])
    out = np.zeros((flat.shape[0], 12), np.uint8)
    for row in range(flat.shape[0]):
        bits = 0
        for f, v in enumerate(flat[row]):
            bits |= int(v) << (width * f)
        out[row] = np.frombuffer(bits.to_bytes(12, "little"), np.uint8)
    return out.reshape(*lead, 12)


def encode_scales(fmt: int, sc: np.ndarray, mn: np.ndarray) -> np.ndarray:
    """per-sub-block scale/min [..., ns] -> logical scale/min bytes [..., SM_BYTES]."""
    sc = np.asarray(sc).astype(np.int64)
    mn = np.asarray(mn).astype(np.int64)
    lo, hi = SCALE_RANGE[fmt]
    assert sc.min() >= lo and sc.max() <= hi
    if fmt == FMT_Q2K:
        assert mn.max() <= 15
        return (sc.astype(np.uint8) | (mn.astype(np.uint8) << 4)).astype(np.uint8)
    if fmt in (FMT_Q4K, FMT_Q5K):
        assert mn.max() <= 63
        return _bits96(np.concatenate([sc, mn], axis=-1))
    if fmt == FMT_Q3K:
        return _bits96(sc + 32)
    if fmt == FMT_IQ2G:
        assert (sc % 2 == 1).all()
        t = ((sc - 1) // 2).astype(np.uint8)
        return (t[..., 0::2] | (t[..., 1::2] << 4)).astype(np.uint8)
    return sc.astype(np.int8).view(np.uint8)


def pack_fields(fmt: int, N: int, K: int, q, sc, mn, d, dmin) -> np.ndarray:
    """Fields of every SB of an [N, K] matrix -> matrix bytes.

    q [N, nb, 256] ints; sc, mn [N, nb, ns] ints; d, dmin [N, nb] floats
    (rounded to fp16; dmin ignored by the symmetric formats)."""
    cb = encode_codes(fmt, np.asarray(q))
    smb = encode_scales(fmt, np.asarray(sc), np.asarray(mn))
    db = np.asarray(d, np.float16).view(np.uint16)
    dmb = np.asarray(dmin, np.float16).view(np.uint16) if layout.HAS_DMIN[fmt] else None
    return layout.pack(fmt, N, K, cb, smb, db, dmb)


def random_fields(fmt: int, N: int, K: int, rng: np.random.Generator):
    nb = K // 256
    ns = layout.N_SUB[fmt]
    if fmt == FMT_IQ2G:
        import oracle
        grid = oracle.iq2g_grid().astype(np.int64)
        u = rng.integers(0, 256, (N, nb, 32))
        neg = rng.integers(0, 2, (N, nb, 32, 8))
        neg[..., 7] = neg[..., :7].sum(axis=-1) % 2      # an even number of minus signs
        q = (grid[u] * (1 - 2 * neg)).reshape(N, nb, 256)
        sc = 2 * rng.integers(0, 16, (N, nb, ns)) + 1
    else:
        q = rng.integers(0, QMAX[fmt] + 1, (N, nb, 256))
        sc = rng.integers(SCALE_RANGE[fmt][0], SCALE_RANGE[fmt][1] + 1, (N, nb, ns))
    mn = rng.integers(MIN_RANGE[fmt][0], MIN_RANGE[fmt][1] + 1, (N, nb, ns))
    d = rng.uniform(1e-4, 1e-3, (N, nb)).astype(np.float16)
    dmin = rng.uniform(0, 5e-4, (N, nb)).astype(np.float16) if layout.HAS_DMIN[fmt] else np.zeros((N, nb), np.float16)
    return q, sc, mn, d, dmin


def dequant_fields(fmt: int, q, sc, mn, d, dmin) -> np.ndarray:
    """W [N, K] in fp64 from fields: d * sc_j * q - dmin * mn_j, or d * sc_j * (q - offset)."""
    N, nb, _ = q.shape
    sl = layout.SUB_LEN[fmt]
    scx = np.repeat(np.asarray(sc, np.float64), sl, axis=2)
    mnx = np.repeat(np.asarray(mn, np.float64), sl, axis=2)
    dd = np.asarray(d, np.float64)[..., None]
    if fmt in SYMMETRIC:
        w = dd * scx * (np.asarray(q, np.float64) - OFFSET[fmt])
    else:
        w = dd * scx * q - np.asarray(dmin, np.float64)[..., None] * mnx
    return w.reshape(N, nb * 256)
