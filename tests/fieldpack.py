"""Test-side encoder: super-block FIELDS -> bytes in the documented layout.

Independent of the oracle's decoder (oracle/moe_oracle.cpp) and of the CUDA
kernels: it encodes chosen codes/scales/mins/d/dmin by the layout rules
(synth/layout.py docstring) so that a decoder can be checked against known
fields.  The slab placement reuses synth.layout.pack (which only moves bytes).
"""
from __future__ import annotations

import numpy as np

from synth import layout
from synth.layout import FMT_Q4K, FMT_Q2K


def encode_codes(fmt: int, q: np.ndarray) -> np.ndarray:
    """codes [..., 256] -> logical code bytes [..., 128 | 64]."""
    q = q.astype(np.uint8)
    lead = q.shape[:-1]
    if fmt == FMT_Q4K:
        assert q.max() <= 15
        sub = q.reshape(*lead, 8, 32)                 # sub-block j, code i
        lo, hi = sub[..., :16], sub[..., 16:]         # byte i = code i | code i+16 << 4
        return (lo | (hi << 4)).reshape(*lead, 128)
    assert q.max() <= 3
    sub = q.reshape(*lead, 16, 4, 4)                  # sub-block j, p, m  (code 4p + m)
    byte = np.zeros((*lead, 16, 4), np.uint8)
    for p in range(4):
        byte |= sub[..., p, :] << (2 * p)             # bits 2p..2p+1 of byte m
    return byte.reshape(*lead, 64)


def encode_scales(fmt: int, sc: np.ndarray, mn: np.ndarray) -> np.ndarray:
    """per-sub-block scale/min [..., ns] -> logical scale/min bytes [..., 12 | 16]."""
    lead = sc.shape[:-1]
    if fmt == FMT_Q2K:
        assert sc.max() <= 15 and mn.max() <= 15
        return (sc.astype(np.uint8) | (mn.astype(np.uint8) << 4)).reshape(*lead, 16)
    assert sc.max() <= 63 and mn.max() <= 63
    out = np.zeros((*lead, 12), np.uint8)
    flat_sc = sc.reshape(-1, 8)
    flat_mn = mn.reshape(-1, 8)
    flat = out.reshape(-1, 12)
    for row in range(flat.shape[0]):
        bits = 0
        for j in range(8):
            bits |= int(flat_sc[row, j]) << (6 * j)
            bits |= int(flat_mn[row, j]) << (48 + 6 * j)
        flat[row] = np.frombuffer(bits.to_bytes(12, "little"), np.uint8)
    return out


def pack_fields(fmt: int, N: int, K: int, q, sc, mn, d, dmin) -> np.ndarray:
    """Fields of every SB of an [N, K] matrix -> matrix bytes.

    q [N, nb, 256] ints; sc, mn [N, nb, ns] ints; d, dmin [N, nb] floats
    (rounded to fp16)."""
    cb = encode_codes(fmt, np.asarray(q))
    smb = encode_scales(fmt, np.asarray(sc), np.asarray(mn))
    db = np.asarray(d, np.float16).view(np.uint16)
    dmb = np.asarray(dmin, np.float16).view(np.uint16)
    return layout.pack(fmt, N, K, cb, smb, db, dmb)


def random_fields(fmt: int, N: int, K: int, rng: np.random.Generator):
    nb = K // 256
    ns = 8 if fmt == FMT_Q4K else 16
    qmax = 15 if fmt == FMT_Q4K else 3
    smax = 63 if fmt == FMT_Q4K else 15
    q = rng.integers(0, qmax + 1, (N, nb, 256))
    sc = rng.integers(0, smax + 1, (N, nb, ns))
    mn = rng.integers(0, smax + 1, (N, nb, ns))
    d = rng.uniform(1e-4, 1e-3, (N, nb)).astype(np.float16)
    dmin = rng.uniform(0, 5e-4, (N, nb)).astype(np.float16)
    return q, sc, mn, d, dmin


def dequant_fields(fmt: int, q, sc, mn, d, dmin) -> np.ndarray:
    """W [N, K] in fp64 from fields: w = d * sc_j * q - dmin * mn_j."""
    N, nb, _ = q.shape
    sl = 32 if fmt == FMT_Q4K else 16
    scx = np.repeat(sc, sl, axis=2)
    mnx = np.repeat(mn, sl, axis=2)
    w = (d.astype(np.float64)[..., None] * scx * q - dmin.astype(np.float64)[..., None] * mnx)
    return w.reshape(N, nb * 256)
