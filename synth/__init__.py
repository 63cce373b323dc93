"""Seeded synthetic inputs for the block-quantized MoE layer.

This module is shared by the CUDA path's tests/bench and by the oracle's tests.
It holds no arithmetic of the method: it only draws random bytes and floats
and lays them out in the documented byte format (``synth.layout``).

Random weights
--------------
Every super-block (SB) of every weight matrix is keyed by
``(seed, layer, expert, matrix, row, sb)`` and draws its bytes from a
counter-based SplitMix64 stream (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014: state += 0x9E3779B97F4A7C15,
then the variant-13 finaliser).  Because the code and scale fields are plain
bit fields, uniformly random bytes give exactly the required distributions:
4-bit codes ~U{0..15}, 6-bit scales/mins ~U{0..63} (Q4_K-style), 2-bit codes
~U{0..3}, 4-bit scales/mins ~U{0..15} (Q2_K-style), 5-bit codes ~U{0..31}
(Q5_K-style), 3-bit codes ~U{0..7} and 6-bit scales ~U{-32..31} (Q3_K-style),
6-bit codes ~U{0..63} and int8 scales ~U{-128..127} (Q6_K-style), grid
indices ~U{0..255}, sign bits ~U{0,1} and 4-bit scales ~U{0..15} (IQ2-style
grid format).  Draws of one SB, in order: the code bytes (8 per draw,
little-endian), two draws of scale/min bytes (the first 4, 12 or 16 bytes
used), one for d, then (formats with a dmin) one for dmin.  The fp16 fields are drawn as d ~ U(1e-4, 1e-3)
and dmin ~ U(0, 5e-4): a 24-bit integer u gives f = u * 2^-24 in fp32
(exact), then ``lo + f * (hi - lo)`` with one fp32 multiply and one fp32
add, each rounded to nearest even, then fp32 -> fp16 round-to-nearest-even.
``synth/csrc/synth_gen.cu`` implements the same generator on the GPU
(weights of the large workloads, tens of GB, are made on the device); a test
checks the two byte-for-byte.

Random floats (activations, router weights, router bias) come from numpy's
``default_rng`` seeded with ``[seed, tag, layer, ...]`` on the host, and are
copied to the device.
"""
from __future__ import annotations

import numpy as np

from . import layout
from .layout import FMT_Q4K, FMT_Q2K, FMT_Q5K, FMT_Q3K, FMT_Q6K, FMT_IQ2G, sb_bytes, matrix_bytes

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15

# draws per super-block: codes, then scale/min bytes, then d, then dmin
_N_CODE_DRAWS = {f: layout.CODE_BYTES[f] // 8 for f in layout.FORMATS}   # 16, 8, 20, 12, 24, 8
_N_SM_DRAWS = 2
DRAWS_PER_SB = 32          # counter stride per super-block (at most 28 used)

# stream tags for the host float draws
TAG_X = 1
TAG_ROUTER = 2
TAG_BIAS = 3
TAG_RESIDUAL = 4


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= np.uint64(0xBF58476D1CE4E5B9)
    z ^= z >> np.uint64(27)
    z *= np.uint64(0x94D049BB133111EB)
    z ^= z >> np.uint64(31)
    return z


def _mix64_int(z: int) -> int:
    z &= MASK64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & MASK64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & MASK64
    z ^= z >> 31
    return z


def matrix_key(seed: int, layer: int, expert: int, mat: int) -> int:
    """64-bit stream key of one weight matrix (mat: 0 gate, 1 up, 2 down)."""
    k = _mix64_int(seed + GAMMA)
    k = _mix64_int(k ^ ((layer + 1) * GAMMA & MASK64))
    k = _mix64_int(k ^ ((expert * 4 + mat + 1) * GAMMA & MASK64))
    return k


def sb_draws(key: int, sb_index: np.ndarray, n_draws: int) -> np.ndarray:
    """uint64 draws [len(sb_index), n_draws] of the given super-blocks."""
    sb = sb_index.astype(np.uint64)
    i = np.arange(n_draws, dtype=np.uint64)
    ctr = sb[:, None] * np.uint64(DRAWS_PER_SB) + i[None, :] + np.uint64(1)
    state = np.uint64(key) + ctr * np.uint64(GAMMA)
    return _mix64(state)


# fp32 constants used by both generators (written as the fp32 literals 1e-4f,
# 9e-4f, 5e-4f in the CUDA generator)
D_LO, D_SPAN = 1e-4, 9e-4
DMIN_SPAN = 5e-4


def _d_bits(draw: np.ndarray) -> np.ndarray:
    u = (draw >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    v = np.float32(D_LO) + (u * np.float32(D_SPAN)).astype(np.float32)
    return v.astype(np.float32).astype(np.float16).view(np.uint16)


def _dmin_bits(draw: np.ndarray) -> np.ndarray:
    u = (draw >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    v = (u * np.float32(DMIN_SPAN)).astype(np.float32)
    return v.astype(np.float16).view(np.uint16)


def gen_sb_fields(fmt: int, key: int, sb_index: np.ndarray):
    """Raw per-super-block bytes (logical order) for the given SB indices.

    Returns (code_bytes [n, code bytes] uint8, sm_bytes [n, 4|12|16] uint8,
    d_bits [n] uint16, dmin_bits [n] uint16 or None for the formats without
    a dmin).
    """
    nc = _N_CODE_DRAWS[fmt]
    has_dmin = layout.HAS_DMIN[fmt]
    dr = sb_draws(key, sb_index, nc + _N_SM_DRAWS + (2 if has_dmin else 1))
    code_bytes = np.ascontiguousarray(dr[:, :nc].astype('<u8')).view(np.uint8).reshape(len(sb_index), nc * 8)
    sm_all = np.ascontiguousarray(dr[:, nc:nc + 2].astype('<u8')).view(np.uint8).reshape(len(sb_index), 16)
    sm_bytes = sm_all[:, :layout.SM_BYTES[fmt]].copy()
    d_bits = _d_bits(dr[:, nc + 2])
    dmin_bits = _dmin_bits(dr[:, nc + 3]) if has_dmin else None
    return code_bytes, sm_bytes, d_bits, dmin_bits


def gen_matrix(fmt: int, N: int, K: int, seed: int, layer: int, expert: int, mat: int) -> np.ndarray:
    """Bytes of one random [N, K] weight matrix in the documented layout."""
    layout.check_shape(N, K)
    nb = K // 256
    key = matrix_key(seed, layer, expert, mat)
    sb = np.arange(N * nb, dtype=np.int64)            # sb = row * nb + b
    code_bytes, sm_bytes, d_bits, dmin_bits = gen_sb_fields(fmt, key, sb)
    return layout.pack(fmt, N, K, code_bytes.reshape(N, nb, -1), sm_bytes.reshape(N, nb, -1),
                       d_bits.reshape(N, nb), None if dmin_bits is None else dmin_bits.reshape(N, nb))


def normal_f32(shape, std: float, seed: int, tag: int, *idx: int) -> np.ndarray:
    rng = np.random.default_rng([int(seed), int(tag), *[int(i) for i in idx]])
    return (rng.standard_normal(shape) * std).astype(np.float32)


def activations(T: int, H: int, seed: int, layer: int = 0, rep: int = 0) -> np.ndarray:
    """x ~ N(0, 1) fp32 [T, H]."""
    return normal_f32((T, H), 1.0, seed, TAG_X, layer, rep)


def router_weight(E: int, H: int, seed: int, layer: int = 0) -> np.ndarray:
    """W_r ~ N(0, std = 1/sqrt(H)) fp32 [E, H]."""
    return normal_f32((E, H), 1.0 / np.sqrt(H), seed, TAG_ROUTER, layer)


def router_bias(E: int, std: float, seed: int, layer: int = 0) -> np.ndarray:
    """Per-expert logit bias ~ N(0, std) fp32 [E] (skewed expert popularity)."""
    return normal_f32((E,), std, seed, TAG_BIAS, layer)


__all__ = [
    "layout", "FMT_Q4K", "FMT_Q2K", "FMT_Q5K", "FMT_Q3K", "FMT_Q6K", "FMT_IQ2G", "sb_bytes", "matrix_bytes", "matrix_key", "sb_draws",
    "gen_sb_fields", "gen_matrix", "activations", "router_weight", "router_bias", "normal_f32",
]
