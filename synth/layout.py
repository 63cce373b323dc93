"""Byte layout of the block-quantized weight matrices ("row-group slabs").

A weight matrix W[N, K] (N rows, K columns, both multiples of 256; N also a
multiple of 32) is cut into 256-wide super-blocks (SB): row n, SB b covers
columns 256*b .. 256*b+255.  Each SB carries the fields of its format:

  Q4_K-style (144 B per SB): fp16 d, fp16 dmin, eight 32-weight sub-blocks
    with a 6-bit scale and a 6-bit min each (12 B), 256 4-bit codes (128 B);
    weight = d * scale_j * q - dmin * min_j.
  Q2_K-style (84 B per SB): fp16 d, fp16 dmin, sixteen 16-weight sub-blocks
    with a 4-bit scale and a 4-bit min each (16 B), 256 2-bit codes (64 B);
    weight = d * scale_j * q - dmin * min_j.

Placement.  Rows are grouped 32 at a time (row group rg = n // 32, lane
r = n % 32).  The matrix is the sequence of slabs (rg, b) in order
rg-major, b-minor; one slab holds SB b of the 32 rows of its group:

  Q4_K slab, 4608 B:
    [   0,  128)  dm:    row r at 4*r, uint32 = d_bits | dmin_bits << 16
    [ 128,  512)  sm:    row r at 128 + 12*r, 12 bytes
    [ 512, 4608)  codes: sub-block j (0..7) of row r at 512 + 512*j + 16*r,
                         16 bytes; byte i holds code i (low nibble) and
                         code i+16 (high nibble) of the sub-block
  Q2_K slab, 2688 B:
    [   0,  128)  dm:    as above
    [ 128,  640)  sm:    row r at 128 + 16*r, 16 bytes; byte j = scale_j | min_j << 4
    [ 640, 2688)  codes: sub-block j (0..15) of row r at
                         640 + 512*(j // 4) + 16*r + 4*(j % 4), 4 bytes; bits
                         2p..2p+1 of byte m hold code 4*p + m of the sub-block

Q4_K scale/min bytes: a 96-bit little-endian bit string; scale j is bits
6j..6j+5 and min j is bits 48+6j..48+6j+5 (bit i of the string is bit i%8 of
byte i//8).

Logical SB bytes (what the generator draws): 128 (Q4_K) / 64 (Q2_K) code
bytes, where code byte i goes to code line i // 16 (Q4_K: sub-block i // 16;
Q2_K: sub-blocks 4*(i//16) .. 4*(i//16)+3), byte i % 16 of that line; the
12 / 16 scale-min bytes in order; d and dmin.

Why this placement: in the decode kernels one lane owns one row, so every
16-byte load of a warp reads 512 contiguous bytes, and a whole row group is
one contiguous run of bytes (nb slabs) for bulk copies.
"""
from __future__ import annotations

import numpy as np

FMT_Q4K = 0
FMT_Q2K = 1

SB_BYTES = {FMT_Q4K: 144, FMT_Q2K: 84}
SM_BYTES = {FMT_Q4K: 12, FMT_Q2K: 16}
CODE_BYTES = {FMT_Q4K: 128, FMT_Q2K: 64}
N_SUB = {FMT_Q4K: 8, FMT_Q2K: 16}
SUB_LEN = {FMT_Q4K: 32, FMT_Q2K: 16}
SLAB_BYTES = {FMT_Q4K: 32 * 144, FMT_Q2K: 32 * 84}
SM_OFFSET = 128
CODE_OFFSET = {FMT_Q4K: 512, FMT_Q2K: 640}
ROWS_PER_GROUP = 32


def sb_bytes(fmt: int) -> int:
    return SB_BYTES[fmt]


def check_shape(N: int, K: int) -> None:
    if N <= 0 or K <= 0 or N % 256 or K % 256:
        raise ValueError(f"matrix [{N}, {K}]: both dimensions must be positive multiples of 256")


def matrix_bytes(fmt: int, N: int, K: int) -> int:
    check_shape(N, K)
    return N * (K // 256) * SB_BYTES[fmt]


def pack(fmt: int, N: int, K: int, code_bytes: np.ndarray, sm_bytes: np.ndarray,
         d_bits: np.ndarray, dmin_bits: np.ndarray) -> np.ndarray:
    """Place logical SB bytes [N, nb, ...] into the slab layout; returns uint8 [bytes]."""
    check_shape(N, K)
    nb = K // 256
    RG = N // 32
    cb = CODE_BYTES[fmt]
    smb = SM_BYTES[fmt]
    assert code_bytes.shape == (N, nb, cb) and sm_bytes.shape == (N, nb, smb)
    dm = (d_bits.astype(np.uint32) | (dmin_bits.astype(np.uint32) << np.uint32(16)))
    # [RG, 32, nb, ...] -> [RG, nb, 32, ...]
    dm = dm.reshape(RG, 32, nb).transpose(0, 2, 1).astype('<u4')
    dm_b = np.ascontiguousarray(dm).view(np.uint8).reshape(RG, nb, 128)
    sm = sm_bytes.reshape(RG, 32, nb, smb).transpose(0, 2, 1, 3).reshape(RG, nb, 32 * smb)
    # code byte i -> line i // 16, byte i % 16; lines are [32 rows][16 B]
    nl = cb // 16
    codes = code_bytes.reshape(RG, 32, nb, nl, 16).transpose(0, 2, 3, 1, 4).reshape(RG, nb, nl * 512)
    slab = np.concatenate([dm_b, sm, codes], axis=2)
    assert slab.shape[2] == SLAB_BYTES[fmt]
    return np.ascontiguousarray(slab).reshape(-1)
