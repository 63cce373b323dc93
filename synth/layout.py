"""Byte layout of the block-quantized weight matrices ("row-group slabs").

A weight matrix W[N, K] (N rows, K columns, both multiples of 256) is cut
into 256-wide super-blocks (SB): row n, SB b covers columns 256*b ..
256*b+255.  Each SB carries the fields of its format (q: unsigned codes):

  Q4_K-style (144 B per SB): fp16 d, fp16 dmin, eight 32-weight sub-blocks
    with a 6-bit scale and a 6-bit min each (12 B), 256 4-bit codes (128 B);
    weight = d * scale_j * q - dmin * min_j.
  Q2_K-style (84 B per SB): fp16 d, fp16 dmin, sixteen 16-weight sub-blocks
    with a 4-bit scale and a 4-bit min each (16 B), 256 2-bit codes (64 B);
    weight = d * scale_j * q - dmin * min_j.
  Q5_K-style (176 B per SB): as Q4_K-style with 5-bit codes: the low 4 bits
    as in Q4_K (128 B) and a plane of the 5th bits (32 B);
    weight = d * scale_j * q - dmin * min_j.
  Q3_K-style (110 B per SB): fp16 d, sixteen 16-weight sub-blocks with a
    6-bit scale u_j each (12 B; the signed scale is u_j - 32), 256 3-bit
    codes: the low 2 bits as in Q2_K (64 B) and a plane of the 3rd bits
    (32 B); weight = d * (u_j - 32) * (q - 4).
  Q6_K-style (210 B per SB): fp16 d, sixteen 16-weight sub-blocks with an
    int8 scale each (16 B), 256 6-bit codes: the low 4 bits (128 B) and a
    plane of the high 2 bits (64 B); weight = d * scale_j * (q - 32).
  IQ2-style grid format (70 B per SB, 2.19 bits per weight): fp16 d, eight
    32-weight sub-blocks with a 4-bit scale t_j each (4 B), and per group
    g of 8 weights (32 groups, sub-block j = groups 4j..4j+3) a grid index
    u_g (1 B) and 7 sign bits (1 B; the 8th sign makes the number of minus
    signs even); weight 8g + i = d * (2 t_j + 1) * s_{g,i} * C[u_g][i].
    The grid C: the 256 vectors of {1, 3, 5}^8 with the smallest sum of
    squares, equal sums in increasing order of the base-3 number whose
    digits are (v_0 - 1)/2 .. (v_7 - 1)/2 (v_0 most significant); u = rank.
    (The pages name i-quant codebook formats but print no grid: this grid
    is this project's own.)

Placement.  Rows are grouped 32 at a time (row group rg = n // 32, lane
r = n % 32).  The matrix is the sequence of slabs (rg, b) in order
rg-major, b-minor; one slab holds SB b of the 32 rows of its group, field
by field:

  header  row r at hb*r: Q4_K/Q2_K/Q5_K: uint32 = d_bits | dmin_bits << 16
          (hb = 4); Q3_K/Q6_K: uint16 d_bits (hb = 2)
  sm      row r at 32*hb + smb*r: the scale(/min) bytes
  codes   code lines of 16 bytes: line l of row r at
          32*hb + 32*smb + 512*l + 16*r; the lines of the low-bit plane
          first, then those of the high-bit plane

  Q4_K: 4608 B per slab; line j (0..7) = sub-block j: byte i holds code i
        (low nibble) and code i+16 (high nibble).
  Q2_K: 2688 B; sub-block j (0..15) in line j // 4, bytes 4*(j%4)..+3:
        bits 2p..2p+1 of byte m hold code 4*p + m.
  Q5_K: 5632 B; lines 0..7: the low 4 bits as Q4_K; lines 8, 9 (5th bits):
        in line 8 + j // 4, byte i, bit 2*(j % 4) + h is bit 4 of code
        i + 16*h of sub-block j.
  Q3_K: 3520 B; lines 0..3: the low 2 bits as Q2_K; lines 4, 5 (3rd bits):
        sub-block j in line 4 + j // 8, bytes 4*((j // 2) % 4)..+3: bit
        p + 4*(j % 2) of byte m is bit 2 of code 4*p + m.
  Q6_K: 6720 B; lines 0..7 (low 4 bits): line l, byte i holds bits 0-3 of
        code i of sub-block 2l (low nibble) and of sub-block 2l + 1 (high
        nibble); lines 8..11 (high 2 bits): line 8 + j // 4, byte i, bits
        2*(j % 4)..+1 are bits 4-5 of code i of sub-block j.
  IQ2G: 2240 B; lines 0, 1: the grid indices, byte 16 l + i of the row =
        u_{16 l + i} (so sub-block j's four indices are word j % 4 of line
        j // 4); lines 2, 3: the sign bytes in the same order (bit i < 7 of
        byte g is 1 when weight 8g + i is negative; bit 7 is ignored).

Scale/min bytes: Q4_K/Q5_K: a 96-bit little-endian bit string; scale j is
bits 6j..6j+5 and min j is bits 48+6j..48+6j+5 (bit i of the string is bit
i%8 of byte i//8).  Q2_K: byte j = scale_j | min_j << 4.  Q3_K: the same
96-bit string holding u_0..u_15 at bits 6j..6j+5.  Q6_K: byte j = scale_j
as int8.  IQ2G: byte j // 2 holds t_j in its low (j even) or high (j odd)
nibble.

Logical SB bytes (what the generator draws): the code bytes of the planes in
order (code byte i of a plane goes to line i // 16 of that plane, byte
i % 16); the scale/min bytes in order; d and (where present) dmin.

Why this placement: in the decode kernels one lane owns one row, so every
16-byte load of a warp reads 512 contiguous bytes, and a whole row group is
one contiguous run of bytes (nb slabs) for bulk copies.
"""
from __future__ import annotations

import numpy as np

FMT_Q4K = 0
FMT_Q2K = 1
FMT_Q5K = 2
FMT_Q3K = 3
FMT_Q6K = 4
FMT_IQ2G = 5
FORMATS = (FMT_Q4K, FMT_Q2K, FMT_Q5K, FMT_Q3K, FMT_Q6K, FMT_IQ2G)
NAMES = {FMT_Q4K: "q4_k", FMT_Q2K: "q2_k", FMT_Q5K: "q5_k", FMT_Q3K: "q3_k", FMT_Q6K: "q6_k", FMT_IQ2G: "iq2_g"}

HDR_BYTES = {FMT_Q4K: 4, FMT_Q2K: 4, FMT_Q5K: 4, FMT_Q3K: 2, FMT_Q6K: 2, FMT_IQ2G: 2}   # per row
HAS_DMIN = {f: HDR_BYTES[f] == 4 for f in FORMATS}
SM_BYTES = {FMT_Q4K: 12, FMT_Q2K: 16, FMT_Q5K: 12, FMT_Q3K: 12, FMT_Q6K: 16, FMT_IQ2G: 4}
PLANES = {FMT_Q4K: (128,), FMT_Q2K: (64,), FMT_Q5K: (128, 32), FMT_Q3K: (64, 32), FMT_Q6K: (128, 64),
          FMT_IQ2G: (32, 32)}
CODE_BYTES = {f: sum(PLANES[f]) for f in FORMATS}
SB_BYTES = {f: HDR_BYTES[f] + SM_BYTES[f] + CODE_BYTES[f] for f in FORMATS}
N_SUB = {FMT_Q4K: 8, FMT_Q2K: 16, FMT_Q5K: 8, FMT_Q3K: 16, FMT_Q6K: 16, FMT_IQ2G: 8}
SUB_LEN = {f: 256 // N_SUB[f] for f in FORMATS}
CODE_BITS = {FMT_Q4K: 4, FMT_Q2K: 2, FMT_Q5K: 5, FMT_Q3K: 3, FMT_Q6K: 6, FMT_IQ2G: 2}
SLAB_BYTES = {f: 32 * SB_BYTES[f] for f in FORMATS}
SM_OFFSET = {f: 32 * HDR_BYTES[f] for f in FORMATS}
CODE_OFFSET = {f: SM_OFFSET[f] + 32 * SM_BYTES[f] for f in FORMATS}
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
         d_bits: np.ndarray, dmin_bits: np.ndarray | None) -> np.ndarray:
    """Place logical SB bytes [N, nb, ...] into the slab layout; returns uint8 [bytes].
    dmin_bits is ignored for the formats without a dmin field."""
    check_shape(N, K)
    nb = K // 256
    RG = N // 32
    cb = CODE_BYTES[fmt]
    smb = SM_BYTES[fmt]
    assert code_bytes.shape == (N, nb, cb) and sm_bytes.shape == (N, nb, smb)
    if HAS_DMIN[fmt]:
        hdr = (d_bits.astype(np.uint32) | (dmin_bits.astype(np.uint32) << np.uint32(16))).astype('<u4')
    else:
        hdr = d_bits.astype('<u2')
    # [RG, 32, nb] -> [RG, nb, 32]
    hdr = np.ascontiguousarray(hdr.reshape(RG, 32, nb).transpose(0, 2, 1))
    hdr_b = hdr.view(np.uint8).reshape(RG, nb, 32 * HDR_BYTES[fmt])
    sm = sm_bytes.reshape(RG, 32, nb, smb).transpose(0, 2, 1, 3).reshape(RG, nb, 32 * smb)
    parts = [hdr_b, sm]
    off = 0
    for pb in PLANES[fmt]:
        # code byte i of the plane -> line i // 16, byte i % 16; lines are [32 rows][16 B]
        nl = pb // 16
        plane = code_bytes[:, :, off:off + pb]
        parts.append(plane.reshape(RG, 32, nb, nl, 16).transpose(0, 2, 3, 1, 4).reshape(RG, nb, nl * 512))
        off += pb
    slab = np.concatenate(parts, axis=2)
    assert slab.shape[2] == SLAB_BYTES[fmt]
    return np.ascontiguousarray(slab).reshape(-1)
