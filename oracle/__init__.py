"""ORACLE — test infrastructure, not product code.

ctypes binding of ``oracle/moe_oracle.cpp``: the plain fp64 CPU definition of
the block-quantized MoE layer.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may import this package.  It shares no code
with the CUDA path (``block_quantized_routed_gb300``), and imports nothing from
it.

Every function takes and returns numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

FMT_Q4K = 0
FMT_Q2K = 1
FMT_Q5K = 2
FMT_Q3K = 3
FMT_Q6K = 4
FMT_IQ2G = 5
ROUTE_SOFTMAX = 0
ROUTE_SIGMOID = 1
N_SUB = {FMT_Q4K: 8, FMT_Q2K: 16, FMT_Q5K: 8, FMT_Q3K: 16, FMT_Q6K: 16, FMT_IQ2G: 8}


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (portable C++17, no intrinsics)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_half_to_double.restype = ctypes.c_double
            lib.orc_iq2g_grid.argtypes = [P]
            lib.orc_iq2g_grid.restype = None
            lib.orc_unpack_sb.argtypes = [P, I, I64, I64, I64, I64, P, P, P, P]
            lib.orc_unpack_sb.restype = None
            lib.orc_dequant_matrix.argtypes = [P, I, I64, I64, P]
            lib.orc_dequant_matrix.restype = None
            lib.orc_q8k_quantize.argtypes = [P, I64, I64, P, P, P]
            lib.orc_q8k_quantize.restype = None
            lib.orc_subblock_dots.argtypes = [P, I, I64, I64, P, I64, P, P]
            lib.orc_subblock_dots.restype = None
            lib.orc_qmatvec.argtypes = [P, I, I64, I64, P, P, I64, P, I]
            lib.orc_qmatvec.restype = None
            lib.orc_superblock_sums.argtypes = [P, I, I64, I64, P, I64, P, P]
            lib.orc_superblock_sums.restype = None
            lib.orc_qmatvec_absterms.argtypes = [P, I, I64, I64, P, P, I64, P, I]
            lib.orc_qmatvec_absterms.restype = None
            lib.orc_route.argtypes = [P, P, P, I64, I64, I64, I64, I, P, P, P, P, P]
            lib.orc_route.restype = None
            lib.orc_bucket.argtypes = [P, I64, I64, I64, I64, P, P, P]
            lib.orc_bucket.restype = None
            lib.orc_expert_ffn.argtypes = [P, P, P, I, I64, I64, P, P, I64, P, P, P, P, I]
            lib.orc_expert_ffn.restype = None
            lib.orc_layer_forward.argtypes = [I, I64, I64, I64, I64, I64, I, P, P, P, P, P, P, P,
                                              I64, P, P, P, P, P, I]
            lib.orc_layer_forward.restype = None
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def half_to_double(bits: int) -> float:
    return _load().orc_half_to_double(int(bits))


def iq2g_grid() -> np.ndarray:
    """The IQ2-style grid C as int32 [256, 8] (magnitudes 1, 3, 5)."""
    out = np.zeros((256, 8), np.int32)
    _load().orc_iq2g_grid(out.ctypes.data)
    return out


def unpack_sb(w: np.ndarray, fmt: int, N: int, K: int, n: int, b: int):
    """Fields of super-block (row n, block b): (q[256], sc[ns], mn[ns], d, dmin);
    mn and dmin are 0 for the formats without a min."""
    w = _c(w, np.uint8)
    q = np.zeros(256, np.int32)
    sc = np.zeros(N_SUB[fmt], np.int32)
    mn = np.zeros(N_SUB[fmt], np.int32)
    dd = np.zeros(2, np.float64)
    _load().orc_unpack_sb(_p(w), fmt, N, K, n, b, _p(q), _p(sc), _p(mn), _p(dd))
    return q, sc, mn, float(dd[0]), float(dd[1])


def dequant_matrix(w: np.ndarray, fmt: int, N: int, K: int) -> np.ndarray:
    w = _c(w, np.uint8)
    out = np.zeros((N, K), np.float64)
    _load().orc_dequant_matrix(_p(w), fmt, N, K, _p(out))
    return out


def q8k_quantize(x: np.ndarray):
    """q8_K of fp32 x[T, K]: (q int8 [T, K], d fp32 [T, K/256], bsum16 int16 [T, K/16])."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x[None, :]
    T, K = x.shape
    if K % 256:
        raise ValueError("K must be a multiple of 256")
    q = np.zeros((T, K), np.int8)
    d = np.zeros((T, K // 256), np.float32)
    bs = np.zeros((T, K // 16), np.int16)
    _load().orc_q8k_quantize(_p(x), T, K, _p(q), _p(d), _p(bs))
    return q, d, bs


def subblock_dots(w: np.ndarray, fmt: int, N: int, K: int, qa: np.ndarray):
    """(isum int32 [T, N, nb, ns], bsum int32 [T, nb, ns])."""
    w = _c(w, np.uint8)
    qa = _c(qa, np.int8)
    T = qa.shape[0]
    nb, ns = K // 256, N_SUB[fmt]
    isum = np.zeros((T, N, nb, ns), np.int32)
    bsum = np.zeros((T, nb, ns), np.int32)
    _load().orc_subblock_dots(_p(w), fmt, N, K, _p(qa), T, _p(isum), _p(bsum))
    return isum, bsum


def superblock_sums(w: np.ndarray, fmt: int, N: int, K: int, qa: np.ndarray):
    """(S int64 [T, N, K/256], M int64 [T, N, K/256]): per super-block
    S = sum_j sc_j * isum_j and M = sum_j mn_j * bsum_j."""
    w = _c(w, np.uint8)
    qa = _c(qa, np.int8)
    T = qa.shape[0]
    S = np.zeros((T, N, K // 256), np.int64)
    M = np.zeros((T, N, K // 256), np.int64)
    _load().orc_superblock_sums(_p(w), fmt, N, K, _p(qa), T, _p(S), _p(M))
    return S, M


def qmatvec(w: np.ndarray, fmt: int, N: int, K: int, qa: np.ndarray, da: np.ndarray,
            nthreads: int | None = None) -> np.ndarray:
    w = _c(w, np.uint8)
    qa = _c(qa, np.int8)
    da = _c(da, np.float32)
    T = qa.shape[0]
    y = np.zeros((T, N), np.float64)
    _load().orc_qmatvec(_p(w), fmt, N, K, _p(qa), _p(da), T, _p(y), nthreads or default_threads())
    return y


def qmatvec_absterms(w: np.ndarray, fmt: int, N: int, K: int, qa: np.ndarray, da: np.ndarray,
                     nthreads: int | None = None) -> np.ndarray:
    """a [T, N]: the sum of the magnitudes of the super-block terms that
    qmatvec adds into each output (|qmatvec| <= a), for error bounds."""
    w = _c(w, np.uint8)
    qa = _c(qa, np.int8)
    da = _c(da, np.float32)
    T = qa.shape[0]
    a = np.zeros((T, N), np.float64)
    _load().orc_qmatvec_absterms(_p(w), fmt, N, K, _p(qa), _p(da), T, _p(a), nthreads or default_threads())
    return a


def route(x, wr, bias, k: int, route_kind: int, forced_ids=None):
    """(logits fp64 [T, E], ids int32 [T, k], gates fp64 [T, k], gap fp64 [T])."""
    x = _c(x, np.float32)
    wr = _c(wr, np.float32)
    T, H = x.shape
    E = wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    f = None if forced_ids is None else _c(forced_ids, np.int32)
    logits = np.zeros((T, E), np.float64)
    ids = np.zeros((T, k), np.int32)
    gates = np.zeros((T, k), np.float64)
    gap = np.zeros(T, np.float64)
    _load().orc_route(_p(x), _p(wr), _p(b), T, H, E, k, route_kind, _p(f), _p(logits), _p(ids),
                      _p(gates), _p(gap))
    return logits, ids, gates, gap


def bucket(ids: np.ndarray, E: int, S: int):
    """(counts [E+S], offsets [E+S+1], perm [T*k + S*T]) of the routed pairs."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.zeros(E + S, np.int32)
    offsets = np.zeros(E + S + 1, np.int32)
    perm = np.zeros(T * k + S * T, np.int32)
    _load().orc_bucket(_p(ids), T, k, E, S, _p(counts), _p(offsets), _p(perm))
    return counts, offsets, perm


def expert_ffn(gate, up, down, fmt: int, H: int, I: int, xq, xd, nthreads: int | None = None,
               return_h: bool = False):
    """y fp64 [T, H] of one expert on q8_K rows (xq [T, H], xd [T, H/256])."""
    gate, up, down = (_c(a, np.uint8) for a in (gate, up, down))
    xq = _c(xq, np.int8)
    xd = _c(xd, np.float32)
    T = xq.shape[0]
    y = np.zeros((T, H), np.float64)
    h = np.zeros((T, I), np.float32)
    hq = np.zeros((T, I), np.int8)
    hd = np.zeros((T, I // 256), np.float32)
    _load().orc_expert_ffn(_p(gate), _p(up), _p(down), fmt, H, I, _p(xq), _p(xd), T, _p(y), _p(h),
                           _p(hq), _p(hd), nthreads or default_threads())
    if return_h:
        return y, h, hq, hd
    return y


def layer_forward(fmt: int, H: int, I: int, E: int, k: int, S: int, route_kind: int,
                  experts, wr, bias, x, residual=None, forced_ids=None, nthreads: int | None = None):
    """The MoE layer.  experts: list of E+S (gate, up, down) byte arrays, or None
    for an expert that is not present.  Returns (out fp64 [T, H], ids, gates, gap)."""
    assert len(experts) == E + S
    keep = []
    arr = [(ctypes.c_void_p * (E + S))() for _ in range(3)]
    for e, ex in enumerate(experts):
        if ex is None:
            for m in range(3):
                arr[m][e] = None
            continue
        mats = [_c(a, np.uint8) for a in ex]
        keep.append(mats)
        for m in range(3):
            arr[m][e] = mats[m].ctypes.data
    x = _c(x, np.float32)
    T = x.shape[0]
    wr = _c(wr, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    r = None if residual is None else _c(residual, np.float32)
    f = None if forced_ids is None else _c(forced_ids, np.int32)
    out = np.zeros((T, H), np.float64)
    ids = np.zeros((T, k), np.int32)
    gates = np.zeros((T, k), np.float64)
    gap = np.zeros(T, np.float64)
    _load().orc_layer_forward(fmt, H, I, E, k, S, route_kind, *[ctypes.cast(a, ctypes.c_void_p) for a in arr],
                              _p(wr), _p(b),
                              _p(x), _p(r), T, _p(f), _p(out), _p(ids), _p(gates), _p(gap),
                              nthreads or default_threads())
    del keep
    return out, ids, gates, gap
