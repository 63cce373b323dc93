"""Device-side weight generator (synth/csrc/synth_gen.cu): the same bytes as
synth.gen_matrix, made on the GPU for workloads of tens of GB."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

from . import layout, matrix_key

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "synth_gen.cu")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libsynth_gen.so")
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            build()
        lib = ctypes.CDLL(LIB)
        lib.synth_fill_matrix.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_uint64, ctypes.c_void_p]
        lib.synth_fill_matrix.restype = ctypes.c_int
        _lib = lib
    return _lib


def fill_matrix(dst_ptr: int, fmt: int, N: int, K: int, seed: int, layer: int, expert: int, mat: int,
                stream_ptr: int = 0) -> None:
    layout.check_shape(N, K)
    rc = _load().synth_fill_matrix(ctypes.c_void_p(dst_ptr), fmt, N, K, matrix_key(seed, layer, expert, mat),
                                   ctypes.c_void_p(stream_ptr))
    if rc != 0:
        raise RuntimeError(f"synth_fill_matrix failed ({rc})")


class ExpertBank:
    """All experts of `layers` MoE layers in one device buffer.

    Matrices of expert e of layer l: gate [I, H], up [I, H], down [H, I]; the
    shared experts are experts E .. E+S-1 of each layer.  Weight bytes follow
    synth.gen_matrix(fmt, ..., seed, l, e, mat)."""

    def __init__(self, fmt, H, I, n_experts, layers, seed, device="cuda", generate=True):
        import torch
        self.fmt, self.H, self.I, self.n_experts, self.layers, self.seed = fmt, H, I, n_experts, layers, seed
        self.gu_bytes = layout.matrix_bytes(fmt, I, H)
        self.dn_bytes = layout.matrix_bytes(fmt, H, I)
        self.expert_bytes = 2 * self.gu_bytes + self.dn_bytes
        total = self.expert_bytes * n_experts * layers
        self.buf = torch.empty(total, dtype=torch.uint8, device=device)
        self.base = self.buf.data_ptr()
        if generate:
            stream = torch.cuda.current_stream().cuda_stream
            for l in range(layers):
                for e in range(n_experts):
                    g, u, d = self.ptrs(l, e)
                    fill_matrix(g, fmt, I, H, seed, l, e, 0, stream)
                    fill_matrix(u, fmt, I, H, seed, l, e, 1, stream)
                    fill_matrix(d, fmt, H, I, seed, l, e, 2, stream)

    def ptrs(self, layer: int, expert: int):
        off = self.base + (layer * self.n_experts + expert) * self.expert_bytes
        return off, off + self.gu_bytes, off + 2 * self.gu_bytes

    def view(self, layer: int, expert: int, mat: int):
        off = (layer * self.n_experts + expert) * self.expert_bytes + (0, self.gu_bytes, 2 * self.gu_bytes)[mat]
        n = self.gu_bytes if mat < 2 else self.dn_bytes
        return self.buf[off:off + n]

    def table(self, layer: int, present=None):
        """int64 [n_experts, 3] device pointer table of one layer; experts not
        in `present` (if given) get NULL pointers."""
        import torch
        rows = []
        for e in range(self.n_experts):
            if present is not None and e not in present:
                rows.append([0, 0, 0])
            else:
                rows.append(list(self.ptrs(layer, e)))
        return torch.tensor(rows, dtype=torch.int64, device=self.buf.device)

    def host_expert(self, layer: int, expert: int):
        """(gate, up, down) bytes of one expert, generated on the host."""
        from . import gen_matrix
        return (gen_matrix(self.fmt, self.I, self.H, self.seed, layer, expert, 0),
                gen_matrix(self.fmt, self.I, self.H, self.seed, layer, expert, 1),
                gen_matrix(self.fmt, self.H, self.I, self.seed, layer, expert, 2))
