"""block_quantized_routed_gb300 — the block-quantized routed MoE layer on GB300.

A thin ctypes binding of the C ABI in include/moe_q8k.h (libmoe_q8k.so, built
in-tree for sm_103a).  Every function has the name of its C entry point and
only marshals arguments: device tensors go in as raw pointers, the stream is
torch's current CUDA stream, and a negative status raises MoeError.  Every
step of the layer runs in the library's CUDA kernels; there is no other
implementation behind these names, and loading fails loudly when the library
has not been built.

torch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = [
    "MoeError", "LayerDesc", "WsLayout", "FMT_Q4K", "FMT_Q2K", "FMT_Q5K", "FMT_Q3K", "FMT_Q6K", "FMT_IQ2G",
    "ROUTE_SOFTMAX",
    "ROUTE_SIGMOID",
    "load", "lib", "moe_q8k_quantize", "moe_route_topk", "moe_bucket", "moe_bucket_workspace_size",
    "moe_expert_ffn", "moe_expert_ffn_workspace_size", "moe_combine", "moe_layer_forward",
    "moe_layer_workspace_size", "moe_workspace_layout", "moe_stack_forward", "moe_stack_workspace_size", "stack_pointer_table", "moe_layer_forward_noalloc", "moe_get_status", "moe_status_string",
    "moe_debug_subblock_dots", "moe_trace_events", "moe_trace_used", "moe_kernel_launch_count", "moe_layer_path",
    "PATH_DECODE_FUSED", "PATH_GEMV", "PATH_TENSOR_PREFILL", "expert_table", "MoeLayer",
    "moe_stack_kernel", "STACK_PIPELINED", "STACK_DATAFLOW", "StackLayerLayout", "moe_stack_layer_layout",
    "ws_view", "moe_debug_prefill_sums", "moe_debug_prefill_sums_workspace_size", "moe_prefill_tile_tokens",
]

FMT_Q4K = 0
FMT_Q2K = 1
FMT_Q5K = 2
FMT_Q3K = 3
FMT_Q6K = 4
FMT_IQ2G = 5
ROUTE_SOFTMAX = 0
ROUTE_SIGMOID = 1
SB_BYTES = {FMT_Q4K: 144, FMT_Q2K: 84, FMT_Q5K: 176, FMT_Q3K: 110, FMT_Q6K: 210, FMT_IQ2G: 70}
N_SUB = {FMT_Q4K: 8, FMT_Q2K: 16, FMT_Q5K: 8, FMT_Q3K: 16, FMT_Q6K: 16, FMT_IQ2G: 8}

PATH_DECODE_FUSED = 0
PATH_GEMV = 1
PATH_TENSOR_PREFILL = 2

STACK_PIPELINED = 1
STACK_DATAFLOW = 2

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_DEVICE_BOUNDS = -5
MOE_ERR_DEVICE_TIMEOUT = -6


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        extra = ""
        if status == MOE_ERR_CUDA:
            extra = f", cudaError {int(load().moe_last_cuda_error())}"
        super().__init__(f"{where}: {moe_status_string(status)} ({status}{extra})")


class LayerDesc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("route", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("T_max", ctypes.c_int32)]


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "xq", "xd", "xbs", "logits", "ids", "gates", "gap", "counts", "offsets", "perm", "inv",
                 "h", "hq", "hd", "hbs", "y", "phase_ns", "total")]


class StackLayerLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("logits", "xq", "xd", "xbs", "ids", "gates", "tok", "slot", "h", "y")]


_lib = None


def load():
    """Load libmoe_q8k.so (built by __graft_entry__.build() or _build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"{_build.LIB} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(_build.LIB)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    D = ctypes.POINTER(LayerDesc)
    sig = {
        "moe_layer_workspace_size": (SZ, [D]),
        "moe_workspace_layout": (ctypes.c_int, [D, ctypes.POINTER(WsLayout)]),
        "moe_q8k_quantize": (ctypes.c_int, [P, I64, I64, P, P, P, P]),
        "moe_route_topk": (ctypes.c_int, [P, P, P, I32, I32, I32, I32, I32, P, P, P, P, P]),
        "moe_bucket_workspace_size": (SZ, [I32, I32, I32, I32]),
        "moe_bucket": (ctypes.c_int, [P, I32, I32, I32, I32, P, P, P, P, P, SZ, P]),
        "moe_expert_ffn_workspace_size": (SZ, [D, I32]),
        "moe_expert_ffn": (ctypes.c_int, [D, P, P, P, P, P, P, P, I32, P, P, SZ, P]),
        "moe_combine": (ctypes.c_int, [P, P, I32, I32, I32, I32, P, P, P]),
        "moe_layer_forward": (ctypes.c_int, [D, P, P, P, P, P, P, I32, P, P, P, SZ, P]),
        "moe_stack_forward": (ctypes.c_int, [D, I32, P, I32, P, SZ, P]),
        "moe_stack_workspace_size": (SZ, [D, I32]),
        "moe_layer_forward_noalloc": (ctypes.c_int, [D, P, P, P, P, P, P, I32, P, P, P]),
        "moe_get_status": (ctypes.c_int, [P, P]),
        "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "moe_debug_subblock_dots": (ctypes.c_int, [I32, P, I32, I32, P, I32, P, P, P]),
        "moe_trace_events": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), I32]),
        "moe_trace_used": (I32, []),
        "moe_kernel_launch_count": (ctypes.c_ulonglong, []),
        "moe_last_cuda_error": (ctypes.c_int, []),
        "moe_debug_wait_timeout": (ctypes.c_int, [P, I32, P]),
        "moe_layer_path": (ctypes.c_int, [D, I32]),
        "moe_prefill_tile_tokens": (ctypes.c_int, []),
        "moe_stack_kernel": (ctypes.c_int, [D, I32, I32, I32]),
        "moe_stack_layer_layout": (ctypes.c_int, [D, I32, I32, I32, ctypes.POINTER(StackLayerLayout)]),
        "moe_debug_prefill_sums_workspace_size": (SZ, [I32, I32, I32]),
        "moe_debug_prefill_sums": (ctypes.c_int, [I32, P, I32, I32, P, P, P, I32, P, P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def lib():
    return load()


# ----------------------------------------------------------------- helpers

def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def _desc(d) -> LayerDesc:
    if isinstance(d, LayerDesc):
        return d
    return LayerDesc(**d)


# ----------------------------------------------------------------- C ABI wrappers

def moe_layer_workspace_size(desc) -> int:
    return int(load().moe_layer_workspace_size(ctypes.byref(_desc(desc))))


def moe_workspace_layout(desc) -> WsLayout:
    out = WsLayout()
    _check(load().moe_workspace_layout(ctypes.byref(_desc(desc)), ctypes.byref(out)), "moe_workspace_layout")
    return out


def moe_q8k_quantize(x, q, d, bsum16=None, stream=None):
    T, K = x.shape
    _check(load().moe_q8k_quantize(_ptr(x), T, K, _ptr(q), _ptr(d), _ptr(bsum16), _stream(stream)),
           "moe_q8k_quantize")


def moe_route_topk(x, w_router, bias, k, route, logits, ids, gates, gap=None, stream=None):
    T, H = x.shape
    E = w_router.shape[0]
    _check(load().moe_route_topk(_ptr(x), _ptr(w_router), _ptr(bias), T, H, E, k, route, _ptr(logits), _ptr(ids),
                                 _ptr(gates), _ptr(gap), _stream(stream)), "moe_route_topk")


def moe_bucket_workspace_size(T, k, E, n_shared) -> int:
    return int(load().moe_bucket_workspace_size(T, k, E, n_shared))


def moe_bucket(ids, E, n_shared, counts, offsets, perm, inv, ws, stream=None):
    T, k = ids.shape
    _check(load().moe_bucket(_ptr(ids), T, k, E, n_shared, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
                             _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_bucket")


def moe_expert_ffn_workspace_size(desc, T) -> int:
    return int(load().moe_expert_ffn_workspace_size(ctypes.byref(_desc(desc)), T))


def moe_expert_ffn(desc, table, q, d, bsum16, counts, offsets, perm, T, y_slots, ws, stream=None):
    _check(load().moe_expert_ffn(ctypes.byref(_desc(desc)), _ptr(table), _ptr(q), _ptr(d), _ptr(bsum16),
                                 _ptr(counts), _ptr(offsets), _ptr(perm), T, _ptr(y_slots), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)), "moe_expert_ffn")


def moe_combine(y_slots, gates, T, H, k, n_shared, residual, out, stream=None):
    _check(load().moe_combine(_ptr(y_slots), _ptr(gates), T, H, k, n_shared, _ptr(residual), _ptr(out),
                              _stream(stream)), "moe_combine")


def moe_layer_forward(desc, table, w_router, router_bias, x, residual, out, ids_out, gates_out, ws, stream=None):
    T = x.shape[0]
    _check(load().moe_layer_forward(ctypes.byref(_desc(desc)), _ptr(table), _ptr(w_router), _ptr(router_bias),
                                    _ptr(x), _ptr(residual), _ptr(out), T, _ptr(ids_out), _ptr(gates_out), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)), "moe_layer_forward")


def moe_layer_forward_noalloc(desc, table, w_router, router_bias, x, residual, out, ids_out=None, gates_out=None,
                              stream=None):
    """moe_layer_forward with the library's own fixed scratch (no workspace, no allocation)."""
    T = x.shape[0]
    _check(load().moe_layer_forward_noalloc(ctypes.byref(_desc(desc)), _ptr(table), _ptr(w_router),
                                            _ptr(router_bias), _ptr(x), _ptr(residual), _ptr(out), T,
                                            _ptr(ids_out), _ptr(gates_out), _stream(stream)),
           "moe_layer_forward_noalloc")


def moe_stack_workspace_size(desc, n_layers) -> int:
    return int(load().moe_stack_workspace_size(ctypes.byref(_desc(desc)), n_layers))


def moe_stack_layer_layout(desc, n_layers, T, layer) -> StackLayerLayout:
    """Byte offsets of one stack layer's buffers in a moe_stack_forward workspace."""
    out = StackLayerLayout()
    _check(load().moe_stack_layer_layout(ctypes.byref(_desc(desc)), n_layers, T, layer, ctypes.byref(out)),
           "moe_stack_layer_layout")
    return out


def ws_view(ws, offset, dtype, shape):
    """A typed view of `shape` elements at byte `offset` of a uint8 workspace tensor."""
    import torch
    n = 1
    for s_ in shape:
        n *= s_
    itemsize = torch.empty((), dtype=dtype).element_size()
    return ws[offset:offset + n * itemsize].view(dtype).view(*shape)


def moe_stack_forward(desc, layers, T, ws, stream=None):
    """layers: int64 device tensor [n_layers, 8] of moe_layer_ptrs records
    (see stack_pointer_table)."""
    _check(load().moe_stack_forward(ctypes.byref(_desc(desc)), layers.shape[0], _ptr(layers), T, _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)), "moe_stack_forward")


def stack_pointer_table(rows, device="cuda"):
    """Device array of moe_layer_ptrs from per-layer dicts with keys table,
    w_router, router_bias, x, residual, out, ids_out, gates_out (tensors or
    None).  The returned tensor keeps references to every tensor it points at."""
    import torch
    keys = ["table", "w_router", "router_bias", "x", "residual", "out", "ids_out", "gates_out"]
    vals = [[0 if r.get(k2) is None else int(r[k2].data_ptr()) for k2 in keys] for r in rows]
    t = torch.tensor(vals, dtype=torch.int64, device=device)
    t._refs = [dict(r) for r in rows]
    return t


def moe_get_status(ws, stream=None) -> int:
    return int(load().moe_get_status(_ptr(ws), _stream(stream)))


_trace_keep = None


def moe_trace_events(events):
    """Profiling hook: `events` is a list of torch.cuda.Event(enable_timing=True)
    (or None to turn the hook off); see include/moe_q8k.h."""
    global _trace_keep
    if not events:
        _trace_keep = None
        _check(load().moe_trace_events(None, 0), "moe_trace_events")
        return
    import torch
    fresh = [ev for ev in events if not ev.cuda_event]
    for ev in fresh:                    # torch creates the CUDA event on its first record
        ev.record(torch.cuda.current_stream())
    if fresh:
        torch.cuda.current_stream().synchronize()
    if any(not ev.cuda_event for ev in events):
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_trace_events")
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(ev.cuda_event) for ev in events])
    _trace_keep = (arr, list(events))
    _check(load().moe_trace_events(arr, len(events)), "moe_trace_events")


def moe_trace_used() -> int:
    return int(load().moe_trace_used())


def moe_debug_wait_timeout(ws, limit_us, stream=None):
    """Test hook: a bounded device wait that runs out (see include/moe_q8k.h)."""
    _check(load().moe_debug_wait_timeout(_ptr(ws), limit_us, _stream(stream)), "moe_debug_wait_timeout")


def moe_kernel_launch_count() -> int:
    return int(load().moe_kernel_launch_count())


def moe_layer_path(desc, T) -> int:
    rc = int(load().moe_layer_path(ctypes.byref(_desc(desc)), T))
    if rc < 0:
        raise MoeError(rc, "moe_layer_path")
    return rc


def moe_prefill_tile_tokens() -> int:
    """Token tile n of the tensor-core prefill path: an expert with c tokens gets ceil(c / n) tiles of
    balanced size."""
    return int(load().moe_prefill_tile_tokens())


def moe_stack_kernel(desc, n_layers, T, n_sms=0) -> int:
    """Which single-launch kernel moe_stack_forward takes (STACK_DATAFLOW or STACK_PIPELINED)."""
    rc = int(load().moe_stack_kernel(ctypes.byref(_desc(desc)), n_layers, T, n_sms))
    if rc < 0:
        raise MoeError(rc, "moe_stack_kernel")
    return rc


def moe_debug_subblock_dots(fmt, w, N, K, q, isum, bsum, stream=None):
    T = q.shape[0]
    _check(load().moe_debug_subblock_dots(fmt, _ptr(w), N, K, _ptr(q), T, _ptr(isum), _ptr(bsum), _stream(stream)),
           "moe_debug_subblock_dots")


def moe_debug_prefill_sums_workspace_size(N, K, T) -> int:
    return int(load().moe_debug_prefill_sums_workspace_size(N, K, T))


def moe_debug_prefill_sums(fmt, w, N, K, q, d, bsum16, S, M, ws, stream=None):
    """Test hook: integer super-block sums S, M (int32 [T, N, K/256]) of the tensor-core path."""
    T = q.shape[0]
    _check(load().moe_debug_prefill_sums(fmt, _ptr(w), N, K, _ptr(q), _ptr(d), _ptr(bsum16), T, _ptr(S), _ptr(M),
                                         _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_debug_prefill_sums")


# ----------------------------------------------------------------- convenience

def expert_table(experts, device="cuda"):
    """Device pointer table (int64 [n, 3]) from a list of (gate, up, down)
    uint8 device tensors or None (not present).  The returned tensor keeps
    references to the expert tensors, so their memory stays allocated for
    as long as the table is alive."""
    import torch
    rows = []
    for ex in experts:
        if ex is None:
            rows.append([0, 0, 0])
        else:
            rows.append([int(m.data_ptr()) for m in ex])
    table = torch.tensor(rows, dtype=torch.int64, device=device)
    table._experts = [None if ex is None else tuple(ex) for ex in experts]
    return table


class MoeLayer:
    """One layer: its descriptor, expert pointer table, router weight and a
    zeroed workspace; forward() runs moe_layer_forward on torch's current stream."""

    def __init__(self, desc, table, w_router, router_bias=None, device="cuda"):
        import torch
        self.desc = _desc(desc)
        self.table = table
        self.w_router = w_router
        self.router_bias = router_bias
        nbytes = moe_layer_workspace_size(self.desc)
        if nbytes == 0:
            raise MoeError(MOE_ERR_UNSUPPORTED, "MoeLayer")
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.layout = moe_workspace_layout(self.desc)

    def forward(self, x, residual=None, out=None, ids_out=None, gates_out=None, stream=None):
        import torch
        if out is None:
            out = torch.empty_like(x)
        moe_layer_forward(self.desc, self.table, self.w_router, self.router_bias, x, residual, out, ids_out,
                          gates_out, self.ws, stream)
        return out

    def ws_view(self, name, dtype, shape):
        """A view of an intermediate region of the workspace (after a call)."""
        return MoeLayer.ws_view_of(self.ws, self.layout, name, dtype, shape)

    @staticmethod
    def ws_view_of(ws, layout, name, dtype, shape):
        import torch
        off = getattr(layout, name)
        n = 1
        for s in shape:
            n *= s
        itemsize = torch.empty((), dtype=dtype).element_size()
        return ws[off:off + n * itemsize].view(dtype).view(*shape)
