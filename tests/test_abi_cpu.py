"""The C-ABI library on the CPU: it builds, loads, exports every function the
header declares, sizes workspaces, and rejects bad arguments on the host
before any GPU work (no compute call is made here)."""
import ctypes

import pytest

import block_quantized_routed_gb300 as moe
from block_quantized_routed_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.load()


def desc(**kw):
    d = dict(H=2048, I=512, E=256, top_k=8, n_shared=1, route=0, fmt=0, T_max=1)
    d.update(kw)
    return moe.LayerDesc(**d)


def test_every_declared_function_is_exported(lib):
    names = _build.header_functions()
    assert len(names) >= 13
    for n in ["moe_q8k_quantize", "moe_route_topk", "moe_bucket", "moe_expert_ffn", "moe_combine",
              "moe_layer_forward"]:
        assert n in names
    raw = ctypes.CDLL(_build.LIB)
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings(lib):
    assert moe.moe_status_string(0) == "ok"
    assert "workspace" in moe.moe_status_string(moe.MOE_ERR_WORKSPACE)
    assert moe.moe_status_string(12345) == "unknown status"


@pytest.mark.parametrize("bad", [dict(H=500), dict(I=0), dict(E=0), dict(E=2000), dict(top_k=0), dict(top_k=17),
                                 dict(E=4, top_k=5), dict(n_shared=3), dict(route=2), dict(fmt=6), dict(T_max=0),
                                 dict(H=16640)])
def test_invalid_descriptors(lib, bad):
    d = desc(**bad)
    assert moe.moe_layer_workspace_size(d) == 0
    with pytest.raises(moe.MoeError):
        moe.moe_workspace_layout(d)


def test_workspace_layout_regions(lib):
    for d in [desc(), desc(H=4096, I=1024, E=512, top_k=10, T_max=8192, fmt=1, route=1),
              desc(H=512, I=256, E=16, top_k=2, n_shared=0, T_max=4)]:
        total = moe.moe_layer_workspace_size(d)
        lay = moe.moe_workspace_layout(d)
        assert lay.total == total > 0
        T, H, I, E, k, S = d.T_max, d.H, d.I, d.E, d.top_k, d.n_shared
        P = T * (k + S)
        sizes = dict(status=16, xq=T * H, xd=T * H // 256 * 4, xbs=T * H // 16 * 2, logits=T * E * 4,
                     ids=T * k * 4, gates=T * k * 4, gap=T * 4, counts=(E + S) * 4, offsets=(E + S + 1) * 4,
                     perm=P * 4, inv=P * 4, h=P * I * 4, hq=P * I, hd=P * I // 256 * 4, hbs=P * I // 16 * 2,
                     y=P * H * 4, phase_ns=128)
        spans = sorted((getattr(lay, n), getattr(lay, n) + s, n) for n, s in sizes.items())
        for (a0, a1, n0), (b0, b1, n1) in zip(spans, spans[1:]):
            assert a1 <= b0, (n0, n1)
        for a0, a1, n in spans:
            assert a0 % 256 == 0 and a1 <= total
    assert moe.moe_layer_workspace_size(desc(T_max=16)) > moe.moe_layer_workspace_size(desc(T_max=1))


def test_host_validation_rejects_before_launch(lib):
    L = moe.load()
    d = desc(T_max=4)
    fake = ctypes.c_void_p(0x10000)     # never dereferenced: validation fails first
    # T > T_max
    rc = L.moe_layer_forward(ctypes.byref(d), fake, fake, None, fake, None, fake, 5, None, None, fake, 1 << 40, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # NULL x
    rc = L.moe_layer_forward(ctypes.byref(d), fake, fake, None, None, None, fake, 1, None, None, fake, 1 << 40, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # workspace too small
    rc = L.moe_layer_forward(ctypes.byref(d), fake, fake, None, fake, None, fake, 1, None, None, fake, 1024, None)
    assert rc == moe.MOE_ERR_WORKSPACE
    # misaligned x
    rc = L.moe_layer_forward(ctypes.byref(d), fake, fake, None, ctypes.c_void_p(0x10004), None, fake, 1, None, None,
                             fake, 1 << 40, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # unsupported shape
    bad = desc(H=300)
    rc = L.moe_layer_forward(ctypes.byref(bad), fake, fake, None, fake, None, fake, 1, None, None, fake, 1 << 40, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    # T == 0 is a no-op
    rc = L.moe_layer_forward(ctypes.byref(d), None, None, None, None, None, None, 0, None, None, None, 0, None)
    assert rc == moe.MOE_OK
    assert L.moe_q8k_quantize(fake, 2, 300, fake, fake, None, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_q8k_quantize(fake, 0, 256, fake, fake, None, None) == moe.MOE_OK
    assert L.moe_route_topk(fake, fake, None, 1, 256, 8, 9, 0, fake, fake, fake, None, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_route_topk(fake, fake, None, 1, 256, 8, 2, 7, fake, fake, fake, None, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_bucket(fake, 4, 2, 8, 0, fake, fake, fake, None, fake, 8, None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_bucket(fake, 4, 2, 4096, 0, fake, fake, fake, None, fake, 1 << 20, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_combine(fake, fake, 1, 258, 2, 0, None, fake, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_debug_subblock_dots(0, fake, 256, 256, fake, 17, fake, fake, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_get_status(None, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_bucket_workspace_size(8192, 10, 512, 1) >= 80 * 513 * 4
    assert moe.moe_expert_ffn_workspace_size(d, 5) == 0


def test_stack_kernel_selection(lib):
    """moe_stack_forward's choice of single-launch kernel (host logic), on a
    152-SM device: layers with at most 2 gate/up + down items per SM, and
    heavier layers in stacks of 4 or more, take the dataflow kernel; heavy
    layers in shorter stacks the barrier-pipelined one."""
    dec = desc(H=2048, I=512, E=256, top_k=8, n_shared=1, T_max=1)          # 0.7 items per SM
    assert moe.moe_stack_kernel(dec, 40, 1, 152) == moe.STACK_DATAFLOW
    assert moe.moe_stack_kernel(dec, 1, 1, 152) == moe.STACK_DATAFLOW
    ver = desc(H=4096, I=1024, E=512, top_k=10, n_shared=1, route=1, fmt=1, T_max=4)  # 13.9 per SM
    assert moe.moe_stack_kernel(ver, 48, 4, 152) == moe.STACK_DATAFLOW
    assert moe.moe_stack_kernel(ver, 3, 4, 152) == moe.STACK_PIPELINED
    wide = desc(H=6144, I=2048, E=192, top_k=8, n_shared=0, T_max=16)     # 4.6 per SM at T = 1
    assert moe.moe_stack_kernel(wide, 1, 1, 152) == moe.STACK_PIPELINED
    assert moe.moe_stack_kernel(wide, 4, 1, 152) == moe.STACK_DATAFLOW
    heavy = desc(H=2048, I=1024, E=64, top_k=8, n_shared=1, T_max=8)      # the GPU test's heavy stack
    assert moe.moe_stack_kernel(heavy, 3, 8, 152) == moe.STACK_PIPELINED
    assert moe.moe_stack_kernel(heavy, 5, 8, 152) == moe.STACK_DATAFLOW
    # the same 0.7-items layer on a 32-SM part: 3.4 per SM
    assert moe.moe_stack_kernel(dec, 2, 1, 32) == moe.STACK_PIPELINED
    with pytest.raises(moe.MoeError) as e:
        moe.moe_stack_kernel(desc(H=512, I=256, E=16, top_k=2, T_max=32), 2, 17, 152)   # beyond 16 tokens
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as e:
        moe.moe_stack_kernel(dec, 0, 1, 152)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG


def test_layer_path_selection(lib):
    assert moe.moe_layer_path(desc(), 1) == moe.PATH_DECODE_FUSED
    # 40 tokens x 10 of 40 experts: 400 pairs, 10 per expert -> GEMV kernels
    assert moe.moe_layer_path(desc(H=512, I=256, E=40, top_k=10, T_max=40), 40) == moe.PATH_GEMV
    d = desc(H=4096, I=1024, E=512, top_k=10, T_max=8192)
    assert moe.moe_layer_path(d, 8192) == moe.PATH_TENSOR_PREFILL
    assert moe.moe_layer_path(d, 820) == moe.PATH_TENSOR_PREFILL      # 8200 pairs >= 16 * 512
    assert moe.moe_layer_path(d, 819) == moe.PATH_GEMV
    assert moe.moe_layer_path(d, 16) == moe.PATH_DECODE_FUSED
    assert moe.moe_layer_path(d, 26) == moe.PATH_GEMV                 # 260 pairs: beyond the single-CTA routing
    with pytest.raises(moe.MoeError):
        moe.moe_layer_path(d, 8193)
    with pytest.raises(moe.MoeError):
        moe.moe_layer_path(desc(H=300), 1)
    # the prefill work-item region exists only where the path can be taken
    assert moe.moe_layer_workspace_size(desc(H=4096, I=1024, E=512, top_k=10, T_max=819)) < \
        moe.moe_layer_workspace_size(desc(H=4096, I=1024, E=512, top_k=10, T_max=820)) - 16 * 1000


def test_kernel_launch_count_is_monotonic(lib):
    a = moe.moe_kernel_launch_count()
    L = moe.load()
    fake = ctypes.c_void_p(0x10000)
    assert L.moe_q8k_quantize(fake, 0, 256, fake, fake, None, None) == moe.MOE_OK   # T = 0: nothing launched
    assert moe.moe_kernel_launch_count() == a >= 0


def test_prefill_parity_cases_take_the_tensor_path(lib):
    # the whole-layer parity cases meant for the tcgen05 GEMMs really reach them
    for fmt, route, H, I, E, k, S, T in [(0, 0, 512, 256, 8, 2, 1, 512), (1, 1, 768, 512, 16, 4, 0, 300),
                                         (0, 1, 1024, 256, 4, 1, 2, 257), (0, 0, 512, 256, 8, 2, 1, 512),
                                         (0, 1, 4096, 1024, 512, 10, 1, 8192)]:
        d = desc(H=H, I=I, E=E, top_k=k, n_shared=S, route=route, fmt=fmt, T_max=T)
        assert moe.moe_layer_path(d, T) == moe.PATH_TENSOR_PREFILL


def test_stack_workspace_size(lib):
    d = desc(T_max=1)
    one = moe.moe_stack_workspace_size(d, 1)
    forty = moe.moe_stack_workspace_size(d, 40)
    assert one > moe.moe_layer_workspace_size(d)
    per_layer = (forty - one) / 39                           # per-layer buffers and counters
    assert 80 * 1024 < per_layer < 1 << 20                   # logits, x codes, routing, h [9, 512], y [9, 2048]
    assert moe.moe_stack_workspace_size(desc(T_max=4), 40) > forty
    assert moe.moe_stack_workspace_size(d, 0) == 0
    assert moe.moe_stack_workspace_size(desc(H=300), 4) == 0


@pytest.mark.parametrize("L,T,kw", [(40, 1, {}), (48, 4, dict(H=4096, I=1024, E=512, top_k=10, fmt=1, route=1))])
def test_stack_layer_layout_regions(lib, L, T, kw):
    """Per-layer buffers of the stack workspace: inside it, 256-byte aligned, one fixed stride per layer,
    and no two regions of one layer overlapping."""
    d = desc(T_max=T, **kw)
    total = moe.moe_stack_workspace_size(d, L)
    k, S = d.top_k, d.n_shared
    P = T * (k + S)
    size = dict(logits=T * d.E * 4, xq=T * d.H, xd=T * d.H // 256 * 4, xbs=T * d.H // 16 * 2, ids=T * k * 4,
                gates=T * k * 4, tok=P * 4, slot=P * 4, h=P * d.I * 4, y=P * d.H * 4)
    lays = [moe.moe_stack_layer_layout(d, L, T, l) for l in range(L)]
    stride = lays[1].logits - lays[0].logits
    assert stride > 0
    for l, lay in enumerate(lays):
        spans = sorted((getattr(lay, n), getattr(lay, n) + b) for n, b in size.items())
        assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))      # disjoint
        assert spans[-1][1] <= total
        assert lay.logits % 256 == 0 and lay.h % 256 == 0 and lay.y % 256 == 0
        assert lay.logits == lays[0].logits + l * stride
    # the layer workspace (status block first) comes before every layer's buffers
    assert lays[0].logits >= moe.moe_layer_workspace_size(d)
    with pytest.raises(moe.MoeError):
        moe.moe_stack_layer_layout(d, L, T, L)
    with pytest.raises(moe.MoeError):
        moe.moe_stack_layer_layout(desc(T_max=32), L, 32, 0)              # beyond the decode shapes
