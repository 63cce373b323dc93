"""moe_layer_forward_noalloc: the allocation-free variant of moe_layer_forward.

Some callers cannot allocate device memory where they run the layer (their
engine owns the whole device through its own pool, or allocating could
synchronise the device mid-step), so this entry point takes no workspace and
uses a fixed array inside the library.  This test calls it through the C ABI
twice in a row and checks each result against moe_layer_forward with a
workspace, under the tolerance the other tests use.  It sits in a file that
pytest collects last."""
import numpy as np
import pytest

import synth
from synth.layout import FMT_Q4K, FMT_Q2K
from tests.gpu_util import assert_close_rows, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


# the first two shapes take the single-launch decode kernel; the third
# (T*k = 320 > 256 pairs) the multi-kernel route/bucket/GEMV path, whose tile
# count and arrival counters also live in the shared array
@pytest.mark.parametrize("fmt,route,H,I,E,k,S,T", [(FMT_Q4K, 0, 2048, 512, 64, 8, 1, 1),
                                                   (FMT_Q2K, 1, 1024, 512, 32, 4, 1, 4),
                                                   (FMT_Q4K, 0, 1024, 256, 32, 8, 1, 40)])
def test_noalloc_matches_workspace_entry_point_twice(fmt, route, H, I, E, k, S, T):
    import block_quantized_routed_gb300 as moe
    moe.load()
    dev = lambda a: to_dev(a, torch)
    seed = 60 + T
    experts = [tuple(dev(synth.gen_matrix(fmt, n, kk, seed, 0, e, m)) for m, (n, kk) in
                     enumerate([(I, H), (I, H), (H, I)])) for e in range(E + S)]
    table = moe.expert_table(experts)
    wr = dev(synth.router_weight(E, H, seed))
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=route, fmt=fmt, T_max=T)
    assert moe.moe_layer_workspace_size(desc) <= 16 << 20
    if T * k > 256:
        assert moe.moe_layer_path(desc, T) == moe.PATH_GEMV
    layer = moe.MoeLayer(desc, table, wr)
    for rep in range(2):                      # two calls in a row: the shared scratch is reused
        x = dev(synth.activations(T, H, seed, rep=rep))
        want = layer.forward(x, residual=x)
        got = torch.empty_like(x)
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        moe.moe_layer_forward_noalloc(desc, table, wr, None, x, x, got, ids_out=ids)
        torch.cuda.synchronize()
        assert_close_rows(got.cpu().numpy(), want.cpu().numpy(), f"call {rep}")
        assert (ids.cpu().numpy() >= 0).all() and (ids.cpu().numpy() < E).all()


def test_noalloc_rejects_oversized_workspace():
    import block_quantized_routed_gb300 as moe
    moe.load()
    desc = dict(H=4096, I=1024, E=512, top_k=10, n_shared=1, route=1, fmt=FMT_Q4K, T_max=8192)
    assert moe.moe_layer_workspace_size(desc) > 16 << 20
    x = torch.zeros((8192, 4096), dtype=torch.float32, device="cuda")
    dummy = torch.zeros(16, dtype=torch.int64, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_forward_noalloc(desc, dummy, x, None, x, None, x)
    assert e.value.status == moe.MOE_ERR_WORKSPACE
