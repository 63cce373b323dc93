"""GPU parity of every step of the layer against the oracle, through the C ABI.

Integer results are compared bit for bit: q8_K codes/scales/16-sums, the
integer sub-block dot sums of the device dot routine, expert ids (away from
near-ties), bucket counts/offsets/permutation.  Floating-point results use
the relative rule of tests/gpu_util.py, and the layer cases also the fp32
forward-error bound of oracle/parity.py.  Sizes span several 32-row
groups, several 256-column blocks and ragged token counts."""
import numpy as np
import pytest

import oracle
import synth
from synth.layout import FMT_Q4K, FMT_Q2K, FMT_Q5K, FMT_Q3K, FMT_Q6K, FMT_IQ2G, FORMATS, N_SUB
from tests import fieldpack
from oracle import parity
from tests.gpu_util import assert_close_rows, routing_ok, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import block_quantized_routed_gb300 as m
    m.load()
    return m


def dev(a):
    return to_dev(a, torch)


# ------------------------------------------------------------------ q8_K

@pytest.mark.parametrize("T,K", [(1, 256), (4, 512), (13, 2048), (64, 6144)])
def test_q8k_quantize_bit_exact(moe, T, K):
    rng = np.random.default_rng(T * K)
    x = (rng.standard_normal((T, K)) * rng.uniform(1e-3, 1e2, (T, 1))).astype(np.float32)
    x[0, :256] = 0.0                                     # all-zero block
    if T > 2:
        x[1, :256] = np.round(x[1, :256] * 2) / 2        # many exact .5 ratios
        x[2, 5] = 1e-42                                  # subnormal inside a block
    q = torch.empty((T, K), dtype=torch.int8, device="cuda")
    d = torch.empty((T, K // 256), dtype=torch.float32, device="cuda")
    bs = torch.empty((T, K // 16), dtype=torch.int16, device="cuda")
    moe.moe_q8k_quantize(dev(x), q, d, bs)
    rq, rd, rbs = oracle.q8k_quantize(x)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(d.cpu().numpy().view(np.uint32), rd.view(np.uint32))
    np.testing.assert_array_equal(bs.cpu().numpy(), rbs)


def test_q8k_golden_blocks(moe):
    import json, os
    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "q8k_blocks.json")))["cases"]
    x = np.zeros((len(cases), 256), np.float32)
    for i, c in enumerate(cases):
        for k, v in c["x"].items():
            x[i, int(k)] = v
    q = torch.empty((len(cases), 256), dtype=torch.int8, device="cuda")
    d = torch.empty((len(cases), 1), dtype=torch.float32, device="cuda")
    bs = torch.empty((len(cases), 16), dtype=torch.int16, device="cuda")
    moe.moe_q8k_quantize(dev(x), q, d, bs)
    q, d, bs = q.cpu().numpy(), d.cpu().numpy(), bs.cpu().numpy()
    for i, c in enumerate(cases):
        want = np.zeros(256, np.int8)
        for k, v in c["q"].items():
            want[int(k)] = v
        np.testing.assert_array_equal(q[i], want)
        assert d[i, 0] == np.float32(c["d"])
        np.testing.assert_array_equal(bs[i], c["bsum16"])


# ------------------------------------------------------------------ integer dots

@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("N,K,T", [(256, 256, 1), (512, 1024, 3), (256, 2048, 16)])
def test_subblock_dots_bit_exact(moe, fmt, N, K, T):
    w = synth.gen_matrix(fmt, N, K, 5, 0, 1, 0)
    x = synth.activations(T, K, 5)
    xq, _, _ = oracle.q8k_quantize(x)
    ns = N_SUB[fmt]
    isum = torch.empty((T, N, K // 256, ns), dtype=torch.int32, device="cuda")
    bsum = torch.empty((T, K // 256, ns), dtype=torch.int32, device="cuda")
    moe.moe_debug_subblock_dots(fmt, dev(w), N, K, dev(xq), isum, bsum)
    risum, rbsum = oracle.subblock_dots(w, fmt, N, K, xq)
    np.testing.assert_array_equal(isum.cpu().numpy(), risum)
    np.testing.assert_array_equal(bsum.cpu().numpy(), rbsum)


@pytest.mark.parametrize("fmt", [FMT_Q5K, FMT_Q3K, FMT_Q6K])
def test_subblock_dots_extreme_fields(moe, fmt):
    """Every code at its largest value (every high bit set) against q_a = -127 and +127."""
    N, K = 256, 512
    ns = N_SUB[fmt]
    q = np.full((N, 2, 256), fieldpack.QMAX[fmt])
    sc = np.full((N, 2, ns), fieldpack.SCALE_RANGE[fmt][1])
    mn = np.full((N, 2, ns), fieldpack.MIN_RANGE[fmt][1])
    w = fieldpack.pack_fields(fmt, N, K, q, sc, mn, np.ones((N, 2), np.float16), np.ones((N, 2), np.float16))
    xq = np.stack([np.full(K, -127, np.int8), np.full(K, 127, np.int8)])
    isum = torch.empty((2, N, 2, ns), dtype=torch.int32, device="cuda")
    bsum = torch.empty((2, 2, ns), dtype=torch.int32, device="cuda")
    moe.moe_debug_subblock_dots(fmt, dev(w), N, K, dev(xq), isum, bsum)
    sl = 256 // ns
    want = np.array([-127, 127])[:, None, None, None] * sl * fieldpack.QMAX[fmt]
    np.testing.assert_array_equal(isum.cpu().numpy(), np.broadcast_to(want, isum.shape))


def test_subblock_dots_iq2g_extreme_groups(moe):
    """IQ2-style grid format: the group of largest magnitude sum (the last grid entry, every sign
    positive) and the all-ones group with seven minus signs (the 8th sign then makes it eight),
    against q_a = -127 and +127: the integer sums equal the hand-computable 4 * (sum of the group)
    * q_a per 32-weight sub-block, bit for bit."""
    fmt, N, K = FMT_IQ2G, 256, 512
    grid = oracle.iq2g_grid()
    top = grid[255].astype(np.int64)
    neg_ones = -np.ones(8, np.int64)
    q = np.empty((N, 2, 256), np.int64)
    q[:, 0] = np.tile(top, 32)
    q[:, 1] = np.tile(neg_ones, 32)
    sc = np.full((N, 2, 8), 31)
    w = fieldpack.pack_fields(fmt, N, K, q, sc, np.zeros((N, 2, 8)), np.ones((N, 2), np.float16),
                              np.zeros((N, 2), np.float16))
    xq = np.stack([np.full(K, -127, np.int8), np.full(K, 127, np.int8)])
    isum = torch.empty((2, N, 2, 8), dtype=torch.int32, device="cuda")
    bsum = torch.empty((2, 2, 8), dtype=torch.int32, device="cuda")
    moe.moe_debug_subblock_dots(fmt, dev(w), N, K, dev(xq), isum, bsum)
    got = isum.cpu().numpy()
    for t, qa in enumerate((-127, 127)):
        assert (got[t, :, 0] == 4 * int(top.sum()) * qa).all()
        assert (got[t, :, 1] == 4 * -8 * qa).all()


def test_subblock_dots_extreme_codes(moe):
    """q_w = 15 with scale 63 against q_a = -127 everywhere: the largest sums."""
    fmt, N, K = FMT_Q4K, 256, 512
    q = np.full((N, 2, 256), 15)
    sc = np.full((N, 2, 8), 63)
    w = fieldpack.pack_fields(fmt, N, K, q, sc, sc, np.ones((N, 2), np.float16), np.ones((N, 2), np.float16))
    xq = np.full((2, K), -127, np.int8)
    isum = torch.empty((2, N, 2, 8), dtype=torch.int32, device="cuda")
    bsum = torch.empty((2, 2, 8), dtype=torch.int32, device="cuda")
    moe.moe_debug_subblock_dots(fmt, dev(w), N, K, dev(xq), isum, bsum)
    assert (isum.cpu().numpy() == 32 * 15 * -127).all()
    assert (bsum.cpu().numpy() == 32 * -127).all()


# ------------------------------------------------------------------ routing

@pytest.mark.parametrize("route", [0, 1])
@pytest.mark.parametrize("T,H,E,k,bias", [(1, 2048, 256, 8, False), (4, 4096, 512, 10, False),
                                          (16, 6144, 192, 8, True), (37, 512, 16, 2, False), (5, 256, 4, 4, False),
                                          # tiled router GEMM: ragged token and expert tiles
                                          (200, 1024, 300, 6, True), (640, 4096, 512, 10, False)])
def test_route_topk(moe, route, T, H, E, k, bias):
    x = synth.activations(T, H, 11)
    wr = synth.router_weight(E, H, 11)
    b = synth.router_bias(E, 2.0, 11) if bias else None
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    gap = torch.empty((T,), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(dev(x), dev(wr), None if b is None else dev(b), k, route, logits, ids, gates, gap)
    rl, rids, rg, rgap = oracle.route(x, wr, b, k, route)
    # logits within the fp32 forward-error bound of a length-H dot product (any order), and within
    # 1e-4 of the largest logit
    l = logits.cpu().numpy().astype(np.float64)
    lbound = (H + 8) * parity.U32 * (np.abs(x.astype(np.float64)) @ np.abs(wr.astype(np.float64)).T)
    if b is not None:
        lbound += parity.U32 * np.abs(b.astype(np.float64))[None, :]
    lerr = np.abs(l - rl)
    assert (lerr <= lbound).all(), f"logit error {lerr.max():.3e} above its bound"
    np.testing.assert_allclose(l, rl, rtol=0, atol=1e-4 * np.abs(rl).max())
    gids = ids.cpu().numpy()
    routing_ok(gids, rids, rgap, rl, tie=np.maximum(parity.NEAR_TIE, 2 * lerr.max(axis=1)))
    # gates against the oracle's gates for the GPU's ids: the first-order change of a renormalised gate
    # under the device's own logit errors, plus the rounding of its exp and division (the parity rule)
    _, _, rg2, _ = oracle.route(x, wr, b, k, route, forced_ids=gids)
    dl = np.take_along_axis(lerr, gids, axis=1).max(axis=1, keepdims=True)
    gtol = np.abs(rg2) * (2 * dl + 16 * parity.U32) + parity.GATE_ATOL
    gd = gates.cpu().numpy().astype(np.float64)
    assert (np.abs(gd - rg2) <= gtol).all(), f"gate error {np.abs(gd - rg2).max():.3e}"
    g = gap.cpu().numpy()
    fin = np.isfinite(rgap)
    np.testing.assert_allclose(g[fin], rgap[fin], rtol=0, atol=1e-4)
    assert (np.isinf(g) == ~fin).all()


def test_route_ties_pick_lower_index(moe):
    T, H, E, k = 2, 256, 64, 4
    x = np.ones((T, H), np.float32)
    wr = np.zeros((E, H), np.float32)
    wr[[5, 9, 30, 31, 40], :] = 1.0 / H               # five equal logits of 1.0
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route_topk(dev(x), dev(wr), None, k, 0, logits, ids, gates)
    np.testing.assert_array_equal(ids.cpu().numpy(), [[5, 9, 30, 31]] * T)
    np.testing.assert_allclose(gates.cpu().numpy(), 0.25, rtol=1e-6)


# ------------------------------------------------------------------ bucketing

@pytest.mark.parametrize("T,k,E,S", [(1, 8, 256, 1), (4, 10, 512, 1), (16, 8, 192, 0), (3, 2, 3, 1),
                                     (300, 10, 512, 1), (1000, 8, 64, 0), (8192, 10, 512, 1)])
def test_bucket_bit_exact(moe, T, k, E, S):
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts = torch.empty(E + S, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + S + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * (k + S), dtype=torch.int32, device="cuda")
    inv = torch.empty(T * (k + S), dtype=torch.int32, device="cuda")
    ws = torch.zeros(moe.moe_bucket_workspace_size(T, k, E, S), dtype=torch.uint8, device="cuda")
    moe.moe_bucket(dev(ids), E, S, counts, offsets, perm, inv, ws)
    rc, ro, rp = oracle.bucket(ids, E, S)
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(perm.cpu().numpy(), rp)
    p = perm.cpu().numpy()
    np.testing.assert_array_equal(inv.cpu().numpy()[p], np.arange(p.size))
    assert moe.moe_get_status(ws) == 0


def test_bucket_flags_out_of_range_ids(moe):
    ids = np.array([[0, 1], [2, 7]], np.int32)        # 7 >= E
    E = 4
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.zeros(4, dtype=torch.int32, device="cuda")
    ws = torch.zeros(moe.moe_bucket_workspace_size(2, 2, E, 0), dtype=torch.uint8, device="cuda")
    moe.moe_bucket(dev(ids), E, 0, counts, offsets, perm, None, ws)
    assert moe.moe_get_status(ws) == moe.MOE_ERR_DEVICE_BOUNDS
    assert moe.moe_get_status(ws) == 0                # read-and-clear
    np.testing.assert_array_equal(counts.cpu().numpy(), [1, 1, 1, 0])


# ------------------------------------------------------------------ expert FFN + combine

def _experts_host(fmt, E, H, I, seed, layer=0):
    return [(synth.gen_matrix(fmt, I, H, seed, layer, e, 0), synth.gen_matrix(fmt, I, H, seed, layer, e, 1),
             synth.gen_matrix(fmt, H, I, seed, layer, e, 2)) for e in range(E)]


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("T,H,I,E,k,S", [(4, 512, 256, 16, 2, 0), (5, 768, 512, 8, 3, 1), (17, 256, 256, 4, 2, 1)])
def test_expert_ffn_and_combine(moe, fmt, T, H, I, E, k, S):
    ex = _experts_host(fmt, E + S, H, I, seed=21)
    table = moe.expert_table([tuple(dev(m) for m in e) for e in ex])
    rng = np.random.default_rng(T * H)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    gates = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    x = synth.activations(T, H, 21)
    xq, xd, xbs = oracle.q8k_quantize(x)
    rc, ro, rp = oracle.bucket(ids, E, S)
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=0, fmt=fmt, T_max=T)
    y = torch.full((T * (k + S), H), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(moe.moe_expert_ffn_workspace_size(desc, T), dtype=torch.uint8, device="cuda")
    moe.moe_expert_ffn(desc, table, dev(xq), dev(xd), dev(xbs), dev(rc), dev(ro), dev(rp), T, y, ws)
    yg = y.cpu().numpy()
    for t in range(T):
        slots = [(t * k + s, ids[t, s]) for s in range(k)] + [(T * k + sh * T + t, E + sh) for sh in range(S)]
        for p, e in slots:
            ref = oracle.expert_ffn(*ex[e], fmt, H, I, xq[t:t + 1], xd[t:t + 1])
            assert_close_rows(yg[p:p + 1], ref, f"y slot {p} (expert {e})")
    res = synth.normal_f32((T, H), 1.0, 21, synth.TAG_RESIDUAL)
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    moe.moe_combine(y, dev(gates), T, H, k, S, dev(res), out)
    want = res.astype(np.float64).copy()
    for t in range(T):
        for s in range(k):
            want[t] += gates[t, s] * yg[t * k + s]
        for sh in range(S):
            want[t] += yg[T * k + sh * T + t]
    np.testing.assert_allclose(out.cpu().numpy(), want, rtol=1e-5, atol=1e-5 * np.abs(want).max())


# ------------------------------------------------------------------ whole layer

CASES = [
    # fmt, route, H, I, E, k, S, T, bias
    (FMT_Q4K, 0, 512, 256, 16, 2, 0, 4, False),      # the tiny workload
    (FMT_Q4K, 0, 2048, 512, 64, 8, 1, 1, False),     # decode, shared expert
    (FMT_Q2K, 1, 1024, 512, 64, 10, 1, 4, False),    # Q2_K, sigmoid, verify window
    (FMT_Q4K, 0, 768, 512, 32, 8, 0, 16, True),      # skewed router, 16 tokens
    (FMT_Q2K, 0, 256, 256, 8, 8, 1, 3, False),       # k = E
    (FMT_Q4K, 1, 256, 768, 1, 1, 0, 7, False),       # one expert
    (FMT_Q4K, 1, 512, 256, 40, 10, 1, 40, False),    # more than the single-CTA bucket (400 pairs)
    # prefill chunks (tensor-core grouped GEMM): several token tiles per expert, ragged tails
    (FMT_Q4K, 0, 512, 256, 8, 2, 1, 512, False),
    (FMT_Q2K, 1, 768, 512, 16, 4, 0, 300, True),     # skewed router: some experts over several token tiles
    (FMT_Q4K, 1, 1024, 256, 4, 1, 2, 257, False),    # two shared experts, one routed slot per token
    # the Q5_K/Q3_K/Q6_K-style formats: decode (single launch), the GEMV path, a prefill chunk
    (FMT_Q5K, 0, 2048, 512, 64, 8, 1, 1, False),
    (FMT_Q3K, 1, 1024, 512, 64, 10, 1, 4, False),
    (FMT_Q6K, 0, 768, 512, 32, 8, 0, 16, True),
    (FMT_Q6K, 1, 512, 256, 40, 10, 1, 40, False),    # 400 pairs: the GEMV path
    (FMT_Q5K, 1, 512, 256, 40, 10, 1, 40, False),
    (FMT_Q3K, 0, 512, 256, 8, 2, 1, 512, False),     # tensor-core prefill
    (FMT_Q5K, 0, 512, 256, 8, 2, 1, 512, False),     # a prefill-size chunk on the GEMV path
    (FMT_Q6K, 1, 768, 512, 16, 4, 0, 300, True),
    # the IQ2-style grid format: decode (single launch), the GEMV path, a prefill-size chunk
    (FMT_IQ2G, 0, 2048, 512, 64, 8, 1, 1, False),
    (FMT_IQ2G, 1, 1024, 512, 64, 10, 1, 4, False),
    (FMT_IQ2G, 1, 512, 256, 40, 10, 1, 40, False),
    (FMT_IQ2G, 0, 512, 256, 8, 2, 1, 512, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "fmt%d_r%d_H%d_I%d_E%d_k%d_S%d_T%d" % c[:8])
def test_layer_forward(moe, case):
    fmt, route, H, I, E, k, S, T, use_bias = case
    seed = H + E + T
    ex = _experts_host(fmt, E + S, H, I, seed)
    table = moe.expert_table([tuple(dev(m) for m in e) for e in ex])
    wr = synth.router_weight(E, H, seed)
    bias = synth.router_bias(E, 2.0, seed) if use_bias else None
    x = synth.activations(T, H, seed)
    res = synth.normal_f32((T, H), 1.0, seed, synth.TAG_RESIDUAL)
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=route, fmt=fmt, T_max=T)
    layer = moe.MoeLayer(desc, table, dev(wr), None if bias is None else dev(bias))
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    out = layer.forward(dev(x), residual=dev(res), ids_out=ids, gates_out=gates)
    assert moe.moe_get_status(layer.ws) == 0
    gids = ids.cpu().numpy()
    rl, rids, _, rgap = oracle.route(x, wr, bias, k, route)
    routing_ok(gids, rids, rgap, rl)
    ref, _, rgates, _ = oracle.layer_forward(fmt, H, I, E, k, S, route, ex, wr, bias, x, residual=res,
                                             forced_ids=gids)
    np.testing.assert_allclose(gates.cpu().numpy(), rgates, rtol=1e-5, atol=1e-6)
    assert_close_rows(out.cpu().numpy(), ref)
    # the intermediate h re-quantization, decided in fp32 on both sides
    P = T * (k + S)
    h = layer.ws_view("h", torch.float32, (P, I)).cpu().numpy()
    hq = layer.ws_view("hq", torch.int8, (P, I)).cpu().numpy()
    hd = layer.ws_view("hd", torch.float32, (P, I // 256)).cpu().numpy()
    rq, rd, _ = oracle.q8k_quantize(h)
    np.testing.assert_array_equal(hq, rq)
    np.testing.assert_array_equal(hd, rd)
    # per-slot y and the output within the fp32 forward-error bound, h-code flips counted
    devd = dict(xq=layer.ws_view("xq", torch.int8, (T, H)).cpu().numpy(), ids=gids, gates=gates.cpu().numpy(),
                logits=layer.ws_view("logits", torch.float32, (T, E)).cpu().numpy(),
                perm=layer.ws_view("perm", torch.int32, (P,)).cpu().numpy(), h=h,
                y=layer.ws_view("y", torch.float32, (P, H)).cpu().numpy(), out=out.cpu().numpy())
    tokens = np.arange(T) if T <= 64 else np.unique(np.linspace(0, T - 1, 64).round().astype(np.int64))
    _, fails = parity.check_layer(fmt, H, I, E, k, S, route, ex, wr, bias, x, res, devd, tokens)
    assert not fails, "; ".join(fails[:5])


def test_layer_forward_is_deterministic(moe):
    fmt, route, H, I, E, k, S, T = FMT_Q4K, 0, 1024, 512, 32, 4, 1, 9
    ex = _experts_host(fmt, E + S, H, I, 3)
    table = moe.expert_table([tuple(dev(m) for m in e) for e in ex])
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=route, fmt=fmt, T_max=T)
    layer = moe.MoeLayer(desc, table, dev(synth.router_weight(E, H, 3)))
    x = dev(synth.activations(T, H, 3))
    a = layer.forward(x).cpu().numpy()
    b = layer.forward(x).cpu().numpy()
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("T", [1, 40, 300])
def test_trace_events_bracket_launches(moe, T):
    """The launch-trace hook records its events eagerly (plain records) and
    under stream capture (event-record nodes): two per single-launch decode
    layer (T = 1), four per expert-FFN sequence (T = 40: GEMV kernels,
    T = 300: tensor prefill); each bracket spans a launch that really ran
    (positive duration, inside the caller's own bracket around the call)."""
    fmt, route, H, I, E, k, S = FMT_Q4K, 0, 1024, 512, 32, 4, 1
    ex = _experts_host(fmt, E + S, H, I, 5)
    table = moe.expert_table([tuple(dev(m) for m in e) for e in ex])
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=route, fmt=fmt, T_max=T)
    layer = moe.MoeLayer(desc, table, dev(synth.router_weight(E, H, 5)))
    x = dev(synth.activations(T, H, 5))
    out = torch.empty_like(x)
    want = 2 if moe.moe_layer_path(desc, T) == 0 else 4
    events = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    outer = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    stream = torch.cuda.current_stream()

    def spans_within(used):
        torch.cuda.synchronize()
        total = outer[0].elapsed_time(outer[1])
        spans = [events[i].elapsed_time(events[i + 1]) for i in range(0, used, 2)]
        assert all(0 < sp <= total for sp in spans), (spans, total)

    # eager: the hook records on the launching stream
    moe.moe_trace_events(events)
    outer[0].record(stream)
    layer.forward(x, out=out)
    outer[1].record(stream)
    used = moe.moe_trace_used()
    moe.moe_trace_events(None)
    assert used == want, used
    spans_within(used)
    # captured: the records become nodes of the graph, replayed with it
    g = torch.cuda.CUDAGraph()
    moe.moe_trace_events(events)
    with torch.cuda.graph(g):
        layer.forward(x, out=out)
    used = moe.moe_trace_used()
    moe.moe_trace_events(None)
    assert used == want, used
    outer[0].record(stream)
    g.replay()
    outer[1].record(stream)
    spans_within(used)
    assert moe.moe_get_status(layer.ws) == 0


@pytest.mark.parametrize("T", [6, 512])
def test_layer_forward_null_expert_is_not_mine(moe, T):
    fmt, H, I, E, k, S = FMT_Q4K, 512, 256, 8, 2, 1
    ex = _experts_host(fmt, E + S, H, I, 8)
    wr = synth.router_weight(E, H, 8)
    x = synth.activations(T, H, 8)
    _, rids, _, _ = oracle.route(x, wr, None, k, 0)
    dead = int(rids[0, 0])
    dev_ex = [None if e == dead else tuple(dev(m) for m in ex[e]) for e in range(E + S)]
    host_ex = [None if e == dead else ex[e] for e in range(E + S)]
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=0, fmt=fmt, T_max=T)
    layer = moe.MoeLayer(desc, moe.expert_table(dev_ex), dev(wr))
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    out = layer.forward(dev(x), ids_out=ids).cpu().numpy()
    ref, _, _, _ = oracle.layer_forward(fmt, H, I, E, k, S, 0, host_ex, wr, None, x, forced_ids=ids.cpu().numpy())
    assert_close_rows(out, ref)


def test_layer_forward_in_place_residual(moe):
    fmt, H, I, E, k, S, T = FMT_Q2K, 512, 256, 8, 2, 0, 2
    ex = _experts_host(fmt, E, H, I, 4)
    wr = synth.router_weight(E, H, 4)
    x = synth.activations(T, H, 4)
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=0, fmt=fmt, T_max=T)
    layer = moe.MoeLayer(desc, moe.expert_table([tuple(dev(m) for m in e) for e in ex]), dev(wr))
    xd = dev(x)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    layer.forward(xd, residual=xd, out=xd, ids_out=ids)
    ref, _, _, _ = oracle.layer_forward(fmt, H, I, E, k, S, 0, ex, wr, None, x, residual=x,
                                        forced_ids=ids.cpu().numpy())
    assert_close_rows(xd.cpu().numpy(), ref)


@pytest.mark.parametrize("fmt,route,S,T", [(FMT_Q4K, 0, 1, 2), (FMT_Q2K, 1, 0, 5)])
def test_stack_forward_chained_layers(moe, fmt, route, S, T):
    """A stack whose layer l+1 reads layer l's output (a decode step through
    the layers), in one launch; each layer matches the oracle run on the
    GPU's own input for that layer."""
    H, I, E, k, L = 512, 256, 16, 4, 3
    ex = [_experts_host(fmt, E + S, H, I, seed=40 + l, layer=l) for l in range(L)]
    tables = [moe.expert_table([tuple(dev(m) for m in e) for e in ex[l]]) for l in range(L)]
    wrs = [synth.router_weight(E, H, 40, l) for l in range(L)]
    x0 = synth.activations(T, H, 40)
    xs = [dev(x0)] + [torch.empty((T, H), dtype=torch.float32, device="cuda") for _ in range(L - 1)]
    outs = xs[1:] + [torch.empty((T, H), dtype=torch.float32, device="cuda")]
    ids = [torch.empty((T, k), dtype=torch.int32, device="cuda") for _ in range(L)]
    rows = [dict(table=tables[l], w_router=dev(wrs[l]), x=xs[l], residual=xs[l], out=outs[l], ids_out=ids[l])
            for l in range(L)]
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=route, fmt=fmt, T_max=T)
    ws = torch.zeros(moe.moe_stack_workspace_size(desc, L), dtype=torch.uint8, device="cuda")
    moe.moe_stack_forward(desc, moe.stack_pointer_table(rows), T, ws)
    assert moe.moe_get_status(ws) == 0
    marker = moe.MoeLayer.ws_view_of(ws, moe.moe_workspace_layout(desc), "phase_ns", torch.int64, (16,))
    assert int(marker[15]) == 4          # chained layers run one after the other (dataflow stack)
    for l in range(L):
        xin = xs[l].cpu().numpy()
        gids = ids[l].cpu().numpy()
        rl, rids, _, rgap = oracle.route(xin, wrs[l], None, k, route)
        routing_ok(gids, rids, rgap, rl)
        ref, _, _, _ = oracle.layer_forward(fmt, H, I, E, k, S, route, ex[l], wrs[l], None, xin, residual=xin,
                                            forced_ids=gids)
        assert_close_rows(outs[l].cpu().numpy(), ref, f"layer {l}")


@pytest.mark.parametrize("chained", [False, True])
@pytest.mark.parametrize("H", [2048, 4096])
def test_stack_forward_sixteen_tokens(moe, chained, H):
    """The largest decode batch (16 tokens) through the dataflow stack (top-1,
    so that the items per SM stay within the dataflow kernel's range),
    chained and independent; at H=4096 the 16 staged token rows leave no
    room for the warps' weight rings, so that shape runs the register-load
    items.  Every layer matches the oracle."""
    fmt, route, S, I, E, k, T, L = FMT_Q4K, 0, 0, 256, 16, 1, 16, 2
    ex = [_experts_host(fmt, E + S, H, I, seed=90 + l, layer=l) for l in range(L)]
    tables = [moe.expert_table([tuple(dev(m) for m in e) for e in ex[l]]) for l in range(L)]
    wrs = [synth.router_weight(E, H, 90, l) for l in range(L)]
    xs_h = [synth.activations(T, H, 90, layer=l) for l in range(L)]
    xs = [dev(xs_h[0])] + ([torch.empty((T, H), dtype=torch.float32, device="cuda")] if chained
                           else [dev(xs_h[1])])
    outs = ([xs[1]] if chained else [torch.empty((T, H), dtype=torch.float32, device="cuda")]) + \
        [torch.empty((T, H), dtype=torch.float32, device="cuda")]
    ids = [torch.empty((T, k), dtype=torch.int32, device="cuda") for _ in range(L)]
    rows = [dict(table=tables[l], w_router=dev(wrs[l]), x=xs[l], residual=xs[l], out=outs[l], ids_out=ids[l])
            for l in range(L)]
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=route, fmt=fmt, T_max=T)
    ws = torch.zeros(moe.moe_stack_workspace_size(desc, L), dtype=torch.uint8, device="cuda")
    moe.moe_stack_forward(desc, moe.stack_pointer_table(rows), T, ws)
    assert moe.moe_get_status(ws) == 0
    marker = moe.MoeLayer.ws_view_of(ws, moe.moe_workspace_layout(desc), "phase_ns", torch.int64, (16,))
    assert int(marker[15]) == (4 if chained else 3)
    for l in range(L):
        xin = xs[l].cpu().numpy()
        gids = ids[l].cpu().numpy()
        rl, rids, _, rgap = oracle.route(xin, wrs[l], None, k, route)
        routing_ok(gids, rids, rgap, rl)
        ref, _, _, _ = oracle.layer_forward(fmt, H, I, E, k, S, route, ex[l], wrs[l], None, xin, residual=xin,
                                            forced_ids=gids)
        assert_close_rows(outs[l].cpu().numpy(), ref, f"layer {l}")


@pytest.mark.parametrize("fmt,route,S,T,L", [(FMT_Q4K, 0, 1, 1, 6), (FMT_Q2K, 1, 1, 4, 5), (FMT_Q4K, 0, 0, 3, 2)])
def test_stack_forward_independent_layers_pipelined(moe, fmt, route, S, T, L):
    """Layers with their own inputs: the kernel pipelines neighbouring layers;
    every layer must still match the oracle (and the schedule must be the
    pipelined one)."""
    H, I, E, k = 512, 512, 32, 6
    ex = [_experts_host(fmt, E + S, H, I, seed=70 + l, layer=l) for l in range(L)]
    tables = [moe.expert_table([tuple(dev(m) for m in e) for e in ex[l]]) for l in range(L)]
    wrs = [synth.router_weight(E, H, 70, l) for l in range(L)]
    xs_h = [synth.activations(T, H, 70, layer=l) for l in range(L)]
    xs = [dev(x) for x in xs_h]
    outs = [torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda") for _ in range(L)]
    ids = [torch.empty((T, k), dtype=torch.int32, device="cuda") for _ in range(L)]
    rows = [dict(table=tables[l], w_router=dev(wrs[l]), x=xs[l], residual=xs[l], out=outs[l], ids_out=ids[l])
            for l in range(L)]
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=route, fmt=fmt, T_max=T)
    ws = torch.zeros(moe.moe_stack_workspace_size(desc, L), dtype=torch.uint8, device="cuda")
    for rep in range(2):
        moe.moe_stack_forward(desc, moe.stack_pointer_table(rows), T, ws)
        assert moe.moe_get_status(ws) == 0
        marker = moe.MoeLayer.ws_view_of(ws, moe.moe_workspace_layout(desc), "phase_ns", torch.int64, (16,))
        assert int(marker[15]) == 3      # dataflow stack, layers overlapped
        for l in range(L):
            gids = ids[l].cpu().numpy()
            rl, rids, _, rgap = oracle.route(xs_h[l], wrs[l], None, k, route)
            routing_ok(gids, rids, rgap, rl)
            ref, _, _, _ = oracle.layer_forward(fmt, H, I, E, k, S, route, ex[l], wrs[l], None, xs_h[l],
                                                residual=xs_h[l], forced_ids=gids)
            assert_close_rows(outs[l].cpu().numpy(), ref, f"layer {l}")


@pytest.mark.parametrize("chained,L", [(False, 3), (True, 2), (False, 5)])
def test_stack_forward_heavy_layers(moe, chained, L):
    """Layers with many expert items per SM (8 tokens, 1024-wide experts):
    short stacks run on the barrier-pipelined kernel, stacks of 4 or more
    layers on the dataflow kernel; every layer must match the oracle."""
    # chained: each layer scales the activations up by orders of magnitude at this
    # shape, so two layers (a third would overflow fp32 in the oracle as well)
    fmt, route, H, I, E, k, S, T = FMT_Q4K, 0, 2048, 1024, 64, 8, 1, 8
    ex = [_experts_host(fmt, E + S, H, I, seed=90 + l, layer=l) for l in range(L)]
    tables = [moe.expert_table([tuple(dev(m) for m in e) for e in ex[l]]) for l in range(L)]
    wrs = [synth.router_weight(E, H, 90, l) for l in range(L)]
    xs_h = [synth.activations(T, H, 90, layer=l) for l in range(L)]
    outs = [torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda") for _ in range(L)]
    xs = [dev(xs_h[0])] + (outs[:-1] if chained else [dev(x) for x in xs_h[1:]])
    ids = [torch.empty((T, k), dtype=torch.int32, device="cuda") for _ in range(L)]
    rows = [dict(table=tables[l], w_router=dev(wrs[l]), x=xs[l], residual=xs[l], out=outs[l], ids_out=ids[l])
            for l in range(L)]
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=route, fmt=fmt, T_max=T)
    ws = torch.zeros(moe.moe_stack_workspace_size(desc, L), dtype=torch.uint8, device="cuda")
    moe.moe_stack_forward(desc, moe.stack_pointer_table(rows), T, ws)
    assert moe.moe_get_status(ws) == 0
    marker = moe.MoeLayer.ws_view_of(ws, moe.moe_workspace_layout(desc), "phase_ns", torch.int64, (16,))
    assert int(marker[15]) == (3 if L >= 4 else 1 if chained else 2)
    for l in range(L):
        xin = xs[l].cpu().numpy()
        gids = ids[l].cpu().numpy()
        rl, rids, _, rgap = oracle.route(xin, wrs[l], None, k, route)
        routing_ok(gids, rids, rgap, rl)
        ref, _, _, _ = oracle.layer_forward(fmt, H, I, E, k, S, route, ex[l], wrs[l], None, xin, residual=xin,
                                            forced_ids=gids)
        assert_close_rows(outs[l].cpu().numpy(), ref, f"layer {l}")


def test_stack_forward_rejects_prefill_shapes(moe):
    desc = dict(H=512, I=256, E=16, top_k=8, n_shared=0, route=0, fmt=FMT_Q4K, T_max=64)
    ws = torch.zeros(moe.moe_layer_workspace_size(desc), dtype=torch.uint8, device="cuda")
    rows = moe.stack_pointer_table([dict()], device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_stack_forward(desc, rows, 64, ws)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED


def test_bounded_wait_runs_out_and_reports(moe):
    """A device wait on a flag nothing sets ends by itself, records a timeout
    in the status word, and the context stays usable for the next layer."""
    desc = dict(H=512, I=256, E=8, top_k=2, n_shared=0, route=0, fmt=FMT_Q4K, T_max=2)
    ex = _experts_host(FMT_Q4K, 8, 512, 256, 5)
    wr = synth.router_weight(8, 512, 5)
    layer = moe.MoeLayer(desc, moe.expert_table([tuple(dev(m) for m in e) for e in ex]), dev(wr))
    moe.moe_debug_wait_timeout(layer.ws, 2000)
    assert moe.moe_get_status(layer.ws) == moe.MOE_ERR_DEVICE_TIMEOUT
    assert moe.moe_get_status(layer.ws) == 0            # read and cleared
    x = synth.activations(2, 512, 5)
    out = layer.forward(dev(x)).cpu().numpy()
    ref, _, _, _ = oracle.layer_forward(FMT_Q4K, 512, 256, 8, 2, 0, 0, ex, wr, None, x)
    assert_close_rows(out, ref)


# ------------------------------------------------------- tensor-core integer sums

@pytest.mark.parametrize("fmt,N,K,T", [(FMT_Q4K, 256, 512, 200), (FMT_Q2K, 256, 768, 130), (FMT_Q4K, 512, 256, 16),
                                       (FMT_Q2K, 256, 256, 1), (FMT_Q3K, 256, 512, 200), (FMT_Q3K, 512, 256, 3),
                                       (FMT_IQ2G, 256, 512, 200), (FMT_IQ2G, 512, 256, 3)])
def test_prefill_integer_sums_bit_exact(moe, fmt, N, K, T):
    """S = sum_j sc_j isum_j and M = sum_j mn_j bsum_j of every (token, row, super-block), as the tcgen05
    GEMM forms them in TMEM, equal the oracle's int64 sums bit for bit.  Rows 0-31 carry an all-extreme
    first super-block (largest codes, scales and mins); tokens 0-2 carry activation codes +127, -127 and
    127 with one 126 there, so that Q4_K sums reach 63*15*127*256 > 2^24, one of them odd.  T = 200 and
    130 span several token tiles with a ragged last one."""
    assert 130 > moe.moe_prefill_tile_tokens() >= 32
    rng = np.random.default_rng(N + K + T + fmt)
    q, sc, mn, d, dmin = fieldpack.random_fields(fmt, N, K, rng)
    if fmt == FMT_IQ2G:  # the grid entry of largest magnitude sum, all signs +, the largest scale
        grid = oracle.iq2g_grid()
        q[:32, 0] = np.tile(grid[np.argmax(grid.sum(axis=1))], 32)
    else:
        q[:32, 0] = fieldpack.QMAX[fmt]
    sc[:32, 0] = fieldpack.SCALE_RANGE[fmt][0] if fmt == FMT_Q3K else fieldpack.SCALE_RANGE[fmt][1]
    mn[:32, 0] = fieldpack.MIN_RANGE[fmt][1]
    w = fieldpack.pack_fields(fmt, N, K, q, sc, mn, d, dmin)
    x = rng.standard_normal((T, K)).astype(np.float32)
    if T >= 3:
        x[0, :256] = 127.0
        x[1, :256] = -127.0
        x[2, :256] = 127.0
        x[2, 5] = 126.0
    xq, xd, bs = oracle.q8k_quantize(x)
    S = torch.empty((T, N, K // 256), dtype=torch.int32, device="cuda")
    M = torch.empty_like(S)
    ws = torch.zeros(moe.moe_debug_prefill_sums_workspace_size(N, K, T), dtype=torch.uint8, device="cuda")
    moe.moe_debug_prefill_sums(fmt, dev(w), N, K, dev(xq), dev(xd), dev(bs), S, M, ws)
    torch.cuda.synchronize()
    Sr, Mr = oracle.superblock_sums(w, fmt, N, K, xq)
    np.testing.assert_array_equal(S.cpu().numpy(), Sr)
    np.testing.assert_array_equal(M.cpu().numpy(), Mr)
    if fmt == FMT_Q4K and T >= 3:
        assert Sr[0, 0, 0] == 63 * 15 * 127 * 256 and Sr[2, 0, 0] % 2 == 1 and Sr[2, 0, 0] > 2 ** 24


def test_workspace_shared_by_launches_of_different_grid_sizes(moe):
    """One workspace used in turn by the single-layer decode kernel (one CTA per SM, three grid barriers)
    and the stack kernel (two CTAs per SM): every result equals, bit for bit, the same call on a fresh
    workspace, and the device status stays clear (a grid barrier keeps no count across launches)."""
    fmt, H, I, E, k, S, T, L = FMT_Q4K, 1024, 512, 64, 8, 1, 1, 2
    ex = _experts_host(fmt, E + S, H, I, 17)
    table = moe.expert_table([tuple(dev(m) for m in e) for e in ex])
    wr = dev(synth.router_weight(E, H, 17))
    desc = dict(H=H, I=I, E=E, top_k=k, n_shared=S, route=0, fmt=fmt, T_max=T)
    xs = [dev(synth.activations(T, H, 17, l)) for l in range(L)]
    outs = [torch.empty_like(xs[0]) for _ in range(L)]
    rows = [dict(table=table, w_router=wr, x=xs[l], residual=xs[l], out=outs[l]) for l in range(L)]
    stack = moe.stack_pointer_table(rows)
    size = moe.moe_stack_workspace_size(desc, L)
    layout = moe.moe_workspace_layout(desc)

    def run_layer(ws):
        out = torch.empty_like(xs[0])
        moe.moe_layer_forward(desc, table, wr, None, xs[0], xs[0], out, None, None, ws)
        return out.cpu().numpy()

    def run_stack(ws):
        moe.moe_stack_forward(desc, stack, T, ws)
        return np.stack([o.cpu().numpy() for o in outs])

    def grid(ws):
        return int(moe.MoeLayer.ws_view_of(ws, layout, "phase_ns", torch.int64, (16,))[14].item())

    want_layer = run_layer(torch.zeros(size, dtype=torch.uint8, device="cuda"))
    want_stack = run_stack(torch.zeros(size, dtype=torch.uint8, device="cuda"))
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    grids = set()
    for _ in range(3):
        np.testing.assert_array_equal(run_layer(ws).view(np.uint32), want_layer.view(np.uint32))
        grids.add(grid(ws))
        np.testing.assert_array_equal(run_stack(ws).view(np.uint32), want_stack.view(np.uint32))
        grids.add(grid(ws))
        assert moe.moe_get_status(ws) == 0
    assert len(grids) == 2, grids          # the two kernels ran with different grid sizes
