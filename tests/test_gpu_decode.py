"""GPU parity of the fused decode kernels that moe_layer_w4 takes for T <= 4
("Perplexity Open Sources Lily: A Rust + Metal Inference Engine for
Qwen3.6-35B-A3B on Apple Silicon", section "Decode: Minimize Bytes Moved Per
Token"): routing bit-identical with the prefill router and the oracle, the
layer output and the next-layer input within the layer's tolerance of the
oracle, deterministic across calls and stacked layers."""
import numpy as np
import pytest
import torch

import bit_moe_expert_histogram_gb300 as m
import oracle
import synth
from moe_case import Case, close, d16, f64, h16

pytestmark = pytest.mark.gpu

FULL = synth.CONFIGS["decode"].shape
TINY = synth.CONFIGS["tiny"].shape
NOSH = synth.LayerShape(H=256, E=16, K=2, I=128, n_shared=0)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    m.load()


_cache = {}


def layer(shape, seed):
    key = (shape, seed)
    if key not in _cache:
        _cache.clear()
        _cache[key] = synth.gen_layer(4, shape, seed=seed)
    return _cache[key]


def check_layer(c, L, x_bits):
    """ids/w against the oracle router, y and x_next against the oracle."""
    K = c.S.K
    ids_o, _, w64 = oracle.topk(oracle.router_logits(x_bits, L.w_router, L.router_bias), K)
    assert np.array_equal(c.ids.cpu().numpy(), ids_o)
    assert np.abs(c.w.cpu().numpy() - w64).max() <= 1e-6
    y_o = oracle.layer_tokens(L, ids_o, w64, x=x_bits)
    y = h16(c.y)
    close(f64(y), f64(y_o), "y")
    close(f64(h16(c.x_next)), f64(oracle.rmsnorm_rows(y)), "x_next")
    return y


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_decode_layer_full_shape(T):
    L = layer(FULL, 3)
    x = L.x[:T]
    c = Case(L, T, FULL)
    c.x = d16(x, c.dev)
    c.run_layer(x_next=True)
    check_layer(c, L, x)


@pytest.mark.parametrize("shape", [TINY, NOSH], ids=["tiny", "no_shared"])
@pytest.mark.parametrize("T", [1, 4])
def test_decode_layer_small_shapes(shape, T):
    L = layer(shape, 5)
    x = L.x[:T]
    c = Case(L, T, shape)
    c.x = d16(x, c.dev)
    c.run_layer(x_next=True)
    check_layer(c, L, x)


@pytest.mark.parametrize("T", [1, 3])
def test_decode_routing_equals_prefill_router(T):
    """The fused router reproduces moe_route bit for bit (same logit order,
    same top-K code)."""
    L = layer(FULL, 3)
    c = Case(L, T, FULL)
    c.x = d16(L.x[:T], c.dev)
    c.run_layer()
    ids_l, w_l = c.ids.cpu().numpy().copy(), c.w.cpu().numpy().copy()
    c.ids.fill_(-1)
    c.w.zero_()
    m.moe_route(c.shape, c.x, c.wr, c.bias, c.ids, c.w, c.ws)
    assert np.array_equal(c.ids.cpu().numpy(), ids_l)
    assert np.array_equal(c.w.cpu().numpy().view(np.uint32), w_l.view(np.uint32))


def test_decode_equals_four_calls_within_tolerance():
    """Decode kernels and the grouped-GEMM path compute the same layer."""
    L = layer(FULL, 3)
    T = 2
    c = Case(L, T, FULL)
    c.x = d16(L.x[:T], c.dev)
    c.run_calls(x_next=True)
    y4 = f64(h16(c.y))
    c.y.zero_()
    c.run_layer(x_next=True)
    close(f64(h16(c.y)), y4, "decode vs grouped GEMM")


def test_decode_deterministic_and_tickets_reset():
    """Back-to-back calls give identical bits: the last-block tickets of the
    router and of the normalisation return to zero every call."""
    L = layer(FULL, 3)
    c = Case(L, 1, FULL)
    c.x = d16(L.x[:1], c.dev)
    c.run_layer(x_next=True)
    y0, xn0 = h16(c.y).copy(), h16(c.x_next).copy()
    for _ in range(20):
        m.moe_layer_w4(c.shape, c.x, c.wr, c.bias, c.ex, c.sh, c.y, c.ws, x_next=c.x_next,
                       topk_ids=c.ids, topk_w=c.w)
    assert m.moe_query_device_status(c.ws) == 0
    assert np.array_equal(h16(c.y), y0)
    assert np.array_equal(h16(c.x_next), xn0)


def test_decode_stacked_layers_teacher_forced():
    """Three stacked layers, x_next feeding the next layer on the device;
    every layer checked against the oracle on the GPU's own input."""
    Ls = [synth.gen_layer(1, TINY, seed=20 + i) for i in range(3)]
    cs = [Case(L, 1, TINY) for L in Ls]
    for i, c in enumerate(cs):
        if i:
            c.x.copy_(cs[i - 1].x_next)
        c.run_layer(x_next=True)
        check_layer(c, Ls[i], h16(c.x))


@pytest.mark.parametrize("shape,T", [(FULL, 1), (FULL, 3), (FULL, 4), (TINY, 2), (NOSH, 1)],
                         ids=["full-1", "full-3", "full-4", "tiny-2", "noshared-1"])
def test_decode_layers_equal_the_moe_layer_chain(shape, T):
    """moe_decode_layers (one persistent launch; the normalisation folded
    into the next layer) gives the bits of the moe_layer_w4 chain."""
    dev = torch.device("cuda")
    Ls = [synth.gen_layer(T, shape, seed=40 + i) for i in range(3)]
    cs = [Case(L, T, shape) for L in Ls]
    x0 = cs[0].x.clone()
    for i, c in enumerate(cs):
        if i:
            c.x.copy_(cs[i - 1].x_next)
        c.run_layer(x_next=True)
    y_chain = h16(cs[-1].y).copy()
    xn_chain = h16(cs[-1].x_next).copy()
    table = m.decode_layer_table([(c.wr, c.bias, c.ex, c.sh) for c in cs])
    ws = m.alloc_workspace(cs[0].shape, dev)
    y = torch.zeros((T, shape.H), dtype=torch.int16, device=dev)
    xn = torch.zeros((T, shape.H), dtype=torch.int16, device=dev)
    for _ in range(3):   # repeated: the epochs and counters carry over between calls
        m.moe_decode_layers(cs[0].shape, table, x0, y, ws, x_next=xn)
        assert m.moe_query_device_status(ws) == 0
        assert np.array_equal(h16(y), y_chain)
        assert np.array_equal(h16(xn), xn_chain)


def test_decode_layers_split_over_launches():
    """More layers than one persistent launch runs (48): the normalised input
    is handed from launch to launch, and the result is the chain's."""
    dev = torch.device("cuda")
    n, T = 50, 2
    Ls = [synth.gen_layer(T, NOSH, seed=100 + i) for i in range(n)]
    cs = [Case(L, T, NOSH) for L in Ls]
    x0 = cs[0].x.clone()
    for i, c in enumerate(cs):
        if i:
            c.x.copy_(cs[i - 1].x_next)
        c.run_layer(x_next=True)
    table = m.decode_layer_table([(c.wr, c.bias, c.ex, c.sh) for c in cs])
    ws = m.alloc_workspace(cs[0].shape, dev)
    y = torch.zeros((T, NOSH.H), dtype=torch.int16, device=dev)
    xn = torch.zeros((T, NOSH.H), dtype=torch.int16, device=dev)
    m.moe_decode_layers(cs[0].shape, table, x0, y, ws, x_next=xn)
    assert m.moe_query_device_status(ws) == 0
    assert np.array_equal(h16(y), h16(cs[-1].y))
    assert np.array_equal(h16(xn), h16(cs[-1].x_next))


def test_decode_layers_share_a_workspace_with_single_layers():
    """moe_layer_w4 calls between moe_decode_layers calls on one workspace
    leave the stacked result unchanged."""
    dev = torch.device("cuda")
    T = 1
    Ls = [synth.gen_layer(T, TINY, seed=60 + i) for i in range(4)]
    cs = [Case(L, T, TINY) for L in Ls]
    table = m.decode_layer_table([(c.wr, c.bias, c.ex, c.sh) for c in cs])
    ws = cs[0].ws
    y = torch.zeros((T, TINY.H), dtype=torch.int16, device=dev)
    m.moe_decode_layers(cs[0].shape, table, cs[0].x, y, ws)
    y0 = h16(y).copy()
    for _ in range(3):
        cs[0].run_layer(x_next=True)
        m.moe_decode_layers(cs[0].shape, table, cs[0].x, y, ws)
        assert m.moe_query_device_status(ws) == 0
        assert np.array_equal(h16(y), y0)


WIDE = synth.LayerShape(H=8192, E=16, K=2, I=128, n_shared=1)


def test_layer_path_on_the_device():
    """The decode shapes take the persistent kernel; T*H > 8192 the three
    per-layer kernels."""
    for T in (1, 2, 3, 4):
        assert m.moe_layer_path(m.make_shape(T, FULL.H, FULL.E, FULL.K, FULL.I, FULL.n_shared, 128)) == 2
    assert m.moe_layer_path(m.make_shape(1, TINY.H, TINY.E, TINY.K, TINY.I, TINY.n_shared, 128)) == 2
    assert m.moe_layer_path(m.make_shape(2, WIDE.H, WIDE.E, WIDE.K, WIDE.I, WIDE.n_shared, 128)) == 1


def test_per_layer_decode_kernels_wide_hidden():
    """The three-kernel decode path (taken when the persistent kernel does
    not hold the shape): one layer against the oracle, and stacked layers
    against the chain of single layers."""
    T = 2
    Ls = [synth.gen_layer(T, WIDE, seed=80 + i) for i in range(3)]
    cs = [Case(L, T, WIDE) for L in Ls]
    for i, c in enumerate(cs):
        if i:
            c.x.copy_(cs[i - 1].x_next)
        c.run_layer(x_next=True)
        check_layer(c, Ls[i], h16(c.x))
    table = m.decode_layer_table([(c.wr, c.bias, c.ex, c.sh) for c in cs])
    dev = torch.device("cuda")
    ws = m.alloc_workspace(cs[0].shape, dev)
    y = torch.zeros((T, WIDE.H), dtype=torch.int16, device=dev)
    x0 = d16(Ls[0].x[:T], dev)
    m.moe_decode_layers(cs[0].shape, table, x0, y, ws)
    assert m.moe_query_device_status(ws) == 0
    assert np.array_equal(h16(y), h16(cs[-1].y))


SWEEP = [
    (synth.LayerShape(H=512, E=100, K=4, I=256, n_shared=1), 1),
    (synth.LayerShape(H=512, E=100, K=4, I=256, n_shared=1), 3),
    (synth.LayerShape(H=1024, E=64, K=1, I=1024, n_shared=0), 2),
    (synth.LayerShape(H=256, E=32, K=16, I=128, n_shared=1), 4),
    (synth.LayerShape(H=2048, E=256, K=8, I=256, n_shared=1), 1),
]


@pytest.mark.parametrize("shape,T", SWEEP, ids=["E100-T1", "E100-T3", "K1-I1024-T2", "K16-T4", "I256-T1"])
def test_persistent_decode_shape_sweep(shape, T):
    """The persistent kernel across expert counts that are not a multiple of
    32, top-1 and top-16, every intermediate size and no shared expert:
    each layer against the oracle, the stacked call against the chain."""
    assert m.moe_layer_path(m.make_shape(T, shape.H, shape.E, shape.K, shape.I,
                                         shape.n_shared, 128)) == 2
    Ls = [synth.gen_layer(T, shape, seed=120 + i) for i in range(2)]
    cs = [Case(L, T, shape) for L in Ls]
    for i, c in enumerate(cs):
        if i:
            c.x.copy_(cs[i - 1].x_next)
        c.run_layer(x_next=True)
        check_layer(c, Ls[i], h16(c.x))
    dev = torch.device("cuda")
    table = m.decode_layer_table([(c.wr, c.bias, c.ex, c.sh) for c in cs])
    ws = m.alloc_workspace(cs[0].shape, dev)
    y = torch.zeros((T, shape.H), dtype=torch.int16, device=dev)
    xn = torch.zeros((T, shape.H), dtype=torch.int16, device=dev)
    m.moe_decode_layers(cs[0].shape, table, d16(Ls[0].x[:T], dev), y, ws, x_next=xn)
    assert m.moe_query_device_status(ws) == 0
    assert np.array_equal(h16(y), h16(cs[-1].y))
    assert np.array_equal(h16(xn), h16(cs[-1].x_next))
