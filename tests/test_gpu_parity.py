"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: top-k ids, histogram, offsets, permutation, block map,
dequantised bf16 weights. Within tolerance (max|g-r| <= 1e-2*max|r| + 1e-3,
sum|g-r|/sum|r| <= 2e-3): top-k weights (|dw| <= 1e-6), h, expert outputs
and the layer output. Workloads: the named configurations of synth plus
ragged token counts, several tile sizes, no shared expert, skewed routing
with empty experts, and bad expert ids."""
import numpy as np
import pytest
import torch

import bit_moe_expert_histogram_gb300 as m
import oracle
import synth
from moe_case import Case, close, d16, f64, h16

pytestmark = pytest.mark.gpu

FULL = synth.CONFIGS["prefill"].shape
TINY = synth.CONFIGS["tiny"].shape


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    m.load()


_cache = {}


def layer(T, shape, seed=0, zipf=0.0):
    key = (T, shape, seed, zipf)
    if key not in _cache:
        _cache.clear()
        _cache[key] = synth.gen_layer(T, shape, seed=seed, zipf_s=zipf)
    return _cache[key]


# ---------------------------------------------------------------- dequant --
def _dequant_inputs():
    """Random words, every nibble value in every position (rows 0..1), scales
    of both signs over five decades with general biases, and the configs'
    scale / -8*scale pairs (rows 2..3)."""
    rng = np.random.default_rng(11)
    N, Kd = 512, 256
    q = rng.integers(0, 1 << 32, (N, Kd // 8), dtype=np.uint64).astype(np.uint32)
    q[0, :] = 0x76543210
    q[1, :] = 0xFEDCBA98
    s = synth.bf16_bits(rng.uniform(1e-4, 10, (N, Kd // 64)) * rng.choice([-1, 1], (N, Kd // 64)))
    b = synth.bf16_bits(rng.uniform(-100, 100, (N, Kd // 64)))
    s[2:4] = synth.bf16_bits(rng.uniform(0.002, 0.02, (2, Kd // 64)))
    b[2:4] = synth.bf16_bits(-8 * f64(s[2:4]))
    return q, s, b


@pytest.mark.parametrize("routine", ["grouped_gemm", "decode"])
def test_dequant_bitexact(routine):
    """Both device rebuild routines (the grouped GEMMs' natural pairs and
    the decode kernels' (i, i+4) pairs) against the oracle, bit for bit."""
    q, s, b = _dequant_inputs()
    N, Kd = q.shape[0], q.shape[1] * 8
    dev = torch.device("cuda")
    qd = torch.from_numpy(q.view(np.int32)).to(dev)
    out = torch.empty((N, Kd), dtype=torch.int16, device=dev)
    fn = m.moe_debug_dequant_w4 if routine == "grouped_gemm" else m.moe_debug_dequant_w4_decode
    fn(qd, d16(s, dev), d16(b, dev), out)
    torch.cuda.synchronize()
    assert np.array_equal(h16(out), oracle.dequant(q, s, b))


# ------------------------------------------------------------------ route --
@pytest.mark.parametrize("T,shape,zipf", [(16, TINY, 0.0), (1, FULL, 0.0), (37, FULL, 0.0),
                                          (512, FULL, 0.0), (2048, FULL, 1.1)])
def test_route_bitexact(T, shape, zipf):
    L = layer(T, shape, 0, zipf)
    c = Case(L, T, shape)
    m.moe_route(c.shape, c.x, c.wr, c.bias, c.ids, c.w, c.ws)
    assert m.moe_query_device_status(c.ws) == 0
    ids, w32, w64 = oracle.route(L, shape.K)
    assert np.array_equal(c.ids.cpu().numpy(), ids)
    assert np.abs(c.w.cpu().numpy() - w64).max() <= 1e-6
    assert np.allclose(c.w.cpu().numpy().sum(1), 1.0, atol=1e-6)


def test_route_ties_lower_id():
    """Equal router rows: every logit ties -> ids 0..K-1, uniform weights."""
    L = layer(16, TINY, 0)
    c = Case(L, 16, TINY)
    row = d16(L.w_router[:1], c.dev)
    c.wr.copy_(row.expand(TINY.E, -1))
    m.moe_route(c.shape, c.x, c.wr, None, c.ids, c.w, c.ws)
    torch.cuda.synchronize()
    assert (c.ids.cpu().numpy() == np.arange(TINY.K)).all()
    assert np.allclose(c.w.cpu().numpy(), 1.0 / TINY.K, atol=1e-7)


def test_route_screen_all_ties():
    """T >= 64 takes the tensor-core screen: equal router rows tie every
    logit, so every expert is a candidate and ids are 0..K-1."""
    L = layer(128, FULL, 0)
    c = Case(L, 128, FULL)
    row = d16(L.w_router[:1], c.dev)
    c.wr.copy_(row.expand(FULL.E, -1))
    m.moe_route(c.shape, c.x, c.wr, None, c.ids, c.w, c.ws)
    assert m.moe_query_device_status(c.ws) == 0
    assert (c.ids.cpu().numpy() == np.arange(FULL.K)).all()
    assert np.allclose(c.w.cpu().numpy(), 1.0 / FULL.K, atol=1e-7)


def test_route_screen_near_ties():
    """Router rows that differ in one element by one bf16 step: logits closer
    than the screen's margin, so the fixed-order logits decide, bit-exactly."""
    L = layer(256, FULL, 0)
    base = synth.bf16_bits_to_f32(L.w_router[:1]).astype(np.float64)
    rng = np.random.default_rng(11)
    wr = np.repeat(base, FULL.E, axis=0)
    k0 = 5
    wr[:, k0] = base[0, k0] * (1.0 + rng.integers(-4, 5, FULL.E) * 2.0 ** -7)
    wbits = synth.bf16_bits(wr)
    c = Case(L, 256, FULL)
    c.wr.copy_(d16(wbits, c.dev))
    m.moe_route(c.shape, c.x, c.wr, c.bias, c.ids, c.w, c.ws)
    assert m.moe_query_device_status(c.ws) == 0
    ids, _, w64 = oracle.topk(oracle.router_logits(L.x, wbits, L.router_bias), FULL.K)
    assert np.array_equal(c.ids.cpu().numpy(), ids)
    assert np.abs(c.w.cpu().numpy() - w64).max() <= 1e-6


def test_route_screen_ragged_experts_and_tokens():
    """E = 100 (a partial expert tile) and T = 200 (a partial token tile)."""
    shape = synth.LayerShape(H=512, E=100, K=4, I=128, n_shared=1)
    L = synth.gen_layer(200, shape, seed=9, zipf_s=1.1)
    c = Case(L, 200, shape)
    m.moe_route(c.shape, c.x, c.wr, c.bias, c.ids, c.w, c.ws)
    assert m.moe_query_device_status(c.ws) == 0
    ids, _, w64 = oracle.route(L, shape.K)
    assert np.array_equal(c.ids.cpu().numpy(), ids)
    assert np.abs(c.w.cpu().numpy() - w64).max() <= 1e-6


# ------------------------------------------------------------------- plan --
@pytest.mark.parametrize("T,shape,zipf,bm", [(16, TINY, 0.0, 128), (16, TINY, 0.0, 1),
                                             (512, FULL, 0.0, 128), (512, FULL, 0.0, 16),
                                             (2048, FULL, 1.1, 128), (2048, FULL, 1.1, 32),
                                             (1, FULL, 0.0, 128), (300, FULL, 0.0, 64)])
def test_plan_bitexact(T, shape, zipf, bm):
    L = layer(T, shape, 0, zipf)
    c = Case(L, T, shape, tile_rows=bm)
    m.moe_route(c.shape, c.x, c.wr, c.bias, c.ids, c.w, c.ws)
    m.moe_plan(c.shape, c.ids, c.plan, c.ws)
    assert m.moe_query_device_status(c.ws) == 0
    P = oracle.plan(c.ids.cpu().numpy(), shape.E, shape.n_shared, bm)
    G = c.plan_np()
    for k in ("counts", "offsets", "sorted_rows", "row_pos", "block_map"):
        assert np.array_equal(G[k], P[k]), k
    assert G["num_blocks"] == P["num_blocks"]


def test_plan_arbitrary_ids_and_no_shared():
    """moe_plan on caller ids (heavy collisions), without a shared expert."""
    shape = synth.LayerShape(H=256, E=64, K=4, I=128, n_shared=0)
    T = 777
    rng = np.random.default_rng(3)
    ids = rng.integers(0, 5, (T, 4)).astype(np.int32)   # only experts 0..4, repeats allowed
    s = m.make_shape(T, 256, 64, 4, 128, 0, 32)
    dev = torch.device("cuda")
    ws = m.alloc_workspace(s, dev)
    plan = m.PlanBuffers(s, dev)
    m.moe_plan(s, torch.from_numpy(ids).to(dev), plan, ws)
    assert m.moe_query_device_status(ws) == 0
    P = oracle.plan(ids, 64, 0, 32)
    nb = int(plan.num_blocks.item())
    assert nb == P["num_blocks"]
    assert np.array_equal(plan.sorted_rows.cpu().numpy(), P["sorted_rows"])
    assert np.array_equal(plan.row_pos.cpu().numpy(), P["row_pos"])
    assert np.array_equal(plan.block_map.cpu().numpy().reshape(-1, 3)[:nb], P["block_map"])


def test_plan_bad_ids_reported():
    s = m.make_shape(8, 256, 16, 2, 128, 1, 128)
    dev = torch.device("cuda")
    ws = m.alloc_workspace(s, dev)
    plan = m.PlanBuffers(s, dev)
    ids = torch.zeros((8, 2), dtype=torch.int32, device=dev)
    ids[3, 1] = 16
    ids[5, 0] = -1
    m.moe_plan(s, ids, plan, ws)
    assert m.moe_query_device_status(ws) == m.MOE_ERR_BAD_INPUT
    assert m.moe_query_device_status(ws) == 0   # cleared


# -------------------------------------------------------------------- FFN --
def _ffn_check(c, L, tokens=None):
    """Compare y_slots and y with the oracle (all tokens or a sample)."""
    ids = c.ids.cpu().numpy()
    w = c.w.cpu().numpy()
    lg = oracle.router_logits(h16(c.x), L.w_router, L.router_bias)
    ids_o, _, w64 = oracle.topk(lg, c.S.K)
    assert np.array_equal(ids, ids_o)
    assert np.abs(w - w64).max() <= 1e-6
    tok = np.arange(c.T) if tokens is None else np.asarray(tokens)
    y_o, d_o = oracle.layer_tokens(L, ids_o, w64, tokens=tok, x=h16(c.x), want_slots=True)
    row_pos = c.plan.row_pos.cpu().numpy().reshape(c.T, c.S.K)
    ys = f64(h16(c.y_slots))
    K = c.S.K
    g_slots = np.concatenate([ys[row_pos[tok]]] +
                             ([ys[c.R + tok][:, None, :]] if c.S.n_shared else []), axis=1)
    r_slots = d_o[:, :K + c.S.n_shared, :]
    close(g_slots, r_slots, "y_slots")
    close(f64(h16(c.y))[tok], f64(y_o), "y")


@pytest.mark.parametrize("bm", [128, 16])
def test_ffn_tiny_full(bm):
    L = layer(16, TINY, 0)
    c = Case(L, 16, TINY, tile_rows=bm)
    c.run_calls()
    _ffn_check(c, L)


def test_ffn_per_expert_tiny():
    """Each expert's rows of y_slots against the oracle's FFN of that expert."""
    L = layer(16, TINY, 0)
    c = Case(L, 16, TINY)
    c.run_calls()
    P = c.plan_np()
    ys = f64(h16(c.y_slots))
    for e in range(TINY.E):
        lo, hi = P["offsets"][e], P["offsets"][e + 1]
        if lo == hi:
            continue
        xr = L.x[P["sorted_rows"][lo:hi] // TINY.K]
        _, d_o = oracle.expert_ffn(L.q_gate_up[e], L.s_gate_up[e], L.b_gate_up[e],
                                   L.q_down[e], L.s_down[e], L.b_down[e], xr)
        close(ys[lo:hi], d_o, "expert %d" % e)
    _, d_sh = oracle.expert_ffn(L.sh_q_gate_up[0], L.sh_s_gate_up[0], L.sh_b_gate_up[0],
                                L.sh_q_down[0], L.sh_s_down[0], L.sh_b_down[0], L.x)
    close(ys[c.R:], d_sh, "shared")


def test_ffn_prefill_full():
    L = layer(512, FULL, 0)
    c = Case(L, 512, FULL)
    c.run_calls()
    _ffn_check(c, L)


def test_ffn_skewed_sampled():
    """T=2048 with Zipf-shifted logits: empty experts and groups of ~2000
    rows; all routing checked, outputs on a sample of 192 tokens."""
    L = layer(2048, FULL, 0, 1.1)
    c = Case(L, 2048, FULL)
    c.run_calls()
    P = c.plan_np()
    assert (P["counts"] == 0).sum() > 0          # empty experts exist
    assert P["counts"].max() > 128               # several tiles for one expert
    rng = np.random.default_rng(5)
    tok = np.sort(rng.choice(2048, 192, replace=False))
    _ffn_check(c, L, tok)


@pytest.mark.parametrize("T", [1, 3, 37])
def test_ffn_small_and_ragged_T(T):
    L = layer(T, FULL, 1)
    c = Case(L, T, FULL)
    c.run_calls()
    _ffn_check(c, L)


def test_ffn_no_shared_expert():
    shape = synth.LayerShape(H=256, E=16, K=2, I=128, n_shared=0)
    L = synth.gen_layer(40, shape, seed=4)
    c = Case(L, 40, shape, tile_rows=32)
    c.run_calls()
    _ffn_check(c, L)


# ------------------------------------------------------------------ layer --
def test_layer_call_equals_four_calls_and_oracle():
    L = layer(512, FULL, 0)
    c = Case(L, 512, FULL)
    c.run_calls(x_next=True)
    y4 = h16(c.y).copy()
    xn4 = h16(c.x_next).copy()
    c.y.zero_()
    c.x_next.zero_()
    c.run_layer(x_next=True)
    assert np.array_equal(h16(c.y), y4)
    assert np.array_equal(h16(c.x_next), xn4)
    close(f64(xn4), f64(oracle.rmsnorm_rows(y4)), "x_next")


@pytest.mark.parametrize("T,zipf", [(64, 0.0), (77, 0.0), (2048, 1.1)])
def test_layer_call_plan_counted_by_router_screen(T, zipf):
    """From 64 tokens the layer call has the router's screen count the plan's
    per-chunk histogram (no histogram launch): the same ids, weights and y as
    the four calls, at the threshold, with a ragged last chunk and with
    skewed routing; a second call on the same workspace (the histogram zeroed
    again) gives the same bits."""
    L = layer(T, FULL, 3, zipf)
    c = Case(L, T, FULL)
    c.run_calls()
    ids4, w4, y4 = c.ids.cpu().numpy().copy(), c.w.cpu().numpy().copy(), h16(c.y).copy()
    for _ in range(2):
        c.ids.fill_(-7)
        c.w.zero_()
        c.y.zero_()
        c.run_layer()
        assert np.array_equal(c.ids.cpu().numpy(), ids4)
        assert np.array_equal(c.w.cpu().numpy(), w4)
        assert np.array_equal(h16(c.y), y4)


def test_determinism_two_runs():
    L = layer(512, FULL, 0)
    c = Case(L, 512, FULL)
    c.run_calls()
    a = h16(c.y).copy()
    b_ = h16(c.y_slots).copy()
    c.run_calls()
    assert np.array_equal(h16(c.y), a)
    assert np.array_equal(h16(c.y_slots), b_)


@pytest.mark.parametrize("E", [16, 100, 256])
def test_plan_after_ffn_dirtied_shared_memory(E):
    """The plan's per-warp count table must be cleared for every expert,
    whatever earlier kernels left in shared memory (the FFN fills it)."""
    L = layer(512, FULL, 0)
    c = Case(L, 512, FULL)
    c.run_calls()                      # leaves FFN data in shared memory
    T, K = 700, 4
    rng = np.random.default_rng(E)
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    s = m.make_shape(T, 256, E, K, 128, 1, 64)
    dev = torch.device("cuda")
    ws = m.alloc_workspace(s, dev)
    plan = m.PlanBuffers(s, dev)
    m.moe_plan(s, torch.from_numpy(ids).to(dev), plan, ws)
    assert m.moe_query_device_status(ws) == 0
    P = oracle.plan(ids, E, 1, 64)
    assert np.array_equal(plan.sorted_rows.cpu().numpy(), P["sorted_rows"])
    assert np.array_equal(plan.row_pos.cpu().numpy(), P["row_pos"])
    nb = int(plan.num_blocks.item())
    assert np.array_equal(plan.block_map.cpu().numpy().reshape(-1, 3)[:nb], P["block_map"])


def test_back_to_back_steps_match_single_step():
    """20 full layer steps queued without a host sync give the same bits as
    one step, and the oracle's output within tolerance."""
    L = layer(512, FULL, 0)
    c = Case(L, 512, FULL)
    c.run_calls()
    y1 = h16(c.y).copy()
    for _ in range(20):
        m.moe_route(c.shape, c.x, c.wr, c.bias, c.ids, c.w, c.ws)
        m.moe_plan(c.shape, c.ids, c.plan, c.ws)
        m.moe_expert_ffn_w4(c.shape, c.x, c.ex, c.sh, c.plan, c.y_slots, c.ws)
        m.moe_combine(c.shape, c.y_slots, c.plan.row_pos, c.w, c.y, None)
    assert m.moe_query_device_status(c.ws) == 0
    assert np.array_equal(h16(c.y), y1)
    _ffn_check(c, L, np.arange(0, 512, 8))


def test_chunked_prefill_reuses_one_workspace():
    """A prompt in two chunks of 256 tokens through two stacked layers with one
    workspace ("Prefill": a long prompt runs in bounded chunks): each call's
    routing is bit-exact and its output within tolerance of the oracle on the
    GPU's own input (teacher-forced), sampled on 24 tokens per call."""
    Tc, S = 256, FULL
    dev = torch.device("cuda")
    layers = [synth.gen_layer(Tc, S, seed=30 + l) for l in range(2)]
    wts = []
    for L in layers:
        wts.append((d16(L.w_router, dev),
                    m.ExpertWeights.from_numpy(L.q_gate_up, L.s_gate_up, L.b_gate_up, L.q_down,
                                               L.s_down, L.b_down, dev),
                    m.ExpertWeights.from_numpy(L.sh_q_gate_up, L.sh_s_gate_up, L.sh_b_gate_up,
                                               L.sh_q_down, L.sh_s_down, L.sh_b_down, dev)))
    shape = m.make_shape(Tc, S.H, S.E, S.K, S.I, S.n_shared, 128)
    ws = m.alloc_workspace(shape, dev)
    ids = torch.empty((Tc, S.K), dtype=torch.int32, device=dev)
    w = torch.empty((Tc, S.K), dtype=torch.float32, device=dev)
    y = torch.empty((Tc, S.H), dtype=torch.int16, device=dev)
    xn = [torch.empty((Tc, S.H), dtype=torch.int16, device=dev) for _ in range(2)]
    rng = np.random.default_rng(3)
    for c in range(2):
        x = d16(synth.gen_tokens(Tc, S.H, 500 + c), dev)
        for l, (L, (wr, ex, sh)) in enumerate(zip(layers, wts)):
            m.moe_layer_w4(shape, x, wr, None, ex, sh, y, ws, x_next=xn[l], topk_ids=ids, topk_w=w)
            assert m.moe_query_device_status(ws) == 0
            xin = h16(x)
            ids_o, _, w64 = oracle.topk(oracle.router_logits(xin, L.w_router, None), S.K)
            assert np.array_equal(ids.cpu().numpy(), ids_o)
            tok = np.sort(rng.choice(Tc, 24, replace=False))
            y_o = oracle.layer_tokens(L, ids_o, w64, tokens=tok, x=xin)
            close(f64(h16(y))[tok], f64(y_o), "chunk %d layer %d" % (c, l))
            x = xn[l]
