"""GPU parity of the two stacked workloads at their stated sizes.

Decode: one token through 40 distinct full-shape layers (H=2048, 256
experts top-8 + 1 shared, I=512; 18.2 GB of packed weights), each layer's
unit-RMS output feeding the next ("Perplexity Open Sources Lily: A Rust +
Metal Inference Engine for Qwen3.6-35B-A3B on Apple Silicon", section
"Decode: Minimize Bytes Moved Per Token"). Every layer is checked against
the oracle on the GPU's own input (teacher-forced), and the single
persistent launch over all 40 layers must give the chain's last bits.

Chunked prefill: a 16384-token prompt in 8 chunks of 2048 tokens through
the same 40 layers with one workspace ("Prefill: Keep Weights Packed, Keep
Routing on the GPU": long prompts run in bounded chunks), chunk-outer and
layer-inner. On every one of the 320 chunk-layer calls the routing and the
plan are checked bit for bit against the oracle on the call's own input,
and the output on a seeded sample of 16 tokens within the layer's
tolerance; the activation scratch stays under 2 GiB.

Only one layer's host copy is alive at a time: the weights live on the
device and the oracle's copy is drawn again, layer by layer, from the
same seed when checking."""
import numpy as np
import pytest
import torch

import bit_moe_expert_histogram_gb300 as m
import oracle
import synth
from moe_case import close, d16, f64, h16

pytestmark = pytest.mark.gpu

FULL = synth.CONFIGS["decode"].shape
N_LAYERS = synth.CONFIGS["decode"].layers          # 40
CHUNK = synth.CONFIGS["chunked"].chunk              # 2048
N_CHUNKS = synth.CONFIGS["chunked"].total_tokens // CHUNK   # 8
SAMPLE = 16
TWO_GIB = 2 * 1024 ** 3


def upload(L, dev):
    ex = m.ExpertWeights.from_numpy(L.q_gate_up, L.s_gate_up, L.b_gate_up, L.q_down, L.s_down,
                                    L.b_down, dev)
    sh = m.ExpertWeights.from_numpy(L.sh_q_gate_up, L.sh_s_gate_up, L.sh_b_gate_up,
                                    L.sh_q_down, L.sh_s_down, L.sh_b_down, dev)
    return d16(L.w_router, dev), None, ex, sh


def sample_tokens(c, l):
    rng = np.random.default_rng(1000 * c + l)
    return np.sort(rng.choice(CHUNK, SAMPLE, replace=False))


@pytest.fixture(scope="module")
def stack():
    """Draws the 40 layers (seed = layer index), keeps their weights on the
    device, and runs the decode chain through them while each layer's host
    copy is at hand, recording what the decode test asserts."""
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    m.load()
    dev = torch.device("cuda")
    H, K = FULL.H, FULL.K
    s1 = m.make_shape(1, H, FULL.E, K, FULL.I, FULL.n_shared, 128)
    ws = m.alloc_workspace(s1, dev)
    ids = torch.empty((1, K), dtype=torch.int32, device=dev)
    w = torch.empty((1, K), dtype=torch.float32, device=dev)
    y = torch.empty((1, H), dtype=torch.int16, device=dev)
    xs = [torch.empty((1, H), dtype=torch.int16, device=dev) for _ in range(2)]
    x0 = d16(synth.gen_tokens(1, H, 10 ** 6), dev)
    x = x0
    layers, decode = [], []
    for l in range(N_LAYERS):
        L = synth.gen_layer(1, FULL, seed=l)
        layers.append(upload(L, dev))
        wr, bias, ex, sh = layers[-1]
        xn = xs[l % 2]
        m.moe_layer_w4(s1, x, wr, bias, ex, sh, y, ws, x_next=xn, topk_ids=ids, topk_w=w)
        st = m.moe_query_device_status(ws)
        xin = h16(x).copy()
        ids_o, _, w64 = oracle.topk(oracle.router_logits(xin, L.w_router, None), K)
        y_o = oracle.layer_tokens(L, ids_o, w64, x=xin)
        y_g = h16(y).copy()
        decode.append(dict(status=st, ids=ids.cpu().numpy().copy(), ids_o=ids_o,
                           w=w.cpu().numpy().copy(), w64=w64, y=y_g, y_o=y_o,
                           xn=h16(xn).copy(), xn_o=oracle.rmsnorm_rows(y_g)))
        x = xn
        del L
    table = m.decode_layer_table(layers)
    ws2 = m.alloc_workspace(s1, dev)
    y2 = torch.zeros((1, H), dtype=torch.int16, device=dev)
    xn2 = torch.zeros((1, H), dtype=torch.int16, device=dev)
    m.moe_decode_layers(s1, table, x0, y2, ws2, x_next=xn2)
    persist = dict(status=m.moe_query_device_status(ws2), y=h16(y2).copy(), xn=h16(xn2).copy(),
                   path=m.moe_layer_path(s1))
    del ws, ws2
    return dict(dev=dev, layers=layers, decode=decode, persist=persist)


def test_decode_forty_full_layers_teacher_forced(stack):
    """Config 3: each of the 40 layers against the oracle on the GPU's own
    input (ids bit-exact, weights within 1e-6, y and the next input within
    the layer's tolerance), then the persistent launch over all 40 layers
    equal to the chain bit for bit."""
    for l, r in enumerate(stack["decode"]):
        assert r["status"] == 0, "layer %d status %d" % (l, r["status"])
        assert np.array_equal(r["ids"], r["ids_o"]), "layer %d ids" % l
        assert np.abs(r["w"] - r["w64"]).max() <= 1e-6, "layer %d weights" % l
        close(f64(r["y"]), f64(r["y_o"]), "layer %d y" % l)
        close(f64(r["xn"]), f64(r["xn_o"]), "layer %d x_next" % l)
    p = stack["persist"]
    assert p["path"] == 2
    assert p["status"] == 0
    assert np.array_equal(p["y"], stack["decode"][-1]["y"])
    assert np.array_equal(p["xn"], stack["decode"][-1]["xn"])


def test_chunked_prefill_8x2048_through_40_layers(stack):
    """Config 4 at its stated size, with one workspace for all 320 calls."""
    dev = stack["dev"]
    H, E, K, I = FULL.H, FULL.E, FULL.K, FULL.I
    shape = m.make_shape(CHUNK, H, E, K, I, FULL.n_shared, 128)
    ws = m.alloc_workspace(shape, dev)
    R, S = CHUNK * K, CHUNK * (K + FULL.n_shared)
    ids = torch.empty((CHUNK, K), dtype=torch.int32, device=dev)
    w = torch.empty((CHUNK, K), dtype=torch.float32, device=dev)
    plan = m.PlanBuffers(shape, dev)
    y_slots = torch.empty((S, H), dtype=torch.int16, device=dev)
    y = torch.empty((CHUNK, H), dtype=torch.int16, device=dev)
    xs = [torch.empty((CHUNK, H), dtype=torch.int16, device=dev) for _ in range(2)]
    buffers = [ids, w, y_slots, y] + xs + [plan.counts, plan.offsets, plan.sorted_rows,
                                          plan.row_pos, plan.block_map, plan.num_blocks]
    scratch = ws.numel() * ws.element_size() + sum(t.numel() * t.element_size()
                                                   for t in buffers)
    assert scratch <= TWO_GIB, "activation scratch %d bytes" % scratch
    # what each call saw and produced, kept on the device for the check
    x_in = torch.empty((N_CHUNKS, N_LAYERS, CHUNK, H), dtype=torch.int16, device=dev)
    ids_all = torch.empty((N_CHUNKS, N_LAYERS, CHUNK, K), dtype=torch.int32, device=dev)
    w_all = torch.empty((N_CHUNKS, N_LAYERS, CHUNK, K), dtype=torch.float32, device=dev)
    sr_all = torch.empty((N_CHUNKS, N_LAYERS, R), dtype=torch.int32, device=dev)
    rp_all = torch.empty((N_CHUNKS, N_LAYERS, R), dtype=torch.int32, device=dev)
    cnt_all = torch.empty((N_CHUNKS, N_LAYERS, E), dtype=torch.int32, device=dev)
    off_all = torch.empty((N_CHUNKS, N_LAYERS, E + 1), dtype=torch.int32, device=dev)
    bm_all = torch.empty((N_CHUNKS, N_LAYERS, plan.block_map.numel()), dtype=torch.int32,
                         device=dev)
    nb_all = torch.empty((N_CHUNKS, N_LAYERS), dtype=torch.int32, device=dev)
    y_smp = torch.empty((N_CHUNKS, N_LAYERS, SAMPLE, H), dtype=torch.int16, device=dev)
    for c in range(N_CHUNKS):
        x = d16(synth.gen_tokens(CHUNK, H, 10 ** 6 + c), dev)
        for l, (wr, bias, ex, sh) in enumerate(stack["layers"]):
            x_in[c, l].copy_(x)
            xn = xs[l % 2]
            m.moe_route(shape, x, wr, bias, ids, w, ws)
            m.moe_plan(shape, ids, plan, ws)
            m.moe_expert_ffn_w4(shape, x, ex, sh, plan, y_slots, ws)
            m.moe_combine(shape, y_slots, plan.row_pos, w, y, xn)
            ids_all[c, l].copy_(ids)
            w_all[c, l].copy_(w)
            sr_all[c, l].copy_(plan.sorted_rows)
            rp_all[c, l].copy_(plan.row_pos)
            cnt_all[c, l].copy_(plan.counts)
            off_all[c, l].copy_(plan.offsets)
            bm_all[c, l].copy_(plan.block_map.view(-1))
            nb_all[c, l].copy_(plan.num_blocks.view(()))
            tok = torch.from_numpy(sample_tokens(c, l)).to(dev)
            y_smp[c, l].copy_(y.index_select(0, tok))
            x = xn
        assert m.moe_query_device_status(ws) == 0, "chunk %d" % c
    for l in range(N_LAYERS):
        L = synth.gen_layer(1, FULL, seed=l)
        for c in range(N_CHUNKS):
            where = "chunk %d layer %d" % (c, l)
            xin = h16(x_in[c, l])
            ids_o, _, w64 = oracle.topk(oracle.router_logits(xin, L.w_router, None), K)
            assert np.array_equal(ids_all[c, l].cpu().numpy(), ids_o), where + " ids"
            assert np.abs(w_all[c, l].cpu().numpy() - w64).max() <= 1e-6, where + " weights"
            P = oracle.plan(ids_o, E, FULL.n_shared, 128)
            nb = int(nb_all[c, l].item())
            assert nb == P["num_blocks"], where + " num_blocks"
            assert np.array_equal(cnt_all[c, l].cpu().numpy(), P["counts"]), where + " counts"
            assert np.array_equal(off_all[c, l].cpu().numpy(), P["offsets"]), where + " offsets"
            assert np.array_equal(sr_all[c, l].cpu().numpy(), P["sorted_rows"]), where + " rows"
            assert np.array_equal(rp_all[c, l].cpu().numpy(), P["row_pos"]), where + " row_pos"
            bm = bm_all[c, l].cpu().numpy().reshape(-1, 3)[:nb]
            assert np.array_equal(bm, P["block_map"]), where + " block map"
            tok = sample_tokens(c, l)
            y_o = oracle.layer_tokens(L, ids_o, w64, tokens=tok, x=xin)
            close(f64(h16(y_smp[c, l])), f64(y_o), where + " y")
        del L
