"""GPU parity of the decoder blocks around the MoE layers (moe_decoder_blocks):
the pre-norm with a learned gain, the layer, the residual add, and the token
feed from device memory ("Perplexity Open Sources Lily: A Rust + Metal
Inference Engine for Qwen3.6-35B-A3B on Apple Silicon", section "Decode:
Minimize Bytes Moved Per Token": the sampled token id stays on the device
and feeds the next step). Each layer is checked against the oracle
teacher-forced on the device's residual stream; launches, aliasing, the
embedding gather and a captured decode loop are checked bit for bit."""
import numpy as np
import pytest
import torch

import bit_moe_expert_histogram_gb300 as m
import oracle
import synth
from moe_case import close, d16, f64, h16

pytestmark = pytest.mark.gpu

FULL = synth.CONFIGS["decode"].shape
TINY = synth.CONFIGS["tiny"].shape


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    m.load()


class Stack:
    """n layers of one shape on the device, their gains, and a workspace."""

    def __init__(self, shape, T, n, seed):
        self.dev = torch.device("cuda")
        self.S, self.T = shape, T
        self.Ls = [synth.gen_layer(T, shape, seed=seed + i) for i in range(n)]
        self.g = [synth.gen_gain(shape.H, seed=seed + 1000 + i) for i in range(n)]
        self.shape = m.make_shape(T, shape.H, shape.E, shape.K, shape.I, shape.n_shared, 128)
        self.keep = []
        rows = []
        for L in self.Ls:
            wr = d16(L.w_router, self.dev)
            bias = None if L.router_bias is None else torch.from_numpy(L.router_bias).to(self.dev)
            ex = m.ExpertWeights.from_numpy(L.q_gate_up, L.s_gate_up, L.b_gate_up, L.q_down,
                                            L.s_down, L.b_down, self.dev)
            sh = None
            if shape.n_shared:
                sh = m.ExpertWeights.from_numpy(L.sh_q_gate_up, L.sh_s_gate_up, L.sh_b_gate_up,
                                                L.sh_q_down, L.sh_s_down, L.sh_b_down, self.dev)
            rows.append((wr, bias, ex, sh))
        self.keep.append(rows)
        self.gd = [d16(g, self.dev) for g in self.g]
        self.table = m.decode_layer_table(rows)
        self.gains = m.gain_table(self.gd)
        self.ws = m.alloc_workspace(self.shape, self.dev)

    def sub(self, lo, hi):
        """Layer table and gain table of layers lo..hi-1."""
        table = (m.LayerWeights * (hi - lo))(*self.table[lo:hi])
        gains = m.gain_table(self.gd[lo:hi])
        return table, gains

    def run(self, h_in, lo=0, hi=None, out=None, **kw):
        hi = len(self.Ls) if hi is None else hi
        table, gains = self.sub(lo, hi)
        out = torch.empty((self.T, self.S.H), dtype=torch.int16, device=self.dev) if out is None else out
        m.moe_decoder_blocks(self.shape, table, gains, out, self.ws, h_in=h_in, **kw)
        return out


@pytest.mark.parametrize("shape,T,n_layers", [(FULL, 1, 3), (FULL, 2, 3), (TINY, 3, 3),
                                              (TINY, 40, 3), (FULL, 64, 2)])
def test_block_layers_teacher_forced(shape, T, n_layers):
    """After each layer the residual stream matches the oracle block applied
    to the device's stream of the layer before (T <= 4: the persistent
    kernel; more tokens: the four calls with the residual add and the next
    pre-norm in the combine)."""
    st = Stack(shape, T, n_layers, seed=200)
    h0 = st.Ls[0].x[:T].copy()
    prev = h0
    for n in range(1, n_layers + 1):
        out = st.run(d16(h0, st.dev), 0, n)
        assert m.moe_query_device_status(st.ws) == 0
        h_o, _ = oracle.decoder_blocks([st.Ls[n - 1]], [st.g[n - 1]], prev, shape.K)
        got = h16(out)
        close(f64(got), f64(h_o), "h after %d layers" % n)
        # the layer's own contribution, against the oracle's
        close(f64(got) - f64(prev), f64(h_o) - f64(prev), "h - h_in, layer %d" % n)
        prev = got


@pytest.mark.parametrize("T", [2, 24])
def test_block_is_deterministic_and_may_write_its_input(T):
    st = Stack(TINY, T, 4, seed=300)
    h0 = d16(st.Ls[0].x[:T], st.dev)
    a = h16(st.run(h0.clone())).copy()
    b = h16(st.run(h0.clone())).copy()
    assert np.array_equal(a, b)
    buf = h0.clone()
    st.run(buf, out=buf)  # h_out aliases h_in
    assert m.moe_query_device_status(st.ws) == 0
    assert np.array_equal(h16(buf), a)


def test_block_split_over_launches():
    """50 layers (one launch runs 48): the residual stream is handed from
    launch to launch, and the result is that of two calls."""
    st = Stack(TINY, 1, 50, seed=400)
    h0 = d16(st.Ls[0].x[:1], st.dev)
    whole = h16(st.run(h0)).copy()
    mid = st.run(h0, 0, 48)
    two = h16(st.run(mid.clone(), 48, 50)).copy()
    assert m.moe_query_device_status(st.ws) == 0
    assert np.array_equal(whole, two)


@pytest.mark.parametrize("shape,T", [(FULL, 3), (TINY, 12)])
def test_block_token_feed_from_the_embedding_table(shape, T):
    """Token ids in device memory: h_0 is the ids' embedding rows, gathered
    on the device; an id outside the table is recorded and reads as zeros."""
    V = 1000
    st = Stack(shape, T, 2, seed=500)
    emb_h = synth.gen_embed(V, shape.H, seed=501)
    emb = d16(emb_h, st.dev)
    pick = (np.arange(T) * 397 + 7) % V
    pick[1] = V - 1
    ids = torch.tensor(pick, dtype=torch.int32, device=st.dev)
    got = h16(st.run(None, token_ids=ids, embed=emb)).copy()
    assert m.moe_query_device_status(st.ws) == 0
    ref = h16(st.run(d16(emb_h[pick], st.dev))).copy()
    assert np.array_equal(got, ref)
    bad_pick = pick.copy()
    bad_pick[1] = V
    bad = torch.tensor(bad_pick, dtype=torch.int32, device=st.dev)
    got_bad = h16(st.run(None, token_ids=bad, embed=emb)).copy()
    assert m.moe_query_device_status(st.ws) == m.MOE_ERR_BAD_INPUT
    h_zero = emb_h[pick].copy()
    h_zero[1] = 0
    ref_bad = h16(st.run(d16(h_zero, st.dev))).copy()
    assert np.array_equal(got_bad, ref_bad)


def test_block_decode_loop_captured_in_a_graph():
    """Four decode steps in one CUDA graph: each step's token id is picked
    on the device from the previous step's residual stream (a stand-in for
    the model's head: the largest of the first V channels) and written into
    the id slot the next step's blocks read. Nothing returns to the host
    between steps; the replay equals the same steps run eagerly."""
    T, V, steps = 1, 200, 4
    st = Stack(TINY, T, 3, seed=600)
    emb = d16(synth.gen_embed(V, TINY.H, seed=601), st.dev)
    ids0 = torch.tensor([42], dtype=torch.int32, device=st.dev)
    tok = torch.empty_like(ids0)
    outs = [torch.empty((T, TINY.H), dtype=torch.int16, device=st.dev) for _ in range(steps)]
    table, gains = st.sub(0, 3)

    def loop():
        tok.copy_(ids0)
        for s in range(steps):
            m.moe_decoder_blocks(st.shape, table, gains, outs[s], st.ws, token_ids=tok, embed=emb)
            h = outs[s].view(torch.bfloat16)[:, :V].float()
            tok.copy_(torch.argmax(h, dim=1).to(torch.int32))

    loop()
    torch.cuda.synchronize()
    eager = [h16(o).copy() for o in outs]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        loop()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        loop()
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert m.moe_query_device_status(st.ws) == 0
    for a, b in zip(eager, outs):
        assert np.array_equal(a, h16(b))
    # the steps differ: each fed the previous step's pick
    assert not np.array_equal(eager[0], eager[1])


def test_block_rejects_bad_arguments():
    st = Stack(TINY, 1, 1, seed=700)
    table, gains = st.sub(0, 1)
    out = torch.empty((1, TINY.H), dtype=torch.int16, device=st.dev)
    with pytest.raises(m.MoeError):
        m.moe_decoder_blocks(st.shape, table, gains, out, st.ws)  # neither h_in nor token ids
    with pytest.raises(ValueError):
        m.moe_decoder_blocks(st.shape, table, m.gain_table([]), out, st.ws, h_in=out)
    wide = m.make_shape(2, 8192, TINY.E, TINY.K, TINY.I, TINY.n_shared, 128)
    with pytest.raises(m.MoeError):  # a workspace sized for another shape
        m.moe_decoder_blocks(wide, table, gains, out, st.ws, h_in=out)
