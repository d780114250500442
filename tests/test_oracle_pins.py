"""Pins of the CPU oracle to facts other than itself: closed forms, library
routines (torch's fp32->bf16 rounding, numpy's stable argsort, scipy's
softmax), a standard floating-point error bound, the hand-worked one-token
example under tests/golden/, invariants, and the independent brute-force
dense reference (oracle/dense.py)."""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
import synth
from oracle import dense

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def f32_bits(v):
    return int(np.float32(v).view(np.uint32))


def torch_bf16_bits(v32):
    t = torch.tensor(np.asarray(v32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


# ------------------------------------------------------------------ bf16 --
def test_bf16_rne_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-30, 30, 5000),
                        np.float32([0.0, -0.0, 1.0, -1.0, 3.0e38, 1.0e-40, -2.5e-39])])
    v = v.astype(np.float32)
    want = torch_bf16_bits(v)
    got = np.array([oracle.bf16_rne(float(a)) for a in v], np.uint16)
    assert (got == want).all()


def test_bf16_rne_ties_to_even_and_single_rounding():
    one = 0x3F80
    assert oracle.bf16_rne(1.0 + 2.0 ** -8) == one              # tie -> even (1.0)
    assert oracle.bf16_rne(1.0 + 3 * 2.0 ** -8) == one + 2      # tie -> even (up)
    # just above a tie, below fp32 resolution: rounding via fp32 would tie to even
    assert oracle.bf16_rne(1.0 + 2.0 ** -8 + 2.0 ** -40) == one + 1
    assert oracle.bf16_rne(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0x8000 | (one + 1)
    assert oracle.bf16_rne(float("inf")) == 0x7F80
    assert oracle.bf16_rne(3.5e38) == 0x7F80                    # overflow
    for b in (0x0001, 0x3F80, 0x7F7F, 0xBF80, 0x0080):
        assert oracle.bf16_rne(oracle.bf16_value(b)) == b


# ---------------------------------------------------------------- router --
def _bits(vals):
    return synth.bf16_bits(np.asarray(vals, np.float64))


def test_router_logit_error_bound_vs_exact():
    """|L - exact| <= (H/32 + 5) * 2^-24 * sum|x w| (Higham, Accuracy and
    Stability of Numerical Algorithms, sec. 3.1: recursive summation of n
    terms errs by at most (n-1)u sum|x_i|; here each partial sums H/32
    exact products, then 5 pairwise levels)."""
    rng = np.random.default_rng(2)
    for H in (256, 2048):
        x = _bits(rng.standard_normal((8, H)))
        w = _bits(rng.standard_normal((32, H)) / math.sqrt(H))
        lg = oracle.router_logits(x, w)
        xf = synth.bf16_bits_to_f32(x).astype(np.float64)
        wf = synth.bf16_bits_to_f32(w).astype(np.float64)
        exact = xf @ wf.T
        bound = (H / 32 + 5) * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf).T)
        assert (np.abs(lg - exact) <= bound).all()


def test_router_logit_tree_order():
    """The fixed fp32 order is observable: big values cancel or absorb
    depending on which partial holds them."""
    H = 256
    B = 2.0 ** 24
    w = np.zeros(H)
    x = np.ones(H)
    # partial 0 holds +B (k=0), partial 1 holds +1 (k=8), partial 16 holds -B (k=128)
    w[0], w[8], w[128] = B, 1.0, -B
    assert oracle.router_logits(_bits(x)[None], _bits(w)[None])[0, 0] == 1.0
    # partial 0 holds +B, partial 1 holds -B, partial 16 holds +1: the +1 is
    # absorbed at the distance-16 step (B + 1 rounds to B in fp32), result 0
    w[:] = 0
    w[0], w[8], w[128] = B, -B, 1.0
    assert oracle.router_logits(_bits(x)[None], _bits(w)[None])[0, 0] == 0.0
    # plain left-to-right summation would give 1 here: the order is not sequential
    assert (np.float32(B) + np.float32(-B)) + np.float32(1.0) == 1.0


def test_router_single_term_and_bias_exact():
    H, E = 256, 4
    x = np.zeros((1, H)); x[0, 77] = 1.5
    w = np.zeros((E, H)); w[:, 77] = [0.25, -2.0, 3.0, 0.0]
    bias = np.float32([0.5, 0.25, -1.0, 7.0])
    lg = oracle.router_logits(_bits(x), _bits(w), bias)
    assert lg.tolist() == [[0.375 + 0.5, -3.0 + 0.25, 4.5 - 1.0, 7.0]]


# ------------------------------------------------------------------ top-k --
def test_topk_ties_lower_id_and_uniform_weights():
    g = json.load(open(os.path.join(GOLD, "tie_router.json")))
    lg = np.zeros((1, 16), np.float32)
    ids, w32, w64 = oracle.topk(lg, 2)
    assert ids[0].tolist() == g["expected"]["ids"]
    assert np.allclose(w64[0], g["expected"]["weights"], atol=0, rtol=1e-15)
    lg = np.full((3, 256), -0.0, np.float32); lg[:, ::2] = 0.0   # -0 == +0
    ids, _, w64 = oracle.topk(lg, 8)
    assert (ids == np.arange(8)).all() and np.allclose(w64, 1 / 8)


def test_topk_matches_lexsort_and_scipy_softmax():
    rng = np.random.default_rng(3)
    lg = rng.integers(-6, 6, size=(200, 64)).astype(np.float32) * 0.5   # many ties
    K = 8
    ids, w32, w64 = oracle.topk(lg, K)
    E = lg.shape[1]
    for t in range(lg.shape[0]):
        order = np.lexsort((np.arange(E), -lg[t]))
        assert ids[t].tolist() == order[:K].tolist()
        assert np.allclose(w64[t], softmax(lg[t, order[:K]].astype(np.float64)), rtol=1e-13)
    assert np.allclose(w64.sum(1), 1.0, atol=1e-14)
    assert np.abs(w32 - w64).max() < 1e-7


# ------------------------------------------------------------------- plan --
@pytest.mark.parametrize("T,E,K,BM,skew", [(16, 16, 2, 128, 0), (513, 256, 8, 128, 0),
                                           (300, 256, 8, 32, 1), (1, 256, 8, 16, 0),
                                           (7, 4, 4, 1, 0)])
def test_plan_invariants_and_stable_sort(T, E, K, BM, skew):
    rng = np.random.default_rng(T + E)
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        ids = np.stack([rng.choice(E, K, replace=False, p=p / p.sum()) for _ in range(T)])
    else:
        ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)])
    ids = ids.astype(np.int32)
    P = oracle.plan(ids, E, 1, BM)
    R = T * K
    flat = ids.ravel()
    assert (P["counts"] == np.bincount(flat, minlength=E)).all()
    assert P["counts"].sum() == R
    assert P["offsets"][0] == 0 and P["offsets"][-1] == R
    assert (np.diff(P["offsets"]) == P["counts"]).all()
    assert (P["sorted_rows"] == np.argsort(flat, kind="stable")).all()
    assert (np.sort(P["sorted_rows"]) == np.arange(R)).all()
    assert (P["row_pos"][P["sorted_rows"]] == np.arange(R)).all()
    bm = P["block_map"]
    assert P["num_blocks"] == sum(-(-int(c) // BM) for c in P["counts"]) + -(-T // BM)
    assert ((bm[:, 2] >= 1) & (bm[:, 2] <= BM)).all()
    assert bm[:, 2].sum() == R + T
    for e, r0, n in bm:
        if e < E:
            assert (flat[P["sorted_rows"][r0:r0 + n]] == e).all()
        else:
            assert r0 >= R and r0 + n <= R + T
    assert (np.diff(bm[:, 0]) >= 0).all()


def test_plan_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.plan(np.array([[0, 16]], np.int32), 16, 1, 8)


# ---------------------------------------------------------------- dequant --
def test_dequant_nibble_order():
    q = np.array([[0x76543210, 0xFEDCBA98] * 4], np.uint32)     # K = 64
    s = _bits([[1.0]])
    b = _bits([[0.0]])
    got = synth.bf16_bits_to_f32(oracle.dequant(q, s, b))[0]
    assert got.tolist() == list(range(16)) * 4


def test_dequant_closed_form_all_q():
    """b = -8s makes s*q + b = s*(q-8), exact in fp32; rounding that fp32
    value to bf16 is torch's fp32->bf16 conversion. q-8 in {+-1,2,4,8,0}
    must come out exactly s*(q-8)."""
    rng = np.random.default_rng(4)
    n = 2000
    s = _bits(rng.uniform(0.002, 0.02, n) * 10.0 ** rng.integers(-3, 4, n))
    sv = synth.bf16_bits_to_f32(s).astype(np.float64)
    b = _bits(-8 * sv)
    for qv in range(16):
        word = sum(qv << (4 * i) for i in range(8))
        q = np.full((n, 8), word, np.uint32)
        got = oracle.dequant(q, s[:, None], b[:, None])
        want = torch_bf16_bits((sv * (qv - 8)).astype(np.float32))
        assert (got == want[:, None]).all(), qv
        if qv - 8 in (0, 1, -1, 2, -2, 4, -4, -8):
            assert (synth.bf16_bits_to_f32(got[:, 0]) == sv * (qv - 8)).all()


def test_dequant_general_bias_matches_dense():
    rng = np.random.default_rng(5)
    q = rng.integers(0, 1 << 32, (64, 32), dtype=np.uint64).astype(np.uint32)
    s = _bits(rng.uniform(-1, 1, (64, 4)))
    b = _bits(rng.uniform(-3, 3, (64, 4)))
    got = synth.bf16_bits_to_f32(oracle.dequant(q, s, b)).astype(np.float64)
    assert (got == dense.dequant(q, s, b)).all()


# -------------------------------------------------------------- hand case --
def _hand_layer():
    g = json.load(open(os.path.join(GOLD, "hand_worked_1token.json")))
    sh = g["shape"]
    H, E, I = sh["H"], sh["E"], sh["I"]
    def word(n):
        return sum(n << (4 * i) for i in range(8))
    s = synth.bf16_bits(np.full(1, 2.0 ** -8))[0]
    b = synth.bf16_bits(np.full(1, -8 * 2.0 ** -8))[0]
    qgu = np.full((E, 2 * I, H // 8), word(9), np.uint32)
    qd = np.full((E, H, I // 8), word(8), np.uint32)
    qd[15] = word(10)
    qd[14] = word(7)
    L = synth.LayerInputs(
        x=synth.bf16_bits(np.ones((1, H))),
        w_router=synth.bf16_bits(np.repeat(np.arange(E)[:, None] / 1024.0, H, 1)),
        router_bias=None,
        q_gate_up=qgu, s_gate_up=np.full((E, 2 * I, H // 64), s, np.uint16),
        b_gate_up=np.full((E, 2 * I, H // 64), b, np.uint16),
        q_down=qd, s_down=np.full((E, H, I // 64), s, np.uint16),
        b_down=np.full((E, H, I // 64), b, np.uint16),
        sh_q_gate_up=qgu[:1].copy(), sh_s_gate_up=np.full((1, 2 * I, H // 64), s, np.uint16),
        sh_b_gate_up=np.full((1, 2 * I, H // 64), b, np.uint16),
        sh_q_down=np.full((1, H, I // 8), word(9), np.uint32),
        sh_s_down=np.full((1, H, I // 64), s, np.uint16),
        sh_b_down=np.full((1, H, I // 64), b, np.uint16))
    return g, L


def test_hand_worked_one_token():
    g, L = _hand_layer()
    ex = g["expected"]
    ids, w32, w64 = oracle.route(L, g["shape"]["K"])
    assert ids[0].tolist() == ex["ids"]
    assert np.allclose(w64[0], ex["weights"], rtol=1e-15)
    h, d = oracle.expert_ffn(L.q_gate_up[15], L.s_gate_up[15], L.b_gate_up[15],
                             L.q_down[15], L.s_down[15], L.b_down[15], L.x)
    assert (synth.bf16_bits_to_f32(h) == ex["h"]).all()
    assert (d == ex["d"][0]).all()
    y, dsl = oracle.layer_tokens(L, ids, w64, want_slots=True)
    assert (dsl[0, 0] == ex["d"][0]).all() and (dsl[0, 1] == ex["d"][1]).all()
    assert (dsl[0, 2] == ex["d"][2]).all()
    assert (y == ex["y_bf16_bits"]).all()
    assert synth.bf16_bits_to_f32(y[0, 0]) == ex["y_bf16"]


# ------------------------------------------------------- dense brute force --
@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_oracle_layer_vs_dense_brute_force(seed):
    shape = synth.CONFIGS["tiny"].shape
    L = synth.gen_layer(16, shape, seed=seed, zipf_s=1.1 if seed == 3 else 0.0)
    ids, w32, w64 = oracle.route(L, shape.K)
    y = oracle.layer_tokens(L, ids, w64)
    yd, idd, wd, lg = dense.layer(L, shape.K)
    # ids agree wherever the K-th / K+1-th exact gap exceeds the fp32 bound
    srt = -np.sort(-lg, axis=1)
    gap = srt[:, shape.K - 1] - srt[:, shape.K]
    clear = gap > 1e-4
    assert clear.sum() >= 12
    assert (ids[clear] == idd[clear]).all()
    assert np.abs(w64[clear] - wd[clear]).max() < 1e-5
    yo = synth.bf16_bits_to_f32(y).astype(np.float64)[clear]
    yr = yd[clear]
    # the final bf16 rounding and h's bf16 rounding are the only gaps
    assert np.abs(yo - yr).max() <= 1e-2 * np.abs(yr).max() + 1e-3
    assert np.abs(yo - yr).sum() / np.abs(yr).sum() <= 2e-3


def test_oracle_detects_planted_mistakes():
    """A dropped shared term or a transposed down operand must break the
    dense comparison (the pin has teeth)."""
    shape = synth.CONFIGS["tiny"].shape
    L = synth.gen_layer(16, shape, seed=7)
    ids, w32, w64 = oracle.route(L, shape.K)
    yd, *_ = dense.layer(L, shape.K)
    y_ok = synth.bf16_bits_to_f32(oracle.layer_tokens(L, ids, w64)).astype(np.float64)
    L2 = synth.gen_layer(16, shape, seed=7)
    L2.sh_q_down = L2.sh_q_down * 0 + np.uint32(0x88888888)   # shared output -> 0
    y_bad = synth.bf16_bits_to_f32(oracle.layer_tokens(L2, ids, w64)).astype(np.float64)
    tol = 1e-2 * np.abs(yd).max() + 1e-3
    assert np.abs(y_ok - yd).max() <= tol
    assert np.abs(y_bad - yd).max() > tol
    # swapped slot weights
    y_sw = synth.bf16_bits_to_f32(oracle.layer_tokens(L, ids, w64[:, ::-1].copy())).astype(np.float64)
    assert np.abs(y_sw - yd).max() > tol


def test_rmsnorm_closed_form():
    H = 256
    y = np.zeros((2, H)); y[0, :] = 2.0; y[1, 0] = 3.0; y[1, 1] = 4.0
    out = synth.bf16_bits_to_f32(oracle.rmsnorm_rows(synth.bf16_bits(y))).astype(np.float64)
    assert np.allclose(out[0], 2.0 / math.sqrt(4.0 + 1e-6), rtol=2 ** -8)
    r = math.sqrt(25.0 / H + 1e-6)
    assert abs(out[1, 0] - 3 / r) <= 2 ** -8 * 3 / r and abs(out[1, 1] - 4 / r) <= 2 ** -8 * 4 / r
    assert (out[1, 2:] == 0).all()


# ----------------------------------------------------- the decoder block --
def test_rmsnorm_gain_constant_rows_return_the_gain():
    """h constant c (|c| >> 1e-3): h / rms(h) = sign(c) (1 - ~5e-7 / c^2),
    which rounds to 1, so each channel's output is its own gain exactly."""
    H = 256
    g = synth.gen_gain(H, seed=3)
    h = np.zeros((2, H)); h[0, :] = 2.0; h[1, :] = -0.75
    out = oracle.rmsnorm_gain_rows(synth.bf16_bits(h), g)
    assert np.array_equal(out[0], g)
    assert np.array_equal(out[1], g ^ np.uint16(0x8000))


def test_rmsnorm_gain_of_ones_is_the_unit_normalisation():
    h = synth.gen_tokens(3, 512, seed=4)
    ones = synth.bf16_bits(np.ones(512))
    assert np.array_equal(oracle.rmsnorm_gain_rows(h, ones), oracle.rmsnorm_rows(h))


def test_rmsnorm_gain_is_per_channel():
    """A one-hot gain keeps that channel of the unit normalisation alone; a
    gain of 2 doubles every output exactly (scaling by 2 is exact in bf16)."""
    H = 256
    h = synth.gen_tokens(2, H, seed=5)
    unit = synth.bf16_bits_to_f32(oracle.rmsnorm_rows(h))
    onehot = np.zeros(H); onehot[37] = 1.0
    out = synth.bf16_bits_to_f32(oracle.rmsnorm_gain_rows(h, synth.bf16_bits(onehot)))
    assert np.array_equal(out[:, 37], unit[:, 37])
    assert (np.delete(out, 37, axis=1) == 0).all()
    g = synth.gen_gain(H, seed=6)
    g2 = synth.bf16_bits(2.0 * synth.bf16_bits_to_f32(g))
    a = synth.bf16_bits_to_f32(oracle.rmsnorm_gain_rows(h, g))
    b = synth.bf16_bits_to_f32(oracle.rmsnorm_gain_rows(h, g2))
    assert np.array_equal(b, 2.0 * a)


def test_residual_add_ties_and_torch():
    """bf16 has spacing 2^-7 at 1.0 and 2^-6 at 3.0: a half-spacing addend
    is a tie (to the even neighbour), anything above it rounds away; a far
    smaller addend vanishes; and random pairs match torch's bf16 addition
    (fp32 sum, one rounding)."""
    one = 1.0
    cases = [(one, 2 ** -8, one), (one + 2 ** -7, 2 ** -8, one + 2 ** -6),
             (one, 2 ** -8 + 2 ** -15, one + 2 ** -7), (one, 2 ** -30, one),
             (1.5, -1.5, 0.0), (-3.0, 2 ** -7, -3.0),
             (-3.0, 2 ** -7 + 2 ** -14, -3.0 + 2 ** -6)]
    h = synth.bf16_bits(np.array([c[0] for c in cases]))
    y = synth.bf16_bits(np.array([c[1] for c in cases]))
    out = synth.bf16_bits_to_f32(oracle.residual_add(h, y)).astype(np.float64)
    assert np.array_equal(out, np.array([c[2] for c in cases]))
    rng = np.random.default_rng(7)
    a = synth.bf16_bits(rng.standard_normal(4096) * 10.0 ** rng.integers(-3, 3, 4096))
    b = synth.bf16_bits(rng.standard_normal(4096))
    ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    tb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    ref = (ta + tb).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.residual_add(a, b), ref)


def test_decoder_blocks_zero_layer_keeps_the_residual_stream():
    """A layer whose experts rebuild to zero (scale and bias 0) outputs y = 0,
    so the block returns its input unchanged, whatever the gain."""
    shape = synth.LayerShape(H=256, E=8, K=2, I=128, n_shared=1)
    L = synth.gen_layer(3, shape, seed=8)
    for name in ("s_down", "b_down", "sh_s_down", "sh_b_down"):
        getattr(L, name)[...] = 0
    h0 = synth.gen_tokens(3, 256, seed=9)
    h, ids = oracle.decoder_blocks([L], [synth.gen_gain(256, seed=10)], h0, 2)
    assert np.array_equal(h, h0)
    assert ids.shape == (3, 2)


# ------------------------------------------------- decode attention (GQA) --
def _dense_kv(k, v, table, L):
    """The cache as contiguous [n_kv][L][D] arrays (positions in order)."""
    B = k.shape[2]
    idx = [(table[j // B], j % B) for j in range(L)]
    kk = np.stack([k[p, :, r] for p, r in idx], axis=1)
    vv = np.stack([v[p, :, r] for p, r in idx], axis=1)
    return kk, vv


def test_attn_matches_torch_sdpa():
    """Against torch's scaled_dot_product_attention in float64 on the same
    numbers (contiguous K/V, each query head given its group's K/V, the
    causal window of each new token as an explicit mask)."""
    T, n_q, n_kv, D, L = 2, 16, 2, 64, 150
    q, k, v, table = synth.gen_attn(T, n_q, n_kv, D, L, seed=11)
    o = synth.bf16_bits_to_f32(oracle.attn_decode(q, k, v, table, L)).astype(np.float64)
    kk, vv = _dense_kv(k, v, table, L)
    qf = torch.from_numpy(synth.bf16_bits_to_f32(q).astype(np.float64)).permute(1, 0, 2)
    kf = torch.from_numpy(synth.bf16_bits_to_f32(kk).astype(np.float64))
    vf = torch.from_numpy(synth.bf16_bits_to_f32(vv).astype(np.float64))
    kf = kf.repeat_interleave(n_q // n_kv, dim=0)
    vf = vf.repeat_interleave(n_q // n_kv, dim=0)
    mask = torch.tensor([[j <= L - T + t for j in range(L)] for t in range(T)])
    ref = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, attn_mask=mask)
    ref = ref.permute(1, 0, 2).numpy()
    assert np.abs(o - ref).max() <= 2 ** -8 * np.abs(ref).max()
    assert np.abs(o - ref).mean() <= 2 ** -9 * np.abs(ref).mean()


def test_attn_closed_forms():
    """One position: o = v_0. Equal keys: o = the mean of the visible
    values. A dominant key: o = its value. Head h reads group h / 8."""
    T, n_q, n_kv, D = 1, 16, 2, 64
    q, k, v, table = synth.gen_attn(T, n_q, n_kv, D, 1, seed=12)
    o = oracle.attn_decode(q, k, v, table, 1)
    for h in range(n_q):
        assert np.array_equal(o[0, h], v[table[0], h // 8, 0])
    L = 100
    q, k, v, table = synth.gen_attn(T, n_q, n_kv, D, L, seed=13)
    k[...] = k[0:1, :, 0:1]  # every key equal within a head group
    o = synth.bf16_bits_to_f32(oracle.attn_decode(q, k, v, table, L)).astype(np.float64)
    _, vv = _dense_kv(k, v, table, L)
    mean = synth.bf16_bits_to_f32(vv).astype(np.float64).mean(axis=1)  # [n_kv][D]
    for h in range(n_q):
        assert np.abs(o[0, h] - mean[h // 8]).max() <= 2 ** -8 * np.abs(mean[h // 8]).max()
    q, k, v, table = synth.gen_attn(T, n_q, n_kv, D, L, seed=14)
    j = 37
    k[table[j // 64], 1, j % 64] = synth.bf16_bits(
        40.0 * synth.bf16_bits_to_f32(q[0, 8]))  # head 8's query, scaled up
    o = oracle.attn_decode(q, k, v, table, L)
    assert np.array_equal(o[0, 8], v[table[j // 64], 1, j % 64])
    v[:, 1] = 0  # group 1 silenced: heads 8..15 output zero, heads 0..7 do not
    o = synth.bf16_bits_to_f32(oracle.attn_decode(q, k, v, table, L))
    assert (o[0, 8:] == 0).all() and (np.abs(o[0, :8]) > 0).any()


def test_attn_causal_window_and_paging():
    """With two new tokens the first does not see the last position; moving
    the blocks to other physical slots changes nothing."""
    n_q, n_kv, D, L = 16, 2, 64, 130
    q, k, v, table = synth.gen_attn(2, n_q, n_kv, D, L, seed=15)
    o2 = oracle.attn_decode(q, k, v, table, L)
    o1 = oracle.attn_decode(q[:1], k, v, table, L - 1)
    assert np.array_equal(o2[0], o1[0])
    perm = np.random.default_rng(16).permutation(k.shape[0])
    k2 = np.empty_like(k); v2 = np.empty_like(v)
    k2[perm] = k; v2[perm] = v
    assert np.array_equal(oracle.attn_decode(q, k2, v2, perm[table], L), o2)
    with pytest.raises(ValueError):
        oracle.attn_decode(q, k, v, np.full_like(table, k.shape[0]), L)


# ------------------------------------------ Gated DeltaNet recurrence --
def test_gdn_pure_decay_and_exact_write():
    """beta = 0 leaves alpha-scaled states (o = the decayed state times q);
    alpha = beta = 1 with k a basis vector e_j replaces column j of the
    state by v and keeps the others (the delta rule's exact write)."""
    T, n_k, n_v, dk, dv = 3, 2, 4, 16, 8
    q, k, v, alpha, beta, s0 = synth.gen_gdn(T, n_k, n_v, dk, dv, seed=21)
    beta0 = np.zeros_like(beta)
    o, s1 = oracle.gdn_scan(q, k, v, alpha, beta0, s0)
    decay = np.prod(alpha.astype(np.float64), axis=0)  # [n_v]
    assert np.allclose(s1, s0 * decay[:, None, None], rtol=1e-6)
    qf = synth.bf16_bits_to_f32(q).astype(np.float64)
    exp_o = np.einsum("hij,hj->hi", s0 * decay[:, None, None], qf[-1][np.arange(n_v) // 2])
    got = synth.bf16_bits_to_f32(o[-1]).astype(np.float64)
    assert np.abs(got - exp_o).max() <= 2 ** -8 * np.abs(exp_o).max()
    j = 5
    kb = np.zeros((1, n_k, dk)); kb[..., j] = 1.0
    ones = np.ones((1, n_v), np.float32)
    _, s2 = oracle.gdn_scan(q[:1], synth.bf16_bits(kb), v[:1], ones, ones, s0)
    vf = synth.bf16_bits_to_f32(v[0]).astype(np.float32)
    assert np.array_equal(s2[:, :, j], vf)
    keep = [c for c in range(dk) if c != j]
    assert np.array_equal(s2[:, :, keep], s0[:, :, keep])


def test_gdn_matches_the_matrix_form_in_torch():
    """The recurrence as matrices in torch float64, S (alpha (I - beta k k^T))
    + beta v k^T, token by token, with each value head reading key head
    h // (n_v / n_k)."""
    T, n_k, n_v, dk, dv = 5, 2, 4, 16, 12
    q, k, v, alpha, beta, s0 = synth.gen_gdn(T, n_k, n_v, dk, dv, seed=22)
    o, s_end = oracle.gdn_scan(q, k, v, alpha, beta, s0)
    S = torch.from_numpy(s0.astype(np.float64))
    qf = torch.from_numpy(synth.bf16_bits_to_f32(q).astype(np.float64))
    kf = torch.from_numpy(synth.bf16_bits_to_f32(k).astype(np.float64))
    vf = torch.from_numpy(synth.bf16_bits_to_f32(v).astype(np.float64))
    eye = torch.eye(dk, dtype=torch.float64)
    for t in range(T):
        for h in range(n_v):
            kk = kf[t, h // 2]
            a, b = float(alpha[t, h]), float(beta[t, h])
            S[h] = S[h] @ (a * (eye - b * torch.outer(kk, kk))) + b * torch.outer(vf[t, h], kk)
        ref = torch.einsum("hij,hj->hi", S, qf[t][torch.arange(n_v) // 2]).numpy()
        got = synth.bf16_bits_to_f32(o[t]).astype(np.float64)
        assert np.abs(got - ref).max() <= 2 ** -8 * np.abs(ref).max()
    assert np.allclose(s_end, S.numpy(), rtol=1e-5, atol=1e-6)


# --------------------------------------- Gated DeltaNet, chunked form --
@pytest.mark.parametrize("C", [1, 16, 64, 24])
def test_gdn_chunked_equals_the_recurrence(C):
    """The chunked (WY / UT) form of the gated delta rule against the
    token-by-token recurrence (itself pinned above to closed forms and to
    the matrix form in torch): in fp64 the state after every chunk and
    every output agree to rounding, for chunk sizes 1, 16, 64 and 24 (a
    ragged last chunk of 16)."""
    T, n_k, n_v, dk, dv = 64, 2, 4, 32, 16
    q, k, v, alpha, beta, s0 = synth.gen_gdn(T, n_k, n_v, dk, dv, seed=31)
    o_c, s_c, o64_c, sc = oracle.gdn_chunked(q, k, v, alpha, beta, s0, C)
    o64_r, s64_r = oracle.gdn_scan64(q, k, v, alpha, beta, s0)
    scale = np.abs(o64_r).max()
    assert np.abs(o64_c - o64_r).max() <= 1e-11 * scale
    for c in range(sc.shape[0]):
        t_end = min((c + 1) * C, T)
        _, s_pref = oracle.gdn_scan64(q[:t_end], k[:t_end], v[:t_end], alpha[:t_end],
                                      beta[:t_end], s0)
        assert np.abs(sc[c] - s_pref).max() <= 1e-11 * np.abs(s_pref).max(), c
    assert np.abs(s_c.astype(np.float64) - s64_r).max() <= 1e-6 * np.abs(s64_r).max()
    o_r, _ = oracle.gdn_scan(q, k, v, alpha, beta, s0)
    # the bf16 outputs may differ only where the fp64 values straddle a rounding boundary
    assert np.mean(o_c != o_r) < 1e-3


def test_gdn_chunked_special_cases():
    """beta = 0: no write, each chunk only decays the state (the triangular
    system is the identity); one chunk holding the whole sequence equals the
    recurrence too; a planted mistake in the decay (alpha squared) is
    caught."""
    T, n_k, n_v, dk, dv = 20, 1, 2, 16, 8
    q, k, v, alpha, beta, s0 = synth.gen_gdn(T, n_k, n_v, dk, dv, seed=32)
    _, _, _, sc = oracle.gdn_chunked(q, k, v, alpha, np.zeros_like(beta), s0, 8)
    decay = np.cumprod(alpha.astype(np.float64), axis=0)
    for c, t_end in enumerate((8, 16, 20)):
        assert np.allclose(sc[c], s0 * decay[t_end - 1][:, None, None], rtol=1e-12)
    _, _, o64_whole, _ = oracle.gdn_chunked(q, k, v, alpha, beta, s0, T)
    o64_r, _ = oracle.gdn_scan64(q, k, v, alpha, beta, s0)
    assert np.abs(o64_whole - o64_r).max() <= 1e-11 * np.abs(o64_r).max()
    _, _, o64_bad, _ = oracle.gdn_chunked(q, k, v, alpha * alpha, beta, s0, 8)
    assert np.abs(o64_bad - o64_r).max() > 1e-3 * np.abs(o64_r).max()
