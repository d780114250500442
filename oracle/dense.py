"""Brute-force dense reference of the MoE layer (numpy fp64), for tiny shapes.

TEST INFRASTRUCTURE; independent of both the C oracle and the CUDA path.
Every expert is evaluated on every token, then masked by the top-K
selection and weighted:
    y_t = sum_e [e in top_K(t)] * w_{t,e} * FFN_e(x_t) + FFN_shared(x_t)
No plan, scatter or permutation is involved. Routing here uses exact fp64
logits (x @ W_r^T); callers compare ids only where the K-th/K+1-th logit gap
exceeds the fp32 rounding bound.
"""
import numpy as np


def _bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _round_bf16(v):
    """fp64 -> nearest-even bf16 value (as fp64), via frexp on the exact value."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(np.abs(v))
    ue = np.maximum(e - 8, -133)
    q = np.rint(np.ldexp(np.abs(v), -ue))  # np.rint: round half to even
    return np.sign(v) * np.ldexp(q, ue)


def unpack(qw):
    """uint32 [N, K/8] -> int [N, K], nibble i of word w is element 8w+i."""
    qw = np.asarray(qw, np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    nib = (qw[..., None] >> shifts) & np.uint32(15)
    return nib.reshape(qw.shape[:-1] + (qw.shape[-1] * 8,)).astype(np.int64)


def dequant(qw, s, b):
    q = unpack(qw).astype(np.float64)
    sv = np.repeat(_bits_to_f64(s), 64, axis=-1)
    bv = np.repeat(_bits_to_f64(b), 64, axis=-1)
    return _round_bf16(sv * q + bv)


def expert(qgu, sgu, bgu, qd, sd, bd, x):
    wgu = dequant(qgu, sgu, bgu)
    wd = dequant(qd, sd, bd)
    I = wd.shape[1]
    g = x @ wgu[:I].T
    u = x @ wgu[I:].T
    h = _round_bf16(g / (1.0 + np.exp(-g)) * u)
    return h @ wd.T


def exact_logits(L):
    x = _bits_to_f64(L.x)
    w = _bits_to_f64(L.w_router)
    lg = x @ w.T
    if L.router_bias is not None:
        lg = lg + np.asarray(L.router_bias, np.float64)
    return lg


def layer(L, K):
    """Returns (y_exact fp64 [T,H] before the final bf16 rounding, ids, w)."""
    x = _bits_to_f64(L.x)
    lg = exact_logits(L)
    T, E = lg.shape
    order = np.lexsort((np.arange(E)[None, :].repeat(T, 0), -lg), axis=1)
    ids = order[:, :K]
    sel = np.take_along_axis(lg, ids, 1)
    w = np.exp(sel - sel[:, :1])
    w = w / w.sum(1, keepdims=True)
    y = np.zeros_like(x)
    for e in range(E):
        fe = expert(L.q_gate_up[e], L.s_gate_up[e], L.b_gate_up[e],
                    L.q_down[e], L.s_down[e], L.b_down[e], x)
        mask = (ids == e)
        we = (w * mask).sum(1)
        y += we[:, None] * fe
    for j in range(L.sh_q_gate_up.shape[0]):
        y += expert(L.sh_q_gate_up[j], L.sh_s_gate_up[j], L.sh_b_gate_up[j],
                    L.sh_q_down[j], L.sh_s_down[j], L.sh_b_down[j], x)
    return y, ids, w, lg
