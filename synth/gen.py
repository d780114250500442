"""Seeded generators (numpy PCG64) for the MoE layer inputs.

Draw order for one layer with seed s (rng = default_rng(s)):
  x       [T, H]   ~ N(0, 1)                       -> bf16 (round to nearest even)
  W_r     [E, H]   ~ N(0, 1/H)                     -> bf16
  then for each routed expert e = 0..E-1, then each shared expert:
    q_gate_up [2I, H/8]  uint32 words, every nibble independent U{0..15}
    s_gate_up [2I, H/64] ~ U[0.002, 0.02]          -> bf16
    q_down    [H, I/8]   uint32 words
    s_down    [H, I/64]  ~ U[0.002, 0.02]          -> bf16
  the bias of every group is -8*scale (exact in bf16: a power-of-two multiple).

Drawing a uint32 uniformly over [0, 2^32) is the same distribution as
drawing its eight nibbles independently from U{0..15} and packing them
low nibble first, so the words are drawn directly.

Tokens for a later step or chunk come from gen_tokens(seed) alone.
All bf16 tensors are returned as their raw uint16 bit patterns.
"""
from dataclasses import dataclass

import numpy as np


def bf16_bits(a) -> np.ndarray:
    """float32/float64 array -> uint16 bf16 bit patterns, round to nearest even.

    Used only to encode synthetic draws as bf16 inputs."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return r


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(np.asarray(b, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def zipf_router_bias(E: int, s: float) -> np.ndarray:
    """Per-expert router-logit shift of a Zipf(s) law: -s*ln(rank), rank = e+1."""
    return (-s * np.log(np.arange(1, E + 1, dtype=np.float64))).astype(np.float32)


@dataclass
class LayerInputs:
    x: np.ndarray          # uint16 [T, H]
    w_router: np.ndarray   # uint16 [E, H]
    router_bias: object    # float32 [E] or None
    q_gate_up: np.ndarray  # uint32 [E, 2I, H/8]
    s_gate_up: np.ndarray  # uint16 [E, 2I, H/64]
    b_gate_up: np.ndarray  # uint16 [E, 2I, H/64]
    q_down: np.ndarray     # uint32 [E, H, I/8]
    s_down: np.ndarray     # uint16 [E, H, I/64]
    b_down: np.ndarray     # uint16 [E, H, I/64]
    sh_q_gate_up: np.ndarray  # shared expert, same layouts with a leading dim n_shared
    sh_s_gate_up: np.ndarray
    sh_b_gate_up: np.ndarray
    sh_q_down: np.ndarray
    sh_s_down: np.ndarray
    sh_b_down: np.ndarray


def _scales(rng, shape):
    s = rng.uniform(0.002, 0.02, size=shape)
    sb = bf16_bits(s)
    # bias = -8 * scale: scale the bf16 value by 8 exactly (exponent + 3), negate
    b = bf16_bits(-8.0 * bf16_bits_to_f32(sb))
    return sb, b


def _expert(rng, H, I):
    qgu = rng.integers(0, 1 << 32, size=(2 * I, H // 8), dtype=np.uint64).astype(np.uint32)
    sgu, bgu = _scales(rng, (2 * I, H // 64))
    qd = rng.integers(0, 1 << 32, size=(H, I // 8), dtype=np.uint64).astype(np.uint32)
    sd, bd = _scales(rng, (H, I // 64))
    return qgu, sgu, bgu, qd, sd, bd


def gen_layer(T, shape, seed=0, zipf_s=0.0) -> LayerInputs:
    H, E, I = shape.H, shape.E, shape.I
    rng = np.random.default_rng(seed)
    x = bf16_bits(rng.standard_normal((T, H)))
    w_r = bf16_bits(rng.standard_normal((E, H)) * np.sqrt(1.0 / H))
    parts = [_expert(rng, H, I) for _ in range(E)]
    sh = [_expert(rng, H, I) for _ in range(shape.n_shared)]

    def stack(lst, i, dtype, tail):
        if not lst:
            return np.zeros((0,) + tail, dtype=dtype)
        return np.stack([p[i] for p in lst])

    bias = zipf_router_bias(E, zipf_s) if zipf_s > 0 else None
    tails = [(2 * I, H // 8), (2 * I, H // 64), (2 * I, H // 64),
             (H, I // 8), (H, I // 64), (H, I // 64)]
    dts = [np.uint32, np.uint16, np.uint16, np.uint32, np.uint16, np.uint16]
    r = [stack(parts, i, dts[i], tails[i]) for i in range(6)]
    s = [stack(sh, i, dts[i], tails[i]) for i in range(6)]
    return LayerInputs(x, w_r, bias, *r, *s)


def gen_tokens(T, H, seed) -> np.ndarray:
    """Hidden states alone (a later decode step or prompt chunk)."""
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.standard_normal((T, H)))


def gen_gain(H, seed) -> np.ndarray:
    """A learned RMSNorm gain: bf16 values 1 + 0.1 N(0, 1)."""
    rng = np.random.default_rng(seed)
    return bf16_bits(1.0 + 0.1 * rng.standard_normal(H))


def gen_embed(V, H, seed) -> np.ndarray:
    """A token embedding table: V rows of bf16 N(0, 1) values."""
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.standard_normal((V, H)))


def gen_attn(T, n_q, n_kv, D, L, B=64, seed=0, spare=3):
    """Decode-attention inputs: q [T][n_q][D], a key/value cache of
    ceil(L / B) + spare physical blocks [n_phys][n_kv][B][D] (bf16 N(0, 1)),
    and a block table mapping the logical blocks to a random permutation of
    them."""
    rng = np.random.default_rng(seed)
    nblk = (L + B - 1) // B
    n_phys = nblk + spare
    q = bf16_bits(rng.standard_normal((T, n_q, D)))
    k = bf16_bits(rng.standard_normal((n_phys, n_kv, B, D)))
    v = bf16_bits(rng.standard_normal((n_phys, n_kv, B, D)))
    table = rng.permutation(n_phys)[:nblk].astype(np.int32)
    return q, k, v, table


def gen_gdn(T, n_k, n_v, dk, dv, seed=0):
    """Gated-DeltaNet scan inputs: q, k unit vectors per head (bf16 of a
    normalised N(0, 1) draw), v ~ N(0, 1) bf16, decay alpha ~ U[0.9, 1),
    write strength beta ~ U[0, 1) (fp32), and a starting state
    ~ N(0, 0.1^2) fp32 [n_v][dv][dk]."""
    rng = np.random.default_rng(seed)

    def unit(shape):
        a = rng.standard_normal(shape)
        return bf16_bits(a / np.linalg.norm(a, axis=-1, keepdims=True))
    q = unit((T, n_k, dk))
    k = unit((T, n_k, dk))
    v = bf16_bits(rng.standard_normal((T, n_v, dv)))
    alpha = rng.uniform(0.9, 1.0, (T, n_v)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (T, n_v)).astype(np.float32)
    state = (0.1 * rng.standard_normal((n_v, dv, dk))).astype(np.float32)
    return q, k, v, alpha, beta, state
