"""CPU oracle of the W4A16 MoE expert layer (plain C, fp64) and an
independent brute-force dense reference (numpy, fp64).

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference legs may import this package. The CUDA path never
does, and shares no code with it.

The C library is compiled with gcc on first use (or by build()):
  gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp -shared -fPIC
"""
import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force=False):
    """Compile the oracle library (host gcc; x86 here, aarch64 on the GPU host)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off",
                               "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            i = C.c_int
            L.orc_bf16_value.restype = C.c_double
            L.orc_bf16_value.argtypes = [C.c_uint16]
            L.orc_bf16_rne.restype = C.c_uint16
            L.orc_bf16_rne.argtypes = [C.c_double]
            L.orc_router_logit.restype = C.c_float
            L.orc_router_logit.argtypes = [P, P, i]
            L.orc_router_logits.argtypes = [P, P, P, i, i, i, P]
            L.orc_topk.argtypes = [P, i, i, i, P, P, P]
            L.orc_plan.restype = i
            L.orc_plan.argtypes = [P, i, i, i, i, i, P, P, P, P, P, i]
            L.orc_dequant.argtypes = [P, P, P, i, i, P]
            L.orc_expert_ffn.argtypes = [P] * 6 + [i, i, P, i, P, P]
            L.orc_layer_tokens.argtypes = [P, i, i, i, i, P, P] + [P] * 12 + [P, i, P, P]
            L.orc_rmsnorm_rows.argtypes = [P, i, i, P]
            L.orc_rmsnorm_gain_rows.argtypes = [P, P, i, i, P]
            L.orc_gdn_scan.argtypes = [P, P, P, P, P, P, i, i, i, i, i, P, P]
            L.orc_gdn_scan64.argtypes = [P, P, P, P, P, P, i, i, i, i, i, P, P]
            L.orc_gdn_chunked.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, P, P, P, P]
            L.orc_attn_decode.restype = i
            L.orc_attn_decode.argtypes = [P, P, P, P, i, i, i, i, i, i, i, P]
            L.orc_residual_add.argtypes = [P, P, C.c_size_t, P]
            L.orc_num_threads.restype = i
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ---------------------------------------------------------------- wrappers --
def bf16_value(bits):
    return lib().orc_bf16_value(int(bits))


def bf16_rne(v):
    return lib().orc_bf16_rne(float(v))


def router_logits(x, w_r, bias=None):
    x = _c(x, np.uint16)
    w_r = _c(w_r, np.uint16)
    T, H = x.shape
    E = w_r.shape[0]
    out = np.empty((T, E), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    lib().orc_router_logits(_p(x), _p(w_r), _p(b), T, H, E, _p(out))
    return out


def topk(logits, K):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, K), np.int32)
    w32 = np.empty((T, K), np.float32)
    w64 = np.empty((T, K), np.float64)
    lib().orc_topk(_p(logits), T, E, K, _p(ids), _p(w32), _p(w64))
    return ids, w32, w64


def max_blocks(T, E, K, n_shared, BM):
    R = T * K
    return (R + BM - 1) // BM + min(E, R) + (((T + BM - 1) // BM) if n_shared else 0)


def plan(ids, E, n_shared, BM):
    ids = _c(ids, np.int32)
    T, K = ids.shape
    R = T * K
    mb = max_blocks(T, E, K, n_shared, BM)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    sorted_rows = np.empty(R, np.int32)
    row_pos = np.empty(R, np.int32)
    bmap = np.zeros((mb, 3), np.int32)
    nb = lib().orc_plan(_p(ids), T, E, K, n_shared, BM, _p(counts), _p(offsets),
                        _p(sorted_rows), _p(row_pos), _p(bmap), mb)
    if nb < 0:
        raise ValueError("oracle plan: expert id out of range or block map overflow")
    return dict(counts=counts, offsets=offsets, sorted_rows=sorted_rows,
                row_pos=row_pos, block_map=bmap[:nb].copy(), num_blocks=nb)


def dequant(q, s, b):
    q = _c(q, np.uint32)
    s = _c(s, np.uint16)
    b = _c(b, np.uint16)
    N, K8 = q.shape
    out = np.empty((N, K8 * 8), np.uint16)
    lib().orc_dequant(_p(q), _p(s), _p(b), N, K8 * 8, _p(out))
    return out


def expert_ffn(q_gu, s_gu, b_gu, q_d, s_d, b_d, x_rows):
    """One expert on bf16 rows -> (h bf16 bits [n, I], d fp64 [n, H])."""
    x_rows = _c(x_rows, np.uint16)
    n, H = x_rows.shape
    I = q_d.shape[1] * 8
    h = np.empty((n, I), np.uint16)
    d = np.empty((n, H), np.float64)
    arrs = [_c(q_gu, np.uint32), _c(s_gu, np.uint16), _c(b_gu, np.uint16),
            _c(q_d, np.uint32), _c(s_d, np.uint16), _c(b_d, np.uint16)]
    lib().orc_expert_ffn(*[_p(a) for a in arrs], H, I, _p(x_rows), n, _p(h), _p(d))
    return h, d


def layer_tokens(L, ids, w64, tokens=None, x=None, want_slots=False):
    """Layer output y (bf16 bits) for a subset of tokens (default: all).

    L: synth.LayerInputs (weights); x overrides L.x (teacher-forced input)."""
    x = _c(L.x if x is None else x, np.uint16)
    T, H = x.shape
    E, K = L.q_gate_up.shape[0], ids.shape[1]
    I = L.q_down.shape[2] * 8
    tok = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    y = np.empty((len(tok), H), np.uint16)
    dsl = np.empty((len(tok), K + 1, H), np.float64) if want_slots else None
    has_sh = L.sh_q_gate_up.shape[0] > 0
    w = [_c(a, np.uint32 if a.dtype == np.uint32 else np.uint16) for a in
         (L.q_gate_up, L.s_gate_up, L.b_gate_up, L.q_down, L.s_down, L.b_down)]
    sh = [(_c(a[0], a.dtype) if has_sh else None) for a in
          (L.sh_q_gate_up, L.sh_s_gate_up, L.sh_b_gate_up, L.sh_q_down, L.sh_s_down,
           L.sh_b_down)]
    ids = _c(ids, np.int32)
    w64 = _c(w64, np.float64)
    lib().orc_layer_tokens(_p(x), H, E, K, I, _p(ids), _p(w64),
                           *[_p(a) for a in w], *[_p(a) for a in sh],
                           _p(tok), len(tok), _p(y), _p(dsl))
    return (y, dsl) if want_slots else y


def rmsnorm_rows(y):
    y = _c(y, np.uint16)
    T, H = y.shape
    out = np.empty_like(y)
    lib().orc_rmsnorm_rows(_p(y), T, H, _p(out))
    return out


def rmsnorm_gain_rows(h, g):
    """Pre-norm of the decoder block: bf16(g * h / sqrt(mean(h^2) + 1e-6))."""
    h = _c(h, np.uint16)
    g = _c(g, np.uint16)
    T, H = h.shape
    out = np.empty_like(h)
    lib().orc_rmsnorm_gain_rows(_p(h), _p(g), T, H, _p(out))
    return out


def residual_add(h, y):
    """The block's residual add: bf16(h + y), one rounding."""
    h = _c(h, np.uint16)
    y = _c(y, np.uint16)
    out = np.empty_like(h)
    lib().orc_residual_add(_p(h), _p(y), C.c_size_t(h.size), _p(out))
    return out


def decoder_blocks(Ls, gains, h0, K):
    """Stacked decoder blocks: for each layer x = rmsnorm_gain_rows(h, g),
    y = the MoE layer on x (router, top-K, experts, combine), h = h + y.
    Returns the last h and the last layer's ids."""
    h = _c(h0, np.uint16)
    ids = None
    for L, g in zip(Ls, gains):
        x = rmsnorm_gain_rows(h, g)
        ids, _, w64 = topk(router_logits(x, L.w_router, L.router_bias), K)
        h = residual_add(h, layer_tokens(L, ids, w64, x=x))
    return h, ids


def attn_decode(q, k_cache, v_cache, table, L):
    """Grouped-query decode attention over a block-paged key/value cache.

    q [T][n_q][D]; k_cache, v_cache [n_phys][n_kv][B][D] (bf16 bits);
    table [ceil(L / B)] physical block of each logical block. Query token t
    is at position L - T + t. Returns o [T][n_q][D] (bf16 bits)."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    table = _c(table, np.int32)
    T, n_q, D = q.shape
    n_phys, n_kv, B, _ = k_cache.shape
    o = np.empty_like(q)
    if lib().orc_attn_decode(_p(q), _p(k_cache), _p(v_cache), _p(table), n_phys, T, n_q, n_kv,
                             D, int(L), B, _p(o)) != 0:
        raise ValueError("oracle attention: block table entry out of range")
    return o


def gdn_scan(q, k, v, alpha, beta, state):
    """Gated delta rule over T tokens: returns (o [T][n_v][dv] bf16 bits,
    the final state [n_v][dv][dk] fp32). q, k [T][n_k][dk], v [T][n_v][dv]
    bf16 bits; alpha, beta [T][n_v] fp32; state [n_v][dv][dk] fp32."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    alpha = _c(alpha, np.float32)
    beta = _c(beta, np.float32)
    state = _c(state, np.float32)
    T, n_k, dk = q.shape
    n_v, dv = v.shape[1], v.shape[2]
    o = np.empty((T, n_v, dv), np.uint16)
    s_out = np.empty_like(state)
    lib().orc_gdn_scan(_p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(state), T, n_k, n_v, dk, dv,
                       _p(s_out), _p(o))
    return o, s_out


def gdn_scan64(q, k, v, alpha, beta, state):
    """The recurrence of gdn_scan with its results in fp64: (o [T][n_v][dv]
    before the bf16 rounding, the final state [n_v][dv][dk])."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    alpha = _c(alpha, np.float32)
    beta = _c(beta, np.float32)
    state = _c(state, np.float32)
    T, n_k, dk = q.shape
    n_v, dv = v.shape[1], v.shape[2]
    o64 = np.empty((T, n_v, dv), np.float64)
    s64 = np.empty((n_v, dv, dk), np.float64)
    lib().orc_gdn_scan64(_p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(state), T, n_k, n_v, dk,
                         dv, _p(s64), _p(o64))
    return o64, s64


def gdn_chunked(q, k, v, alpha, beta, state, C):
    """The gated delta rule in chunks of C tokens (the chunked form written
    out in orc_gdn_chunked): returns (o bf16 bits, final state fp32, o in
    fp64, the fp64 state after every chunk [n_chunks][n_v][dv][dk])."""
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    alpha = _c(alpha, np.float32)
    beta = _c(beta, np.float32)
    state = _c(state, np.float32)
    T, n_k, dk = q.shape
    n_v, dv = v.shape[1], v.shape[2]
    nc = (T + C - 1) // C
    o = np.empty((T, n_v, dv), np.uint16)
    s_out = np.empty_like(state)
    o64 = np.empty((T, n_v, dv), np.float64)
    sc = np.empty((nc, n_v, dv, dk), np.float64)
    lib().orc_gdn_chunked(_p(q), _p(k), _p(v), _p(alpha), _p(beta), _p(state), T, n_k, n_v, dk,
                          dv, C, _p(s_out), _p(o), _p(o64), _p(sc))
    return o, s_out, o64, sc


def route(L, K):
    """Logits -> (ids, w32, w64) for all tokens of L."""
    lg = router_logits(L.x, L.w_router, L.router_bias)
    return topk(lg, K)


def num_threads():
    return lib().orc_num_threads()
