"""W4A16 Mixture-of-Experts expert layer for GB300 (sm_103a).

Thin Python binding of the C ABI in include/moe_w4.h. Every function here
only marshals arguments (device pointers from torch tensors, the current
CUDA stream) and raises MoeError on a non-zero status; all arithmetic runs
in the CUDA kernels of libmoe_w4.so. There is no CPU fallback: if the
library has not been built, load() raises.

Names follow the C ABI: moe_route, moe_plan, moe_expert_ffn_w4,
moe_combine, moe_layer_w4, moe_workspace_bytes, moe_max_blocks,
moe_workspace_init, moe_query_device_status, moe_debug_dequant_w4,
moe_debug_dequant_w4_decode.
"""
import ctypes as C
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe_w4.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_BAD_INPUT = 5
MOE_ERR_TIMEOUT = 6

EXPORTS = ("moe_workspace_bytes", "moe_max_blocks", "moe_workspace_init", "moe_route",
           "moe_plan", "moe_expert_ffn_w4", "moe_combine", "moe_layer_w4",
           "moe_query_device_status", "moe_debug_dequant_w4", "moe_debug_dequant_w4_decode",
           "moe_status_string",
           "moe_last_error", "moe_plan_noalloc", "moe_layer_path", "moe_decode_layers",
           "moe_decoder_blocks", "moe_attn_workspace_bytes", "moe_attn_decode",
           "moe_gdn_scan", "moe_gdn_chunked_workspace_bytes", "moe_gdn_chunked_scan")


class MoeError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        lib = _lib
        text = lib.moe_status_string(status).decode() if lib else str(status)
        detail = lib.moe_last_error().decode() if lib else ""
        super().__init__("%s: %s (%d)%s" % (where, text, status, (" - " + detail) if detail else ""))


class Shape(C.Structure):
    _fields_ = [("T", C.c_int32), ("H", C.c_int32), ("E", C.c_int32), ("K", C.c_int32),
                ("I", C.c_int32), ("n_shared", C.c_int32), ("tile_rows", C.c_int32)]

    def __repr__(self):
        return "Shape(T=%d, H=%d, E=%d, K=%d, I=%d, n_shared=%d, tile_rows=%d)" % (
            self.T, self.H, self.E, self.K, self.I, self.n_shared, self.tile_rows)


class AttnShape(C.Structure):
    _fields_ = [("T", C.c_int32), ("n_q", C.c_int32), ("n_kv", C.c_int32), ("D", C.c_int32),
                ("L", C.c_int32), ("block", C.c_int32)]


class GdnShape(C.Structure):
    _fields_ = [("T", C.c_int32), ("n_k", C.c_int32), ("n_v", C.c_int32), ("dk", C.c_int32),
                ("dv", C.c_int32)]


class W4Weights(C.Structure):
    _fields_ = [("q_gate_up", C.c_void_p), ("s_gate_up", C.c_void_p), ("b_gate_up", C.c_void_p),
                ("q_down", C.c_void_p), ("s_down", C.c_void_p), ("b_down", C.c_void_p)]


class LayerWeights(C.Structure):
    _fields_ = [("w_router", C.c_void_p), ("router_bias", C.c_void_p),
                ("experts", W4Weights), ("shared", W4Weights)]


class PlanPtrs(C.Structure):
    _fields_ = [("counts", C.c_void_p), ("offsets", C.c_void_p), ("sorted_rows", C.c_void_p),
                ("row_pos", C.c_void_p), ("block_map", C.c_void_p), ("num_blocks", C.c_void_p)]


_lib = None
_lock = threading.Lock()


def load():
    """Load libmoe_w4.so (built by __graft_entry__.build()); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise FileNotFoundError(
                    "libmoe_w4.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
            L = C.CDLL(LIB_PATH)
            P, I32, SZ = C.c_void_p, C.c_int32, C.c_size_t
            pS, pW, pP = C.POINTER(Shape), C.POINTER(W4Weights), C.POINTER(PlanPtrs)
            L.moe_workspace_bytes.restype = SZ
            L.moe_workspace_bytes.argtypes = [pS]
            L.moe_max_blocks.restype = I32
            L.moe_max_blocks.argtypes = [pS]
            L.moe_layer_path.restype = I32
            L.moe_layer_path.argtypes = [pS]
            L.moe_gdn_chunked_workspace_bytes.restype = SZ
            L.moe_gdn_chunked_workspace_bytes.argtypes = [C.POINTER(GdnShape)]
            L.moe_attn_workspace_bytes.restype = SZ
            L.moe_attn_workspace_bytes.argtypes = [C.POINTER(AttnShape)]
            for name, args in (
                    ("moe_workspace_init", [P, SZ, P]),
                    ("moe_route", [pS, P, P, P, P, P, P, SZ, P]),
                    ("moe_plan", [pS, P, pP, P, SZ, P]),
                    ("moe_expert_ffn_w4", [pS, P, pW, pW, pP, P, P, SZ, P]),
                    ("moe_combine", [pS, P, P, P, P, P, P]),
                    ("moe_layer_w4", [pS, P, P, P, pW, pW, P, P, P, P, P, SZ, P]),
                    ("moe_query_device_status", [P, SZ, P]),
                    ("moe_debug_dequant_w4", [P, P, P, P, I32, I32, P]),
                    ("moe_debug_dequant_w4_decode", [P, P, P, P, I32, I32, P]),
                    ("moe_plan_noalloc", [pS, P, pP, P]),
                    ("moe_decode_layers", [pS, I32, P, P, P, P, P, SZ, P]),
                    ("moe_decoder_blocks", [pS, I32, P, P, P, P, P, I32, P, P, SZ, P]),
                    ("moe_attn_decode", [C.POINTER(AttnShape), P, P, P, P, I32, P, P, SZ, P]),
                    ("moe_gdn_scan", [C.POINTER(GdnShape), P, P, P, P, P, P, P, P, P]),
                    ("moe_gdn_chunked_scan",
                     [C.POINTER(GdnShape), P, P, P, P, P, P, P, P, P, SZ, P])):
                f = getattr(L, name)
                f.restype = C.c_int
                f.argtypes = args
            L.moe_status_string.restype = C.c_char_p
            L.moe_status_string.argtypes = [C.c_int]
            L.moe_last_error.restype = C.c_char_p
            L.moe_last_error.argtypes = []
            _lib = L
    return _lib


def _check(status, where):
    if status != MOE_OK:
        raise MoeError(status, where)


def _p(t):
    """Device pointer of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return C.c_void_p(t.data_ptr())


def _s(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def make_shape(T, H, E, K, I, n_shared=1, tile_rows=128):
    return Shape(T, H, E, K, I, n_shared, tile_rows)


def moe_workspace_bytes(shape):
    return load().moe_workspace_bytes(C.byref(shape))


def moe_max_blocks(shape):
    return load().moe_max_blocks(C.byref(shape))


def moe_layer_path(shape):
    """1: moe_layer_w4 runs the fused decode kernels; 0: the four calls; -1: bad shape."""
    return load().moe_layer_path(C.byref(shape))


def moe_workspace_init(ws, stream=None):
    _check(load().moe_workspace_init(_p(ws), ws.numel() * ws.element_size(), _s(stream)),
           "moe_workspace_init")


def moe_route(shape, x, w_router, router_bias, topk_ids, topk_w, ws, stream=None):
    _check(load().moe_route(C.byref(shape), _p(x), _p(w_router), _p(router_bias), _p(topk_ids),
                            _p(topk_w), _p(ws), ws.numel(), _s(stream)), "moe_route")


def moe_plan(shape, topk_ids, plan, ws, stream=None):
    _check(load().moe_plan(C.byref(shape), _p(topk_ids), C.byref(plan.ptrs), _p(ws), ws.numel(),
                           _s(stream)), "moe_plan")


def moe_expert_ffn_w4(shape, x, experts, shared, plan, y_slots, ws, stream=None):
    _check(load().moe_expert_ffn_w4(C.byref(shape), _p(x), C.byref(experts.ptrs),
                                    C.byref(shared.ptrs) if shared is not None else None,
                                    C.byref(plan.ptrs), _p(y_slots), _p(ws), ws.numel(),
                                    _s(stream)), "moe_expert_ffn_w4")


def moe_plan_noalloc(shape, topk_ids, plan, stream=None):
    """moe_plan without a workspace (static device scratch; see moe_w4.h)."""
    _check(load().moe_plan_noalloc(C.byref(shape), _p(topk_ids), C.byref(plan.ptrs), _s(stream)),
           "moe_plan_noalloc")


def moe_combine(shape, y_slots, row_pos, topk_w, y, x_next=None, stream=None):
    _check(load().moe_combine(C.byref(shape), _p(y_slots), _p(row_pos), _p(topk_w), _p(y),
                              _p(x_next), _s(stream)), "moe_combine")


def decode_layer_table(layers):
    """Host array of moe_layer_weights_t from (w_router, router_bias or None,
    experts, shared or None) tuples; keep it alive while it is used."""
    arr = (LayerWeights * len(layers))()
    for i, (wr, bias, ex, sh) in enumerate(layers):
        arr[i].w_router = _p(wr)
        arr[i].router_bias = _p(bias)
        arr[i].experts = ex.ptrs
        if sh is not None:
            arr[i].shared = sh.ptrs
    return arr


def moe_decode_layers(shape, layer_table, x, y, ws, x_next=None, stream=None):
    """n stacked decode layers (layer_table from decode_layer_table)."""
    _check(load().moe_decode_layers(C.byref(shape), len(layer_table),
                                    C.cast(layer_table, C.c_void_p), _p(x), _p(y), _p(x_next),
                                    _p(ws), ws.numel(), _s(stream)), "moe_decode_layers")


def make_attn_shape(T, n_q, n_kv, D, L, block=64):
    return AttnShape(T, n_q, n_kv, D, L, block)


def alloc_attn_workspace(shape, device="cuda", stream=None):
    n = load().moe_attn_workspace_bytes(C.byref(shape))
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED_SHAPE, "alloc_attn_workspace")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws


def moe_attn_decode(shape, q, k_cache, v_cache, table, o, ws, stream=None):
    """Grouped-query decode attention over a block-paged key/value cache."""
    _check(load().moe_attn_decode(C.byref(shape), _p(q), _p(k_cache), _p(v_cache), _p(table),
                                  k_cache.shape[0], _p(o), _p(ws), ws.numel(), _s(stream)),
           "moe_attn_decode")


def make_gdn_shape(T, n_k, n_v, dk, dv):
    return GdnShape(T, n_k, n_v, dk, dv)


def moe_gdn_scan(shape, q, k, v, alpha, beta, state_in, state_out, o, stream=None):
    """Gated delta rule over shape.T tokens (state_out may be state_in)."""
    _check(load().moe_gdn_scan(C.byref(shape), _p(q), _p(k), _p(v), _p(alpha), _p(beta),
                               _p(state_in), _p(state_out), _p(o), _s(stream)), "moe_gdn_scan")


def alloc_gdn_workspace(shape, device):
    """Device workspace of the chunked scan (moe_gdn_chunked_workspace_bytes),
    zero-filled: its status header must start at zero."""
    nbytes = load().moe_gdn_chunked_workspace_bytes(C.byref(shape))
    if nbytes == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED_SHAPE, "moe_gdn_chunked_workspace_bytes")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def moe_gdn_chunked_scan(shape, q, k, v, alpha, beta, state_in, state_out, o, ws, stream=None):
    """Chunked (parallel) form of the gated delta rule; same results as
    moe_gdn_scan within fp32 rounding (state_out may be state_in)."""
    _check(load().moe_gdn_chunked_scan(C.byref(shape), _p(q), _p(k), _p(v), _p(alpha), _p(beta),
                                       _p(state_in), _p(state_out), _p(o), _p(ws),
                                       ws.numel() * ws.element_size(), _s(stream)),
           "moe_gdn_chunked_scan")


def gain_table(gains):
    """Host array of device pointers to per-layer bf16 [H] gains; keep it
    alive while it is used."""
    arr = (C.c_void_p * len(gains))()
    for i, g in enumerate(gains):
        arr[i] = _p(g)
    return arr


def moe_decoder_blocks(shape, layer_table, gains, h_out, ws, h_in=None, token_ids=None,
                     embed=None, stream=None):
    """n decoder blocks (pre-norm with gain, MoE layer, residual add); h_0 is
    h_in, or the rows of embed named by the device token ids."""
    if len(gains) != len(layer_table):
        raise ValueError("one gain table entry per layer")
    vocab = embed.shape[0] if embed is not None else 0
    _check(load().moe_decoder_blocks(C.byref(shape), len(layer_table),
                                   C.cast(layer_table, C.c_void_p), C.cast(gains, C.c_void_p),
                                   _p(h_in), _p(token_ids), _p(embed), vocab, _p(h_out),
                                   _p(ws), ws.numel(), _s(stream)), "moe_decoder_blocks")


def moe_layer_w4(shape, x, w_router, router_bias, experts, shared, y, ws, x_next=None,
                 topk_ids=None, topk_w=None, stream=None):
    _check(load().moe_layer_w4(C.byref(shape), _p(x), _p(w_router), _p(router_bias),
                               C.byref(experts.ptrs),
                               C.byref(shared.ptrs) if shared is not None else None,
                               _p(y), _p(x_next), _p(topk_ids), _p(topk_w), _p(ws), ws.numel(),
                               _s(stream)), "moe_layer_w4")


def moe_query_device_status(ws, stream=None):
    """Synchronises the stream; returns the device status code (and clears it)."""
    return load().moe_query_device_status(_p(ws), ws.numel(), _s(stream))


def moe_debug_dequant_w4(q, s, b, out, stream=None):
    N, K8 = q.shape
    _check(load().moe_debug_dequant_w4(_p(q), _p(s), _p(b), _p(out), N, K8 * 8, _s(stream)),
           "moe_debug_dequant_w4")


def moe_debug_dequant_w4_decode(q, s, b, out, stream=None):
    N, K8 = q.shape
    _check(load().moe_debug_dequant_w4_decode(_p(q), _p(s), _p(b), _p(out), N, K8 * 8,
                                              _s(stream)),
           "moe_debug_dequant_w4_decode")


# ----------------------------------------------------- device-side holders --
class ExpertWeights:
    """Packed 4-bit weights of n experts resident on the device (layouts of
    moe_w4_weights_t); bf16 arrays are kept as int16 storage."""

    def __init__(self, q_gate_up, s_gate_up, b_gate_up, q_down, s_down, b_down):
        self.tensors = (q_gate_up, s_gate_up, b_gate_up, q_down, s_down, b_down)
        for t in self.tensors:
            if not (t.is_cuda and t.is_contiguous()):
                raise ValueError("expert weights must be contiguous CUDA tensors")
        self.ptrs = W4Weights(*[t.data_ptr() for t in self.tensors])

    @classmethod
    def from_numpy(cls, q_gate_up, s_gate_up, b_gate_up, q_down, s_down, b_down, device="cuda"):
        def dev(a):
            a = a.view("int32") if a.dtype.itemsize == 4 else a.view("int16")
            return torch.from_numpy(a.copy()).to(device)
        return cls(*[dev(a) for a in (q_gate_up, s_gate_up, b_gate_up, q_down, s_down, b_down)])

    @property
    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in self.tensors)


class PlanBuffers:
    """Caller-owned plan buffers (moe_plan_t) for one shape."""

    def __init__(self, shape, device="cuda"):
        R = shape.T * shape.K
        mb = moe_max_blocks(shape)
        z = lambda n: torch.zeros(n, dtype=torch.int32, device=device)  # noqa: E731
        self.counts = z(shape.E)
        self.offsets = z(shape.E + 1)
        self.sorted_rows = z(R)
        self.row_pos = z(R)
        self.block_map = z(mb * 3)
        self.num_blocks = z(1)
        self.ptrs = PlanPtrs(*[t.data_ptr() for t in (self.counts, self.offsets, self.sorted_rows,
                                                      self.row_pos, self.block_map,
                                                      self.num_blocks)])


def alloc_workspace(shape, device="cuda", stream=None):
    n = moe_workspace_bytes(shape)
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED_SHAPE, "alloc_workspace")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws
