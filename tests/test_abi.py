"""The C-ABI library loads and exports every symbol the header declares;
host-side validation returns its errors before any device work (no GPU
needed)."""
import ctypes as C
import os
import re

import pytest

import bit_moe_expert_histogram_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_w4.h")


def declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", txt, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return m.load()


def test_header_declares_the_calls():
    names = declared()
    for n in ("moe_route", "moe_plan", "moe_expert_ffn_w4", "moe_combine", "moe_layer_w4",
              "moe_workspace_bytes", "moe_max_blocks", "moe_query_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = C.CDLL(m.LIB_PATH)
    missing = [n for n in declared() if not hasattr(raw, n)]
    assert not missing, missing
    assert set(m.EXPORTS) <= set(declared())


def test_workspace_and_block_bounds(lib):
    s = m.make_shape(512, 2048, 256, 8, 512, 1, 128)
    assert m.moe_max_blocks(s) == 4096 // 128 + 256 + 512 // 128
    ws = m.moe_workspace_bytes(s)
    R, S = 512 * 8, 512 * 9
    assert ws >= S * 2048 * 2 + S * 512 * 2 + 512 * 256 * 4
    assert ws % 256 == 0
    s1 = m.make_shape(1, 2048, 256, 8, 512, 1, 128)
    assert m.moe_max_blocks(s1) == 1 + 8 + 1


def test_layer_path_choice(lib):
    # 2 (persistent kernel) needs a device that holds its blocks; without one, 1
    assert m.moe_layer_path(m.make_shape(1, 2048, 256, 8, 512, 1, 128)) in (1, 2)
    assert m.moe_layer_path(m.make_shape(4, 2048, 256, 8, 512, 1, 128)) in (1, 2)
    assert m.moe_layer_path(m.make_shape(5, 2048, 256, 8, 512, 1, 128)) == 0
    assert m.moe_layer_path(m.make_shape(512, 2048, 256, 8, 512, 1, 128)) == 0
    assert m.moe_layer_path(m.make_shape(1, 8192, 256, 8, 512, 1, 128)) in (1, 2)
    assert m.moe_layer_path(m.make_shape(2, 8192, 256, 8, 512, 1, 128)) == 1   # T*H > 8192
    assert m.moe_layer_path(m.make_shape(4, 8192, 256, 8, 512, 1, 128)) == 0   # 64 KiB of x
    assert m.moe_layer_path(m.make_shape(1, 2048, 256, 8, 384, 1, 128)) == 0   # I not 2^n
    assert m.moe_layer_path(m.make_shape(1, 2048, 256, 8, 2048, 1, 128)) == 0  # I > 1024
    assert m.moe_layer_path(m.make_shape(1, 2048, 1024, 32, 512, 1, 128)) == 0  # E > 256
    assert m.moe_layer_path(m.make_shape(1, 2048, 512, 8, 512, 1, 128)) == 0    # E > 256
    assert m.moe_layer_path(m.make_shape(1, 2048, 256, 32, 1024, 1, 128)) in (1, 2)  # 33 slots
    assert m.moe_layer_path(m.make_shape(0, 2048, 256, 8, 512, 1, 128)) == -1


@pytest.mark.parametrize("bad", [dict(H=200), dict(H=128), dict(I=64), dict(K=0), dict(K=17, E=16),
                                 dict(E=2048), dict(n_shared=2), dict(tile_rows=0),
                                 dict(tile_rows=129), dict(T=0), dict(K=33, E=64)])
def test_unsupported_shapes(lib, bad):
    kw = dict(T=16, H=256, E=16, K=2, I=128, n_shared=1, tile_rows=128)
    kw.update(bad)
    s = m.make_shape(**kw)
    assert m.moe_workspace_bytes(s) == 0
    assert m.moe_max_blocks(s) == 0
    st = lib.moe_route(C.byref(s), C.c_void_p(16), C.c_void_p(16), None, C.c_void_p(16),
                       C.c_void_p(16), C.c_void_p(256), 1 << 30, None)
    assert st == m.MOE_ERR_UNSUPPORTED_SHAPE


def test_argument_errors_before_any_launch(lib):
    s = m.make_shape(16, 256, 16, 2, 128, 1, 128)
    need = m.moe_workspace_bytes(s)
    P = C.c_void_p
    # null input
    assert lib.moe_route(C.byref(s), None, P(16), None, P(16), P(16), P(256), need, None) == \
        m.MOE_ERR_INVALID_ARG
    # misaligned hidden states
    assert lib.moe_route(C.byref(s), P(18), P(16), None, P(16), P(16), P(256), need, None) == \
        m.MOE_ERR_INVALID_ARG
    # workspace too small / misaligned
    assert lib.moe_route(C.byref(s), P(16), P(16), None, P(16), P(16), P(256), need - 1, None) == \
        m.MOE_ERR_WORKSPACE
    assert lib.moe_route(C.byref(s), P(16), P(16), None, P(16), P(16), P(128), need, None) == \
        m.MOE_ERR_INVALID_ARG
    # plan with a null buffer
    plan = m.PlanPtrs(16, 16, 16, 16, 16, 0)
    assert lib.moe_plan(C.byref(s), P(16), C.byref(plan), P(256), need, None) == \
        m.MOE_ERR_INVALID_ARG
    # ffn: shared expert required when n_shared == 1
    w = m.W4Weights(16, 16, 16, 16, 16, 16)
    plan = m.PlanPtrs(16, 16, 16, 16, 16, 16)
    assert lib.moe_expert_ffn_w4(C.byref(s), P(16), C.byref(w), None, C.byref(plan), P(16),
                                 P(256), need, None) == m.MOE_ERR_INVALID_ARG
    wbad = m.W4Weights(16, 16, 24, 16, 16, 16)
    assert lib.moe_expert_ffn_w4(C.byref(s), P(16), C.byref(wbad), C.byref(w), C.byref(plan),
                                 P(16), P(256), need, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(C.byref(s), P(16), None, P(16), P(16), None, None) == \
        m.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_dequant_w4(P(16), P(16), P(16), P(16), 4, 100, None) == \
        m.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_dequant_w4_decode(P(16), P(16), P(16), P(16), 4, 100, None) == \
        m.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_dequant_w4_decode(P(16), P(16), P(16), P(24), 4, 64, None) == \
        m.MOE_ERR_INVALID_ARG


def test_status_strings(lib):
    for code in range(7):
        assert lib.moe_status_string(code)
    assert lib.moe_status_string(99) == b"unknown status"


def test_decode_layers_argument_errors(lib):
    s = m.make_shape(1, 256, 16, 2, 128, 1, 128)
    big = m.make_shape(5, 256, 16, 2, 128, 1, 128)   # T=5 takes the grouped-GEMM path
    table = (m.LayerWeights * 1)()
    assert lib.moe_decode_layers(C.byref(big), 1, C.cast(table, C.c_void_p), None, None, None,
                                 None, 0, None) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_decode_layers(C.byref(s), 0, C.cast(table, C.c_void_p), None, None, None,
                                 None, 0, None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_layers(C.byref(s), 1, None, None, None, None, None, 0,
                                 None) == m.MOE_ERR_INVALID_ARG


def test_workspace_of_the_chunked_prefill_fits_two_gib(lib):
    """The chunked workload reuses one workspace per chunk of 2048 tokens;
    it stays far below 2 GiB (the plan, h, the plan-ordered activations and
    the slot outputs at T=2048)."""
    s = m.make_shape(2048, 2048, 256, 8, 512, 1, 128)
    n = m.moe_workspace_bytes(s)
    assert 0 < n <= 2 << 30
    # and it grows no faster than linearly in T: twice the tokens, at most
    # twice the bytes plus the fixed part
    n2 = m.moe_workspace_bytes(m.make_shape(4096, 2048, 256, 8, 512, 1, 128))
    n1 = m.moe_workspace_bytes(m.make_shape(1, 2048, 256, 8, 512, 1, 128))
    assert n2 <= 2 * n + n1


def test_attention_workspace_and_argument_errors(lib):
    """Host checks of moe_attn_decode, in order: the shape, the pointers,
    the workspace size; none reaches the device."""
    ok = m.make_attn_shape(1, 16, 2, 128, 32768)
    n = lib.moe_attn_workspace_bytes(C.byref(ok))
    # the status word and the partials of at most one chunk per cache block
    assert n == 256 + 2 * 512 * 16 * (128 + 2) * 4
    for bad in [(3, 16, 2, 128, 100), (1, 16, 3, 128, 100), (1, 16, 2, 96, 100),
                (2, 16, 1, 128, 100), (1, 16, 2, 128, 0), (1, 16, 2, 128, 100, 32)]:
        s = m.make_attn_shape(*bad)
        assert lib.moe_attn_workspace_bytes(C.byref(s)) == 0
        assert lib.moe_attn_decode(C.byref(s), None, None, None, None, 1, None, None, 0,
                                   None) == m.MOE_ERR_UNSUPPORTED_SHAPE
    p = C.c_void_p(0x10000)
    assert lib.moe_attn_decode(C.byref(ok), None, p, p, p, 1, p, p, n,
                               None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_attn_decode(C.byref(ok), C.c_void_p(0x10008), p, p, p, 1, p, p, n,
                               None) == m.MOE_ERR_INVALID_ARG  # q not 16-byte aligned
    assert lib.moe_attn_decode(C.byref(ok), p, p, p, p, 0, p, p, n,
                               None) == m.MOE_ERR_INVALID_ARG  # an empty block pool
    assert lib.moe_attn_decode(C.byref(ok), p, p, p, p, 1, p, p, n - 1,
                               None) == m.MOE_ERR_WORKSPACE


def test_gdn_scan_argument_errors(lib):
    p = C.c_void_p(0x10000)
    for bad in [(1, 16, 32, 64, 128), (1, 16, 24, 128, 128), (1, 16, 32, 128, 40),
                (0, 16, 32, 128, 128), (1, 0, 32, 128, 128)]:
        s = m.make_gdn_shape(*bad)
        assert lib.moe_gdn_scan(C.byref(s), p, p, p, p, p, p, p, p,
                                None) == m.MOE_ERR_UNSUPPORTED_SHAPE
    ok = m.make_gdn_shape(4, 16, 32, 128, 128)
    assert lib.moe_gdn_scan(C.byref(ok), p, p, p, p, None, p, p, p,
                            None) == m.MOE_ERR_INVALID_ARG
    assert lib.moe_gdn_scan(C.byref(ok), p, p, p, p, p, C.c_void_p(0x10004), p, p,
                            None) == m.MOE_ERR_INVALID_ARG  # the state not 16-byte aligned


def test_decoder_blocks_argument_errors(lib):
    s = m.make_shape(1, 256, 16, 2, 128, 1, 128)
    table = (m.LayerWeights * 1)()
    gains = (C.c_void_p * 1)(0x10000)
    out = C.c_void_p(0x20000)
    call = lambda shape, n, tab, g, h_in, tok, emb, vocab, h_out, wsb=0: lib.moe_decoder_blocks(
        C.byref(shape), n, tab, g, h_in, tok, emb, vocab, h_out, None, wsb, None)
    T = C.cast(table, C.c_void_p)
    G = C.cast(gains, C.c_void_p)
    bad_shape = m.make_shape(1, 100, 16, 2, 128, 1, 128)  # H not a multiple of 256
    assert call(bad_shape, 1, T, G, out, None, None, 0, out) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert call(s, 0, T, G, out, None, None, 0, out) == m.MOE_ERR_INVALID_ARG     # no layers
    assert call(s, 1, T, None, out, None, None, 0, out) == m.MOE_ERR_INVALID_ARG  # no gains
    assert call(s, 1, T, G, None, None, None, 0, out) == m.MOE_ERR_INVALID_ARG   # no h_0
    tok = C.c_void_p(0x30000)
    assert call(s, 1, T, G, None, tok, None, 10, out) == m.MOE_ERR_INVALID_ARG   # ids, no table
    assert call(s, 1, T, G, None, tok, out, 0, out) == m.MOE_ERR_INVALID_ARG     # empty table
    # the layer table itself: a router pointer is required
    assert call(s, 1, T, G, out, None, None, 0, out) == m.MOE_ERR_INVALID_ARG
