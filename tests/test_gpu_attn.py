"""GPU parity of grouped-query decode attention over a block-paged cache
(moe_attn_decode; "Perplexity Open Sources Lily: A Rust + Metal Inference
Engine for Qwen3.6-35B-A3B on Apple Silicon", sections "Three Workload
Shapes" and "Decode: Minimize Bytes Moved Per Token") against the oracle:
lengths with ragged last blocks, one chunk and many, two new tokens under
the causal window, other head groupings, the 32K context of the bench, and a
bad block-table entry."""
import numpy as np
import pytest
import torch

import bit_moe_expert_histogram_gb300 as m
import oracle
import synth
from moe_case import close as close_layer, d16, f64, h16

pytestmark = pytest.mark.gpu


def close(g, r, what=""):
    """The attention tolerance: each softmax weight is rounded to bf16
    before it multiplies V (relative 2^-9), and so is the output, so the
    mean relative error is allowed twice the layer's 2e-3."""
    return close_layer(g, r, what, mre_bound=4e-3)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    m.load()


def run(T, n_q, n_kv, D, L, seed, table=None):
    q, k, v, tab = synth.gen_attn(T, n_q, n_kv, D, L, seed=seed)
    if table is not None:
        tab = table
    dev = torch.device("cuda")
    shape = m.make_attn_shape(T, n_q, n_kv, D, L)
    ws = m.alloc_attn_workspace(shape, dev)
    o = torch.zeros((T, n_q, D), dtype=torch.int16, device=dev)
    m.moe_attn_decode(shape, d16(q, dev), d16(k, dev), d16(v, dev),
                      torch.from_numpy(np.ascontiguousarray(tab, np.int32)).to(dev), o, ws)
    st = m.moe_query_device_status(ws)
    return h16(o).copy(), (q, k, v, tab), st


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 200, 1000, 4113])
def test_attn_lengths(L):
    o, (q, k, v, tab), st = run(1, 16, 2, 128, L, seed=L)
    assert st == 0
    close(f64(o), f64(oracle.attn_decode(q, k, v, tab, L)), "o at L=%d" % L)


@pytest.mark.parametrize("T,n_q,n_kv,D,L", [(2, 16, 2, 128, 777), (2, 16, 2, 64, 3000),
                                            (1, 8, 8, 64, 500), (1, 32, 2, 128, 129),
                                            (2, 4, 1, 128, 70)])
def test_attn_shapes(T, n_q, n_kv, D, L):
    o, (q, k, v, tab), st = run(T, n_q, n_kv, D, L, seed=7 * L + T)
    assert st == 0
    close(f64(o), f64(oracle.attn_decode(q, k, v, tab, L)), "o")


def test_attn_long_context_of_the_bench():
    """32K positions, the bench's context: every query row against the oracle."""
    L = 32768
    o, (q, k, v, tab), st = run(1, 16, 2, 128, L, seed=32)
    assert st == 0
    close(f64(o), f64(oracle.attn_decode(q, k, v, tab, L)), "o at 32K")


def test_attn_is_deterministic():
    a, _, _ = run(1, 16, 2, 128, 5000, seed=5)
    b, _, _ = run(1, 16, 2, 128, 5000, seed=5)
    assert np.array_equal(a, b)


def test_attn_bad_table_entry_is_recorded_and_left_out():
    L = 300
    q, k, v, tab = synth.gen_attn(1, 16, 2, 128, L, seed=9)
    bad = tab.copy()
    bad[2] = k.shape[0]  # past the pool
    o, _, st = run(1, 16, 2, 128, L, seed=9, table=bad)
    assert st == m.MOE_ERR_BAD_INPUT
    # the reference: the same attention without positions 128..191
    keep = [j for j in range(L) if j // 64 != 2]
    kk = np.stack([k[tab[j // 64], :, j % 64] for j in keep], axis=1)
    vv = np.stack([v[tab[j // 64], :, j % 64] for j in keep], axis=1)
    n = len(keep)
    nb = (n + 63) // 64
    kp = np.zeros((nb, 2, 64, 128), np.uint16); vp = np.zeros_like(kp)
    for j in range(n):
        kp[j // 64, :, j % 64] = kk[:, j]
        vp[j // 64, :, j % 64] = vv[:, j]
    ref = oracle.attn_decode(q, kp, vp, np.arange(nb, dtype=np.int32), n)
    close(f64(o), f64(ref), "o without the bad block")


def test_attn_rejects_unsupported_shapes():
    for args in [(3, 16, 2, 128, 100), (1, 16, 3, 128, 100), (1, 16, 2, 96, 100),
                 (2, 16, 1, 128, 100), (1, 16, 2, 128, 0)]:
        assert m.load().moe_attn_workspace_bytes(m.make_attn_shape(*args)) == 0
