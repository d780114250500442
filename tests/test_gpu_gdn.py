"""GPU parity of the Gated DeltaNet recurrence (moe_gdn_scan; "Perplexity
Open Sources Lily: A Rust + Metal Inference Engine for Qwen3.6-35B-A3B on
Apple Silicon", sections "Three Workload Shapes" and "Prefill": a
register-resident scan of the gated delta rule) against the oracle: the
model's head counts at one decode token and at a 64-token scan, other head
groupings, the state carried across calls and updated in place, and
unsupported shapes."""
import numpy as np
import pytest
import torch

import bit_moe_expert_histogram_gb300 as m
import oracle
import synth
from moe_case import close, d16, f64, h16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    m.load()


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def run(T, n_k, n_v, dk, dv, seed, inputs=None, state=None):
    q, k, v, alpha, beta, s0 = inputs if inputs is not None else synth.gen_gdn(
        T, n_k, n_v, dk, dv, seed=seed)
    if state is not None:
        s0 = state
    shape = m.make_gdn_shape(T, n_k, n_v, dk, dv)
    sd = dev_f32(s0)
    o = torch.zeros((T, n_v, dv), dtype=torch.int16, device="cuda")
    m.moe_gdn_scan(shape, d16(q, "cuda"), d16(k, "cuda"), d16(v, "cuda"), dev_f32(alpha),
                   dev_f32(beta), sd, sd, o)
    torch.cuda.synchronize()
    return h16(o).copy(), sd.cpu().numpy(), (q, k, v, alpha, beta, s0)


@pytest.mark.parametrize("T,n_k,n_v,dv", [(1, 16, 32, 128), (64, 16, 32, 128), (7, 4, 4, 64),
                                          (3, 2, 8, 16)])
def test_gdn_scan_against_the_oracle(T, n_k, n_v, dv):
    o, s_end, inp = run(T, n_k, n_v, 128, dv, seed=T * 7 + n_v)
    o_ref, s_ref = oracle.gdn_scan(*inp)
    close(f64(o), f64(o_ref), "o")
    close(s_end, s_ref, "state")


def test_gdn_state_carries_across_calls():
    """Two calls of 5 tokens each give the state and outputs of one call of
    10 (the scan is exactly sequential in the state it keeps)."""
    T, n_k, n_v, dv = 10, 16, 32, 128
    inp = synth.gen_gdn(T, n_k, n_v, 128, dv, seed=5)
    q, k, v, alpha, beta, s0 = inp
    o_all, s_all, _ = run(T, n_k, n_v, 128, dv, 0, inputs=inp)
    o_a, s_a, _ = run(5, n_k, n_v, 128, dv, 0, inputs=(q[:5], k[:5], v[:5], alpha[:5], beta[:5], s0))
    o_b, s_b, _ = run(5, n_k, n_v, 128, dv, 0, inputs=(q[5:], k[5:], v[5:], alpha[5:], beta[5:], s_a))
    assert np.array_equal(np.concatenate([o_a, o_b]), o_all)
    assert np.array_equal(s_b, s_all)


def test_gdn_rejects_unsupported_shapes():
    z = torch.zeros(16, dtype=torch.float32, device="cuda")
    for args in [(1, 16, 32, 64, 128), (1, 16, 24, 128, 128), (1, 16, 32, 128, 40),
                 (0, 16, 32, 128, 128)]:
        with pytest.raises(m.MoeError):
            m.moe_gdn_scan(m.make_gdn_shape(*args), z, z, z, z, z, z, z, z)


# ----------------------------------------------------- chunked form --
def run_chunked(T, n_k, n_v, dk, dv, inputs, state=None):
    q, k, v, alpha, beta, s0 = inputs
    if state is not None:
        s0 = state
    shape = m.make_gdn_shape(T, n_k, n_v, dk, dv)
    ws = m.alloc_gdn_workspace(shape, "cuda")
    sd = dev_f32(s0)
    o = torch.zeros((T, n_v, dv), dtype=torch.int16, device="cuda")
    m.moe_gdn_chunked_scan(shape, d16(q, "cuda"), d16(k, "cuda"), d16(v, "cuda"), dev_f32(alpha),
                           dev_f32(beta), sd, sd, o, ws)
    torch.cuda.synchronize()
    assert m.moe_query_device_status(ws) == 0  # the workspace's status word stays clear
    return h16(o).copy(), sd.cpu().numpy()


@pytest.mark.parametrize("T,n_k,n_v,dv", [(1, 16, 32, 128), (64, 16, 32, 128), (2048, 16, 32, 128),
                                          (100, 4, 8, 64), (65, 2, 2, 16), (130, 16, 32, 128)])
def test_gdn_chunked_against_the_oracle(T, n_k, n_v, dv):
    """The chunked scan (chunks of 64, ragged last chunks included) against
    the oracle's token-by-token recurrence, outputs and final state."""
    inp = synth.gen_gdn(T, n_k, n_v, 128, dv, seed=T * 3 + n_v)
    o, s_end = run_chunked(T, n_k, n_v, 128, dv, inp)
    o_ref, s_ref = oracle.gdn_scan(*inp)
    close(f64(o), f64(o_ref), "o")
    close(s_end, s_ref, "state")


@pytest.mark.parametrize("lo,hi", [(0.05, 0.5), (0.0, 0.02)])
def test_gdn_chunked_fast_decay(lo, hi):
    """Heads that forget fast: alpha in [lo, hi) drives the running product
    of a 64-token chunk far below the smallest fp32 number (and alpha = 0
    occurs), where the chunk's gate ratios still have to come out right."""
    T, n_k, n_v, dv = 160, 16, 32, 128
    q, k, v, _, beta, s0 = synth.gen_gdn(T, n_k, n_v, 128, dv, seed=21)
    alpha = np.random.default_rng(22).uniform(lo, hi, (T, n_v)).astype(np.float32)
    alpha[::7, ::3] = np.float32(lo)
    inp = (q, k, v, alpha, beta, s0)
    o, s_end = run_chunked(T, n_k, n_v, 128, dv, inp)
    o_ref, s_ref = oracle.gdn_scan(*inp)
    assert np.isfinite(f64(o)).all() and np.isfinite(s_end).all()
    close(f64(o), f64(o_ref), "o")
    close(s_end, s_ref, "state")


def test_gdn_chunked_equals_the_recurrent_kernel_and_carries_state():
    """Both device forms give the same outputs and state within the layer's
    tolerance; the chunked form's state carries across calls (two calls of
    96 tokens against one of 192)."""
    T, n_k, n_v, dv = 192, 16, 32, 128
    inp = synth.gen_gdn(T, n_k, n_v, 128, dv, seed=9)
    q, k, v, alpha, beta, s0 = inp
    o_r, s_r, _ = run(T, n_k, n_v, 128, dv, 0, inputs=inp)
    o_c, s_c = run_chunked(T, n_k, n_v, 128, dv, inp)
    close(f64(o_c), f64(o_r), "o")
    close(s_c, s_r, "state")
    o_a, s_a = run_chunked(96, n_k, n_v, 128, dv, (q[:96], k[:96], v[:96], alpha[:96], beta[:96], s0))
    o_b, s_b = run_chunked(96, n_k, n_v, 128, dv, (q[96:], k[96:], v[96:], alpha[96:], beta[96:], s_a))
    close(f64(np.concatenate([o_a, o_b])), f64(o_c), "o in two calls")
    close(s_b, s_c, "state in two calls")


def test_gdn_chunked_rejects_unsupported_shapes_and_small_workspace():
    z = torch.zeros(64, dtype=torch.float32, device="cuda")
    shape = m.make_gdn_shape(4, 2, 2, 128, 256)   # dv > 128
    assert m.load().moe_gdn_chunked_workspace_bytes(shape) == 0
    with pytest.raises(m.MoeError):
        m.moe_gdn_chunked_scan(shape, z, z, z, z, z, z, z, z, z)
    shape = m.make_gdn_shape(4, 2, 2, 128, 16)
    with pytest.raises(m.MoeError):
        m.moe_gdn_chunked_scan(shape, z, z, z, z, z, z, z, z, z)   # 256 bytes of workspace
