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
