"""moe_plan_noalloc against moe_plan.

moe_plan_noalloc serves callers that cannot allocate device memory where they
build a routing plan (for example code running inside an allocator callback)
and so cannot hand over a workspace; its scratch is a static device array.
Its plan must equal moe_plan's bit for bit (integer results), also on the
second of two calls in a row, whose inputs differ from the first's. The file
is named so that pytest collects it last."""
import ctypes as C

import numpy as np
import pytest
import torch

import bit_moe_expert_histogram_gb300 as m

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    return m.load()


def _ids(T, E, K, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)


def test_noalloc_plan_equals_workspace_plan_on_two_calls(lib):
    dev = torch.device("cuda")
    # second call: other sizes, so stale scratch from the first would show
    for T, E, K, bm, seed in ((2048, 256, 8, 128, 1), (300, 64, 4, 32, 2)):
        shape = m.make_shape(T, 256, E, K, 128, 1, bm)
        ids = torch.from_numpy(_ids(T, E, K, seed)).to(dev)
        ws = m.alloc_workspace(shape, dev)
        ref = m.PlanBuffers(shape, dev)
        m.moe_plan(shape, ids, ref, ws)
        got = m.PlanBuffers(shape, dev)
        st = lib.moe_plan_noalloc(C.byref(shape), C.c_void_p(ids.data_ptr()), C.byref(got.ptrs),
                                  C.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == m.MOE_OK, lib.moe_last_error()
        torch.cuda.synchronize()
        # the reference plan (moe_plan, through its workspace) saw no error;
        # moe_plan_noalloc reports none by design
        assert m.moe_query_device_status(ws) == 0
        nb = int(ref.num_blocks.item())
        assert int(got.num_blocks.item()) == nb
        for name in ("counts", "offsets", "sorted_rows", "row_pos"):
            assert torch.equal(getattr(got, name), getattr(ref, name)), name
        assert torch.equal(got.block_map[:3 * nb], ref.block_map[:3 * nb])


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    # ceil(16384*8/2048) * 1024 = 65536 > 65472 histogram entries
    shape = m.make_shape(16384, 256, 1024, 8, 128, 1, 128)
    plan = m.PlanPtrs(16, 16, 16, 16, 16, 16)
    st = lib.moe_plan_noalloc(C.byref(shape), C.c_void_p(16), C.byref(plan), None)
    assert st == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert b"static scratch" in lib.moe_last_error()


def test_noalloc_skips_bad_ids_like_moe_plan(lib):
    """Ids outside [0, E) (here -1 and E) are left out of the plan by both
    calls: counts, offsets, the sorted rows that exist, row_pos of every
    valid item and the block map must still agree bit for bit."""
    dev = torch.device("cuda")
    T, E, K, bm = 200, 32, 4, 16
    shape = m.make_shape(T, 256, E, K, 128, 1, bm)
    ids_np = _ids(T, E, K, 5)
    ids_np[3, 1] = -1
    ids_np[77, 0] = E
    ids_np[199, 3] = -1
    ids = torch.from_numpy(ids_np).to(dev)
    ws = m.alloc_workspace(shape, dev)
    ref = m.PlanBuffers(shape, dev)
    m.moe_plan(shape, ids, ref, ws)
    got = m.PlanBuffers(shape, dev)
    st = lib.moe_plan_noalloc(C.byref(shape), C.c_void_p(ids.data_ptr()), C.byref(got.ptrs),
                              C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == m.MOE_OK, lib.moe_last_error()
    torch.cuda.synchronize()
    # the workspace plan records the bad ids in its status word
    assert m.moe_query_device_status(ws) == m.MOE_ERR_BAD_INPUT
    valid = ((ids_np >= 0) & (ids_np < E)).reshape(-1)
    n_valid = int(valid.sum())
    assert torch.equal(got.counts, ref.counts)
    assert torch.equal(got.offsets, ref.offsets)
    assert int(ref.offsets[E].item()) == n_valid
    assert torch.equal(got.sorted_rows[:n_valid], ref.sorted_rows[:n_valid])
    vi = torch.from_numpy(np.nonzero(valid)[0]).to(dev)
    assert torch.equal(got.row_pos[vi], ref.row_pos[vi])
    nb = int(ref.num_blocks.item())
    assert int(got.num_blocks.item()) == nb
    assert torch.equal(got.block_map[:3 * nb], ref.block_map[:3 * nb])
