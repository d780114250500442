"""The bench's gpu_launches figure against the kernels a profiled step runs.

bench.py reports launches_per_step() x steps as its kernel-launch count.
Here one step of each stacked workload runs under the CUDA activity tracer
of torch.profiler, and the kernels it records (those of the library, not
PyTorch's own fills or copies) must number exactly launches_per_step()."""
import dataclasses

import pytest
import torch

import bit_moe_expert_histogram_gb300 as m
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    m.load()


def _library_kernels(fn):
    from torch.autograd import DeviceType
    from torch.profiler import ProfilerActivity, profile
    names = []
    for _ in range(2):  # the first trace of a process can come back empty
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if e.device_type == DeviceType.CUDA]
        if names:
            break
    if not names:
        pytest.skip("the profiler recorded no CUDA activity on this device")
    # PyTorch's own kernels are in its at:: namespace; copies and fills are
    # not kernels of the library
    return [n for n in names if "at::" not in n and not n.startswith(("Memcpy", "Memset"))]


@pytest.mark.parametrize("name,layers", [("prefill", 0), ("skewed", 0), ("decode", 2)])
def test_launches_per_step_matches_a_profiled_step(name, layers):
    import bench
    wl = synth.CONFIGS[name]
    if layers:
        wl = dataclasses.replace(wl, layers=layers)
    G = bench.GpuWorkload(wl, torch.device("cuda"), m)
    G.step()  # first-call set-up (function attributes, tensor maps) outside the trace
    kernels = _library_kernels(G.step)
    assert len(kernels) == G.launches_per_step(), kernels
    assert m.moe_query_device_status(G.ws) == 0
