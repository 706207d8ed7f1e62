"""The reduce-scatter entry point that allocates nothing.

Some callers cannot call cudaMalloc (a framework whose caching allocator owns
all device memory, a process under a hard memory cap, a step that cannot take
the synchronisation of a cudaFree).  tide_rs_bf16_to_fp32_noalloc serves them
from a fixed device array inside the library.  This file is collected last so
that a run stopping at its first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth  # noqa: E402
from synth.device import DeviceJob  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

import layout_aware_collectives_gb300 as tide  # noqa: E402
from layout_aware_collectives_gb300 import tide as T  # noqa: E402


def _call_noalloc(layout, job, scale, stream):
    """Direct C-ABI call (ctypes), no binding helpers in between."""
    g = (ctypes.c_void_p * (job.N * job.P))(*[t.data_ptr() for t in job.grad_ptrs()])
    s = (ctypes.c_void_p * (job.N * job.P))(*[t.data_ptr() for t in job.shard_ptrs()])
    fn = T._lib.tide_rs_bf16_to_fp32_noalloc
    return fn(layout.handle, ctypes.addressof(g), ctypes.addressof(s), ctypes.c_float(scale),
              ctypes.c_void_p(stream.cuda_stream))


def _shards(job):
    return [s.view(torch.int32).clone() for row in job.shards for s in row]


@pytest.mark.parametrize("name", ["tiny", "llama8b"])
def test_noalloc_matches_regular_entry_point_twice(name):
    wl = synth.WORKLOADS[name]()
    stream = torch.cuda.Stream()
    with tide.Layout(wl.shapes, wl.num_ranks) as lay:
        job = DeviceJob(wl, lay, guard=True)
        torch.cuda.synchronize()
        lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), wl.scale, stream)
        stream.synchronize()
        want = _shards(job)
        for call in range(2):
            job.reset_outputs()
            torch.cuda.synchronize()
            assert _call_noalloc(lay, job, wl.scale, stream) == tide.TIDE_OK, tide.tide_last_error()
            stream.synchronize()
            got = _shards(job)
            for a, b in zip(got, want):
                assert torch.equal(a, b), f"call {call}"  # bit-exact, like every RS comparison
            assert job.guards_intact()


def test_noalloc_capped_mode_and_size_limit():
    wl = synth.tiny()
    stream = torch.cuda.Stream()
    with tide.Layout(wl.shapes, wl.num_ranks) as lay:
        job = DeviceJob(wl, lay)
        torch.cuda.synchronize()
        lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), wl.scale, stream)
        stream.synchronize()
        want = _shards(job)
        lay.set_mode(tide.TIDE_MODE_CAPPED, 3)
        job.reset_outputs()
        assert _call_noalloc(lay, job, wl.scale, stream) == tide.TIDE_OK
        stream.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(_shards(job), want))
    # a layout whose tile list alone exceeds the fixed array is refused up front
    big = synth.sweep(64)
    with tide.Layout(big.shapes, big.num_ranks) as lay:
        n = big.num_ranks * big.num_params
        fake = (ctypes.c_void_p * n)(*[0x100000 * (i + 1) for i in range(n)])
        st = T._lib.tide_rs_bf16_to_fp32_noalloc(lay.handle, ctypes.addressof(fake),
                                                 ctypes.addressof(fake), ctypes.c_float(1.0), None)
        assert st == tide.TIDE_ERR_INVALID_ARG
        assert "at most" in tide.tide_last_error()
