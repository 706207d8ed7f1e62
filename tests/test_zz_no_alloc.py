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

import gpu_checks  # noqa: E402
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


MODES = [("uncapped", tide.TIDE_MODE_UNCAPPED, 0), ("capped3", tide.TIDE_MODE_CAPPED, 3),
         ("bulk", tide.TIDE_MODE_BULK, 0), ("bulk_cap4", tide.TIDE_MODE_BULK, 4)]


@pytest.mark.parametrize("mode", MODES, ids=[m[0] for m in MODES])
@pytest.mark.parametrize("name", ["tiny", "llama8b"])
def test_noalloc_matches_regular_entry_point_twice(name, mode):
    """Two calls in a row, each bit-exact against the regular entry point in
    the same mode and against the CPU oracle (every element of the tiny
    block; sampled elements of every rank and parameter of the 8B layer)."""
    wl = synth.WORKLOADS[name]()
    stream = torch.cuda.Stream()
    with tide.Layout(wl.shapes, wl.num_ranks) as lay:
        lay.set_mode(*mode[1:])
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
            if name == "tiny":
                gpu_checks.full_check_rs(job)
            else:
                assert gpu_checks.sampled_check_rs(job, seed=call) > 0


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


def test_noalloc_repeats_alternating_layouts_pointers_and_streams():
    """A repeated call on the same stream with the same layout and pointers
    copies nothing; any change (another layout in between, new output
    buffers, another stream) copies again.  Every result bit-exact."""
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    wla, wlb = synth.tiny(), synth.custom("small_b", 3, [(37, 24), (5,), (64, 8)], seed=9)
    with tide.Layout(wla.shapes, wla.num_ranks) as la, tide.Layout(wlb.shapes, wlb.num_ranks) as lb:
        ja, jb = DeviceJob(wla, la), DeviceJob(wlb, lb)
        torch.cuda.synchronize()
        want = {}
        for lay, job, wl in ((la, ja, wla), (lb, jb, wlb)):
            lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), wl.scale, s1)
            s1.synchronize()
            want[id(job)] = _shards(job)
        calls = [(la, ja, wla, s1), (la, ja, wla, s1), (lb, jb, wlb, s1), (la, ja, wla, s1),
                 (la, ja, wla, s2), (la, ja, wla, s2), (lb, jb, wlb, s1)]
        for i, (lay, job, wl, st) in enumerate(calls):
            job.reset_outputs()
            torch.cuda.synchronize()
            assert _call_noalloc(lay, job, wl.scale, st) == tide.TIDE_OK, tide.tide_last_error()
            st.synchronize()
            assert all(torch.equal(a, b) for a, b in zip(_shards(job), want[id(job)])), f"call {i}"
            assert job.guards_intact()
        # new output buffers, same layout and stream: the pointer table is copied again
        outs = [[torch.full_like(s, float("nan")) for s in row] for row in ja.shards]
        g = (ctypes.c_void_p * (ja.N * ja.P))(*[t.data_ptr() for t in ja.grad_ptrs()])
        o = (ctypes.c_void_p * (ja.N * ja.P))(*[t.data_ptr() for row in outs for t in row])
        assert T._lib.tide_rs_bf16_to_fp32_noalloc(la.handle, ctypes.addressof(g), ctypes.addressof(o),
                                                   ctypes.c_float(wla.scale),
                                                   ctypes.c_void_p(s2.cuda_stream)) == tide.TIDE_OK
        s2.synchronize()
        got = [t.view(torch.int32).clone() for row in outs for t in row]
        assert all(torch.equal(a, b) for a, b in zip(got, want[id(ja)]))


def test_noalloc_refused_inside_stream_capture():
    """Pageable copies cannot be replayed from a graph: inside a capture the
    call is refused before it enqueues anything, and the capture stays valid."""
    wl = synth.tiny()
    with tide.Layout(wl.shapes, wl.num_ranks) as lay:
        job = DeviceJob(wl, lay)
        x = torch.zeros(16, device="cuda")
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            graph.capture_begin()
            x.add_(1.0)
            st = _call_noalloc(lay, job, wl.scale, s)
            graph.capture_end()
        assert st == tide.TIDE_ERR_UNSUPPORTED
        assert "captured" in tide.tide_last_error()
        graph.replay()
        torch.cuda.synchronize()
        assert float(x[0]) == 1.0


def test_noalloc_across_device_reset(tmp_path):
    """A plain C program (its own process: a device reset would end this
    one's CUDA context) calls the entry point, resets the device, allocates
    again (often at the same addresses), refills with other values and calls
    twice more on the same stream: the library must see the new context,
    look its array up again and copy, and every shard is exact."""
    import subprocess

    from test_c_abi_driver import build_reset_driver

    exe = tmp_path / "reset_driver"
    build_reset_driver(exe)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.startswith("ok:"), res.stdout
