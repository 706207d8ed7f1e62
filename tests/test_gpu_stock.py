"""The stock-FSDP2 emulation used as a baseline by bench.py computes the
same shards and parameters as the TIDE path (both sum in fp32 in rank order
from +0), so the time comparison compares equal work."""
import pytest

torch = pytest.importorskip("torch")

import synth  # noqa: E402
from synth.device import DeviceJob  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("no CUDA device", allow_module_level=True)

import bench  # noqa: E402
import gpu_checks  # noqa: E402
import layout_aware_collectives_gb300 as tide  # noqa: E402


@pytest.mark.parametrize("name", ["tiny", "llama8b"])
def test_stock_emulation_matches_tide(name):
    wl = synth.WORKLOADS[name]()
    with tide.Layout(wl.shapes, wl.num_ranks) as lay:
        job = DeviceJob(wl, lay, guard=False)
        lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), wl.scale)
        lay.place(job.gathered, job.param_ptrs())
        st = bench.StockFSDP2(job)
        st.copy_in()
        st.flat_reduce(wl.scale)
        st.copy_out()
        torch.cuda.synchronize()
        for r in range(job.N):
            for p in range(job.P):
                assert torch.equal(st.shard(r, p).view(torch.int32), job.shards[r][p].view(torch.int32))
        for p in range(job.P):
            assert torch.equal(st.param(p).view(torch.int16), job.params[p])
        if name == "tiny":
            gpu_checks.full_check_rs(job)
