"""Seeded random layouts through every entry point, against the CPU oracle,
bit for bit.

Each case draws a rank count (1 to 100), one to six parameter shapes
(scalars, 1-D to 3-D tensors, zero-size tensors, dim 0 below and above N,
some large enough that the capped grids exceed half the SMs), an offset
alignment, a generator scale, a reduce-scatter scale and a mode: over every
SM, capped on either side of half the SM count (per-warp and whole-CTA
capped forms), or TMA-staged with a cap from 0 to 40.  It then runs the
reduce-scatter of all ranks, the single-rank reduce-scatter of a random
rank, the no-allocation reduce-scatter, placement, per-rank placement, the
all-gather input pack, Slot-Reuse staging and the staged reduce-scatter,
and compares each with the oracle; guard bands must stay intact.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gpu_checks  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from synth import SENTINEL_BF16  # noqa: E402
from synth.device import DeviceJob  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only hosts
    pytest.skip("no CUDA device", allow_module_level=True)

import layout_aware_collectives_gb300 as tide  # noqa: E402

RANKS = [1, 2, 3, 4, 5, 7, 8, 9, 13, 16, 31, 32, 33, 64, 65, 100]
ALIGNS = [1, 2, 4, 8, 16, 64]
CASES = 96


def draw_case(i, sms):
    rng = np.random.default_rng(7000 + i)
    n = int(rng.choice(RANKS))
    big = rng.random() < 0.4  # a few parameters of up to ~0.5M elements
    shapes = []
    for _ in range(int(rng.integers(1, 7))):
        nd = int(rng.integers(0, 4))
        if nd == 0:
            shapes.append(())
            continue
        hi = 800 if big and rng.random() < 0.5 else 40
        d0 = int(rng.integers(0, 3 * n + hi))
        rest = [0 if rng.random() < 0.05 else int(rng.integers(1, hi if k == 0 else 6)) for k in range(nd - 1)]
        shapes.append((d0, *rest))
    align = int(rng.choice(ALIGNS))
    kind = int(rng.integers(0, 4))
    if kind == 0:
        mode = (tide.TIDE_MODE_UNCAPPED, 0)
    elif kind == 1:
        mode = (tide.TIDE_MODE_CAPPED, int(rng.integers(1, sms // 2 + 1)))
    elif kind == 2:
        mode = (tide.TIDE_MODE_CAPPED, int(rng.integers(sms // 2 + 1, 2 * sms + 1)))
    else:
        mode = (tide.TIDE_MODE_BULK, int(rng.integers(0, 41)))
    sigma = float(rng.choice([1e-3, 0.5, 8.0]))
    scale = float(rng.choice([1.0 / n, 0.3, -1.0, 1.0]))
    rank = int(rng.integers(0, n))
    return n, shapes, align, mode, sigma, scale, rank


def _staging(job, scale):
    wl, lay = job.wl, job.layout
    offs, S = oracle.layout(wl.shapes, job.N, job.align)
    job.make_slots()
    for k in range(job.N):
        lay.stage([job.grads[k][p] for p in range(job.P)], job.slots[k])
    torch.cuda.synchronize()
    for k in range(job.N):
        want = np.full(job.N * S, SENTINEL_BF16, dtype=np.uint16)
        oracle.rs_stage(wl.shapes, job.N, offs, S, [wl.host_grad(k, p) for p in range(job.P)], want)
        assert np.array_equal(job.slots[k].cpu().numpy().view(np.uint16), want), f"staging of rank {k}"
    job.reset_outputs()
    lay.reduce_scatter_staged(job.slots, job.shard_ptrs(), scale)
    torch.cuda.synchronize()
    gpu_checks.full_check_rs(job, scale=scale)
    del job.slots


@pytest.mark.parametrize("i", range(CASES))
def test_random_layout_every_entry_point(i):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n, shapes, align, mode, sigma, scale, rank = draw_case(i, sms)
    wl = synth.custom(f"fuzz{i}", n, shapes, sigma=sigma, seed=i)
    with tide.Layout(wl.shapes, n, align_elems=align) as lay:
        lay.set_mode(*mode)
        job = DeviceJob(wl, lay, align=align)
        gpu_checks.check_layout(job)
        # reduce-scatter of every rank, then placement and per-rank placement
        lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), scale)
        lay.place(job.gathered, job.param_ptrs())
        torch.cuda.synchronize()
        lay.check_device()
        gpu_checks.full_check_rs(job, scale=scale)
        gpu_checks.full_check_ag(job)
        assert job.guards_intact()
        job.reset_outputs()
        lay.place_ranks([job.gathered] * n, job.param_ptrs())
        torch.cuda.synchronize()
        gpu_checks.full_check_ag(job)
        # the no-allocation form (load/store kernels in every mode)
        lay.reduce_scatter_noalloc(job.grad_ptrs(), job.shard_ptrs(), scale)
        torch.cuda.synchronize()
        gpu_checks.full_check_rs(job, scale=scale)
        assert job.guards_intact()
        # one rank's shards
        bufs = [gpu_checks.guarded(m, torch.int32, job.device, -0x5A5A5A5B) for m in job.shard_numel]
        outs = [b[1].view(torch.float32) for b in bufs]
        lay.reduce_scatter_rank(rank, job.grad_ptrs(), outs, scale)
        torch.cuda.synchronize()
        gpu_checks.check_rank_rs(job, rank, outs, scale)
        for buf, view, g in bufs:
            assert bool((buf[:g] == -0x5A5A5A5B).all()) and bool((buf[g + view.numel():] == -0x5A5A5A5B).all())
        # all-gather input pack of every rank
        job.make_pack_inputs()
        lay.pack(-1, job.pack_src_ptrs(), job.packed)
        torch.cuda.synchronize()
        gpu_checks.check_pack(job, range(n))
        del job.pack_src, job.packed
        # Slot-Reuse staging and the staged reduce-scatter
        _staging(job, scale)
        lay.check_device()
