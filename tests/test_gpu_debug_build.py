"""The debug build (libtide_debug.so: every kernel checks each tile it fetches
against the extents of its call's buffers, skips a failing tile and flags
it in the device error word) on valid work: the tiny block and ragged
layouts, every operation in every mode, bit-exact against the oracle and
with the error word clear after every call.  Runs in a child process with
TIDE_LIBRARY=debug, since the binding picks its library when imported."""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only hosts
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path[:0] = [ROOT, TESTS]
import numpy as np
import torch

import layout_aware_collectives_gb300 as tide
assert tide.tide_build_info().startswith("debug"), tide.tide_build_info()
assert tide.LIB_PATH.endswith("libtide_debug.so"), tide.LIB_PATH
import gpu_checks
import oracle
import synth
from synth.device import DeviceJob

# capped 3: per-warp tiles; capped 120: whole-CTA tiles wherever the list has more than 76 tiles
MODES = [(tide.TIDE_MODE_UNCAPPED, 0), (tide.TIDE_MODE_CAPPED, 3), (tide.TIDE_MODE_CAPPED, 120),
         (tide.TIDE_MODE_BULK, 0), (tide.TIDE_MODE_BULK, 3), (tide.TIDE_MODE_COPY_ENGINE, 0)]


def cases():
    rng = np.random.default_rng(11)
    out = [(synth.tiny(), 8)]
    for n in (1, 3, 8, 13, 64):
        shapes = [(int(rng.integers(1, 3 * n + 5)), int(rng.integers(1, 40))) for _ in range(4)]
        shapes += [(n - 1 if n > 1 else 1, 24), (3 * n + 1,), (), (0, 16), (7, 0, 3), (2 * n, 3, 5)]
        for align in (8, 1):
            out.append((synth.custom(f"ragged{n}", n, shapes, sigma=0.5, seed=n), align))
    return out


calls = 0
for wl, align in cases():
    with tide.Layout(wl.shapes, wl.num_ranks, align_elems=align) as lay:
        job = DeviceJob(wl, lay, align=align)
        job.make_pack_inputs()
        job.make_slots()
        offs, S = oracle.layout(wl.shapes, job.N, align)
        for mode in MODES:
            lay.set_mode(*mode)
            ce = mode[0] == tide.TIDE_MODE_COPY_ENGINE
            job.reset_outputs()
            if not ce:
                lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), wl.scale)
            lay.place(job.gathered, job.param_ptrs())
            torch.cuda.synchronize()
            lay.check_device()  # TIDE_ERR_RANGE would raise here
            if not ce:
                gpu_checks.full_check_rs(job)
            gpu_checks.full_check_ag(job)
            assert job.guards_intact()
            if not ce:
                for r in sorted({0, job.N - 1}):
                    outs = [torch.empty(n, dtype=torch.float32, device="cuda") for n in job.shard_numel]
                    lay.reduce_scatter_rank(r, job.grad_ptrs(), outs, wl.scale)
                    torch.cuda.synchronize()
                    lay.check_device()
                    gpu_checks.check_rank_rs(job, r, outs)
                job.packed.fill_(synth.SENTINEL_BF16)
                lay.pack(-1, job.pack_src_ptrs(), job.packed)
                torch.cuda.synchronize()
                lay.check_device()
                gpu_checks.check_pack(job, range(job.N))
            for k in range(job.N):
                job.slots[k].fill_(synth.SENTINEL_BF16)
                lay.stage([job.grads[k][p] for p in range(job.P)], job.slots[k])
            torch.cuda.synchronize()
            lay.check_device()
            for k in range(job.N):
                want = oracle.rs_stage(wl.shapes, job.N, offs, S, [wl.host_grad(k, p) for p in range(job.P)],
                                       np.full(job.N * S, synth.SENTINEL_BF16, np.uint16))
                assert np.array_equal(job.slots[k].cpu().numpy().view(np.uint16), want), (wl.name, mode, k)
            if not ce:
                job.reset_outputs()
                lay.reduce_scatter_staged(job.slots, job.shard_ptrs(), wl.scale)
                torch.cuda.synchronize()
                lay.check_device()
                gpu_checks.full_check_rs(job)
            calls += 1
print(f"ok: {calls} (layout, mode) runs of the debug build, error word clear after every call")
"""


def test_debug_build_on_valid_work_matches_the_oracle_with_no_range_flag():
    env = dict(os.environ, TIDE_LIBRARY="debug")
    code = CHILD.replace("ROOT", repr(ROOT)).replace("TESTS", repr(os.path.join(ROOT, "tests")))
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stdout[-4000:] + res.stderr[-4000:]
    assert res.stdout.strip().splitlines()[-1].startswith("ok:"), res.stdout[-2000:]
