"""One process per rank over peer memory, on one GPU: every rank process
keeps its own gradients and rank-major buffer, exports them, maps its
peers' (CUDA IPC between processes sharing the device) and runs the
library's single-rank reduce-scatter on a pointer table of its own and its
peers' gradients, then packs its shard into its own block and places every
rank's block straight from that rank's buffer.  Each process checks its
shards against the oracle's single-rank reduce-scatter and its parameters
against bf16 of the oracle's full reduction, bit for bit.  The processes
synchronise on the host (gloo barriers) between steps; no kernel waits on
another process."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gpu_checks  # noqa: E402
import synth  # noqa: E402
from synth.device import DeviceJob  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only hosts
    pytest.skip("no CUDA device", allow_module_level=True)

import layout_aware_collectives_gb300 as tide  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_PROCESS = r"""
import os
import sys
sys.path[:0] = [ROOT, TESTS]
import numpy as np
import torch
import torch.distributed as dist

rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
mode = os.environ["IPC_TEST_MODE"]
torch.cuda.set_device(0)
dist.init_process_group("gloo", rank=rank, world_size=world)
import layout_aware_collectives_gb300 as tide
from layout_aware_collectives_gb300 import ipc
import oracle
import synth
from synth.device import fill_bf16

shapes = [(37, 24), (3 * world + 1,), (max(1, world - 1), 16), (), (2 * world, 3, 5), (64, 64), (0, 8)]
wl = synth.custom("ipc_ranks", world, shapes, sigma=0.5, seed=7)
P = wl.num_params
CANARY32, CANARY16 = -0x5A5A5A5B, 0x7FA5
with tide.Layout(shapes, world) as lay:
    if mode == "capped":
        lay.set_mode(tide.TIDE_MODE_CAPPED, 3)
    numels = [synth.numel(s) for s in shapes]
    offs, total = ipc.arena_offsets(numels, 2)
    # 4 MiB apiece: each buffer gets an allocation of its own from torch's allocator
    arena = torch.empty(max(total, 4 << 20) // 2, dtype=torch.int16, device="cuda")
    grads = [arena[o // 2: o // 2 + n] for o, n in zip(offs, numels)]
    for p in range(P):
        if numels[p]:
            fill_bf16(grads[p], wl.grad_key(rank, p), 0, wl.sigma)
    S = lay.block_numel
    gathered = torch.full((max(world * S, 2 << 20),), synth.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    torch.cuda.synchronize()
    ex = ipc.exchange({"grads": tide.tide_ipc_export(arena), "gathered": tide.tide_ipc_export(gathered)})
    peers = ipc.PeerMap()
    gtab = ipc.grad_table(ipc.rank_addresses(ex, rank, "grads", arena.data_ptr(), peers), offs)
    shard_n = [lay.shard_numel(p) for p in range(P)]
    sbufs = [torch.full((n + 128,), CANARY32, dtype=torch.int32, device="cuda") for n in shard_n]
    shards = [b[64: 64 + n].view(torch.float32) for b, n in zip(sbufs, shard_n)]
    dist.barrier()  # every rank's gradients are written
    lay.reduce_scatter_rank(rank, gtab, shards, wl.scale)
    torch.cuda.synchronize()
    host = [[wl.host_grad(k, p) for p in range(P)] for k in range(world)]
    want = oracle.rs_rank(shapes, world, host, wl.scale, rank)
    for p in range(P):
        got = shards[p].view(torch.int32).cpu().numpy().view(np.uint32)
        assert np.array_equal(got, want[p].view(np.uint32)), f"rank {rank}: shard of param {p}"
        b = sbufs[p]
        assert bool((b[:64] == CANARY32).all()) and bool((b[64 + shard_n[p]:] == CANARY32).all())
    # all-gather: own block packed, then every block read from its rank's buffer
    lay.pack(rank, shards, gathered)
    torch.cuda.synchronize()
    dist.barrier()  # every rank's block is packed
    bufs = ipc.rank_addresses(ex, rank, "gathered", gathered.data_ptr(), peers)
    if mode == "copy_engine":
        lay.set_mode(tide.TIDE_MODE_COPY_ENGINE)
    pbufs = [torch.full((n + 256,), CANARY16, dtype=torch.int16, device="cuda") for n in numels]
    params = [b[128: 128 + n] for b, n in zip(pbufs, numels)]
    lay.place_ranks(bufs, params)
    torch.cuda.synchronize()
    full = oracle.rs(shapes, world, host, wl.scale)
    for p in range(P):
        d0 = shapes[p][0] if shapes[p] else 1
        inner = numels[p] // d0 if d0 else 0
        reduced = np.concatenate([full[r][p][: oracle.valid_rows(d0, world, r) * inner] for r in range(world)])
        got = params[p].view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, oracle.f32_to_bf16(reduced)), f"rank {rank}: parameter {p}"
        b = pbufs[p]
        assert bool((b[:128] == CANARY16).all()) and bool((b[128 + numels[p]:] == CANARY16).all())
    lay.check_device()
    dist.barrier()  # every peer is done reading this rank's buffers
    peers.close()
    dist.barrier()
print(f"ok rank {rank}")
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world,mode", [(2, "uncapped"), (3, "capped"), (2, "copy_engine")])
def test_rank_processes_over_peer_memory(world, mode):
    port = _free_port()
    code = RANK_PROCESS.replace("ROOT", repr(ROOT)).replace("TESTS", repr(os.path.join(ROOT, "tests")))
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), IPC_TEST_MODE=mode)
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            outs.append(p.communicate(timeout=300))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    for r, (p, (so, se)) in enumerate(zip(procs, outs)):
        assert p.returncode == 0, f"rank {r}:\n{so[-2000:]}\n{se[-3000:]}"
        assert f"ok rank {r}" in so


@pytest.mark.parametrize("mode", [(tide.TIDE_MODE_UNCAPPED, 0), (tide.TIDE_MODE_CAPPED, 2),
                                  (tide.TIDE_MODE_BULK, 0), (tide.TIDE_MODE_COPY_ENGINE, 0)],
                         ids=["uncapped", "capped2", "bulk", "copy_engine"])
def test_place_ranks_with_one_buffer_is_the_placement(mode):
    """Every rank's buffer the same: the per-rank placement is the oracle's
    placement of that buffer (tiny block and a ragged layout, alignment 1)."""
    for wl, align in ((synth.tiny(), 8),
                      (synth.custom("ragged_ranks", 5, [(13, 24), (4, 7), (16,), (), (0, 8), (10, 3, 5)],
                                    sigma=0.5, seed=5), 1)):
        with tide.Layout(wl.shapes, wl.num_ranks, align_elems=align) as lay:
            lay.set_mode(*mode)
            job = DeviceJob(wl, lay, align=align)
            lay.place_ranks([job.gathered] * job.N, job.param_ptrs())
            torch.cuda.synchronize()
            gpu_checks.full_check_ag(job)
            assert job.guards_intact()


def test_ipc_export_refuses_memory_outside_device_allocations():
    buf = np.zeros(16, dtype=np.uint8)
    with pytest.raises(tide.TideError) as e:
        tide.tide_ipc_export(buf.ctypes.data)
    assert e.value.status == tide.TIDE_ERR_INVALID_ARG
    t = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    h, off = tide.tide_ipc_export(t[4096:])
    h0, off0 = tide.tide_ipc_export(t)
    assert h == h0 and off - off0 == 4096 and len(h) == tide.TIDE_IPC_HANDLE_BYTES
    torch.zeros(1, device="cuda").add_(1)  # no CUDA error left behind
    torch.cuda.synchronize()


@pytest.mark.parametrize("mode", [(tide.TIDE_MODE_UNCAPPED, 0), (tide.TIDE_MODE_CAPPED, 3),
                                  (tide.TIDE_MODE_BULK, 2), (tide.TIDE_MODE_COPY_ENGINE, 0)],
                         ids=["uncapped", "capped3", "bulk_cap2", "copy_engine"])
def test_place_ranks_reads_each_block_from_its_own_buffer(mode):
    """N distinct buffers, buffer k holding real data only in block k and the
    padding sentinel everywhere else: every rank's rows must come from that
    rank's own buffer (a block read from another buffer brings sentinels
    into the parameters), bit for bit the oracle's placement."""
    from synth import SENTINEL_BF16

    cases = [(synth.tiny(), 8),
             (synth.custom("ragged_ranks5", 5, [(13, 24), (4, 7), (16,), (), (0, 8), (10, 3, 5)],
                           sigma=0.5, seed=5), 1),
             (synth.custom("ragged_ranks13", 13, [(40, 9), (12, 16), (3 * 13 + 1,), (26, 3, 5)],
                           sigma=0.5, seed=13), 8)]
    for wl, align in cases:
        with tide.Layout(wl.shapes, wl.num_ranks, align_elems=align) as lay:
            lay.set_mode(*mode)
            job = DeviceJob(wl, lay, align=align)
            S, N = lay.block_numel, job.N
            bufs = []
            for k in range(N):
                b = torch.full_like(job.gathered, SENTINEL_BF16)
                b[k * S:(k + 1) * S] = job.gathered[k * S:(k + 1) * S]
                bufs.append(b)
            torch.cuda.synchronize()
            lay.place_ranks(bufs, job.param_ptrs())
            torch.cuda.synchronize()
            gpu_checks.full_check_ag(job)
            assert job.guards_intact()
