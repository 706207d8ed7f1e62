"""The rank-process plumbing on the CPU (no GPU): two and three gloo ranks
exchange their buffers' (handle, offset) pairs, map their peers through a
stand-in opener, and build the pointer tables the reduce-scatter and the
per-rank placement take.  Checks: rank order of the exchange, own addresses
used for the own rank, every peer handle opened exactly once even when two
buffers share an allocation, offsets added to the mapped bases, the
rank-major gradient table, and the arena offsets every rank computes alike."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _fake_handle(rank, which):
    return bytes([rank, which]) + bytes(62)


def _worker(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from layout_aware_collectives_gb300 import ipc

    numels = [5, 8, 0, 13]
    offs, total = ipc.arena_offsets(numels, 2)
    # both buffers of a rank live in one allocation: one handle, two offsets
    local = {"grads": (_fake_handle(rank, 1), 4096), "gathered": (_fake_handle(rank, 1), 65536)}
    ex = ipc.exchange(local)
    opened = []

    def opener(h):
        opened.append(h)
        return 0x10_0000_0000 * (h[0] + 1)  # a distinct fake base per peer

    closed = []
    peers = ipc.PeerMap(opener=opener, closer=closed.append)
    own_arena, own_buf = 0xAA000, 0xBB000
    arenas = ipc.rank_addresses(ex, rank, "grads", own_arena, peers)
    bufs = ipc.rank_addresses(ex, rank, "gathered", own_buf, peers)
    table = ipc.grad_table(arenas, offs)
    peers.close()
    out[rank] = dict(ex=ex, opened=opened, closed=closed, arenas=arenas, bufs=bufs, table=table,
                     offs=offs, total=total)
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_and_tables(world):
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        x = res[r]
        assert [e["grads"][0][0] for e in x["ex"]] == list(range(world)), "rank order of the exchange"
        # each peer's allocation opened once, its own never
        assert sorted(h[0] for h in x["opened"]) == [k for k in range(world) if k != r]
        assert len(x["closed"]) == world - 1
        for k in range(world):
            base = 0x10_0000_0000 * (k + 1)
            assert x["arenas"][k] == (0xAA000 if k == r else base + 4096)
            assert x["bufs"][k] == (0xBB000 if k == r else base + 65536)
        # rank-major N*P table, each entry arena base + parameter offset
        P = len(x["offs"])
        assert len(x["table"]) == world * P
        for k in range(world):
            for p in range(P):
                assert x["table"][k * P + p] == x["arenas"][k] + x["offs"][p]
        assert x["offs"] == [0, 16, 32, 32] and x["total"] == 64  # 16-byte starts, same on every rank
        assert x["offs"] == res[0]["offs"]
