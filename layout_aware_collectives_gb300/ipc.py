"""Rank processes over peer memory: one process per rank.

Set-up plumbing around the library (no data moves through it): each rank
process keeps its per-parameter bf16 gradients in one arena and its
rank-major buffer in another, exports both (tide_ipc_export), the handles
are exchanged over torch.distributed (all_gather_object; any backend, gloo
suffices), and every peer allocation is mapped once (tide_ipc_open).  Rank r
then runs the library's kernels on pointer tables that mix its own
addresses with its peers' mapped ones:

  reduce-scatter  tide_rs_bf16_to_fp32_rank(r, grads = every rank's gradients)
  all-gather      tide_ag_pack_bf16(r) into its own block, a barrier, then
                  tide_ag_place_ranks(gathered = every rank's buffer)

("FSDP通信终局：TIDE零拷贝集合通信优化" §TIDE的设计思路: TIDE-RS reads the
per-parameter gradients directly, TIDE-AG places shards straight into
parameter storage.)
"""
from __future__ import annotations

from . import tide as _t

ALIGN_BYTES = 16


def arena_offsets(numels, elem_bytes: int, align: int = ALIGN_BYTES):
    """Byte offsets of tensors of `numels` elements packed into one arena,
    each starting on `align` bytes, and the arena's size in bytes.  Every
    rank computes the same offsets from the same shapes, so a peer's tensor
    is its arena's base plus the local offset."""
    offs, pos = [], 0
    for n in numels:
        offs.append(pos)
        pos += -(-int(n) * elem_bytes // align) * align
    return offs, max(pos, align)


def exchange(local: dict, group=None) -> list:
    """Every rank's {name: (handle bytes, offset)} in rank order."""
    import torch.distributed as dist

    out = [None] * dist.get_world_size(group)
    dist.all_gather_object(out, local, group=group)
    return out


class PeerMap:
    """Peer allocations mapped into this process, each handle opened once."""

    def __init__(self, opener=None, closer=None):
        self._open = opener or _t.tide_ipc_open
        self._close = closer or _t.tide_ipc_close
        self.bases = {}

    def address(self, handle: bytes, offset: int) -> int:
        base = self.bases.get(handle)
        if base is None:
            base = self._open(handle)
            self.bases[handle] = base
        return base + offset

    def close(self) -> None:
        for base in self.bases.values():
            self._close(base)
        self.bases = {}


def rank_addresses(exchanged: list, rank: int, name: str, local_address: int, peers: PeerMap) -> list:
    """Address of buffer `name` of every rank as seen from `rank`: its own
    address for itself, the mapped peer address for the others."""
    return [local_address if k == rank else peers.address(*exchanged[k][name])
            for k in range(len(exchanged))]


def grad_table(arena_addresses: list, offsets: list) -> list:
    """Rank-major table of N*P gradient addresses: rank k's gradient of
    parameter p at its arena base plus the parameter's offset."""
    return [a + o for a in arena_addresses for o in offsets]
