"""Owning wrapper around a tide_layout_t handle (marshalling only)."""
from __future__ import annotations

from . import tide as _t


class Layout:
    """Layout of `shapes` sharded over `num_ranks` ranks; see include/tide.h."""

    def __init__(self, shapes, num_ranks: int, align_elems: int | None = None):
        self.shapes = [tuple(int(d) for d in s) for s in shapes]
        self.handle = _t.tide_layout_create(self.shapes, num_ranks, align_elems)

    # -------- queries
    @property
    def num_params(self) -> int:
        return _t.tide_layout_num_params(self.handle)

    @property
    def num_ranks(self) -> int:
        return _t.tide_layout_num_ranks(self.handle)

    @property
    def block_numel(self) -> int:
        return _t.tide_layout_rank_block_numel(self.handle)

    def shard_numel(self, p: int) -> int:
        return _t.tide_layout_shard_numel(self.handle, p)

    def param_offset(self, p: int) -> int:
        return _t.tide_layout_param_offset(self.handle, p)

    def valid_rows(self, p: int, r: int) -> int:
        return _t.tide_layout_valid_rows(self.handle, p, r)

    def chunk_rows(self, p: int) -> int:
        return _t.tide_layout_chunk_rows(self.handle, p)

    def tiles(self, op: int):
        return _t.tide_layout_tiles(self.handle, op)

    def check_tiles(self, op: int, rows) -> int:
        return _t.tide_layout_check_tiles(self.handle, op, rows)

    def launch_shape(self, op: int):
        return _t.tide_layout_launch_shape(self.handle, op)

    def get_mode(self):
        return _t.tide_layout_get_mode(self.handle)

    def set_mode(self, mode: int, cta_cap: int = 0) -> None:
        _t.tide_layout_set_mode(self.handle, mode, cta_cap)

    def check_device(self) -> None:
        _t.tide_layout_check_device(self.handle)

    def set_test_stall(self, ns: int) -> None:
        _t.tide_layout_set_test_stall(self.handle, ns)

    # -------- compute
    def reduce_scatter(self, grads, shards, scale: float, stream=None) -> None:
        _t.tide_rs_bf16_to_fp32(self.handle, grads, shards, scale, stream)

    def reduce_scatter_noalloc(self, grads, shards, scale: float, stream=None) -> None:
        _t.tide_rs_bf16_to_fp32_noalloc(self.handle, grads, shards, scale, stream)

    def reduce_scatter_rank(self, rank: int, grads, shards, scale: float, stream=None) -> None:
        _t.tide_rs_bf16_to_fp32_rank(self.handle, rank, grads, shards, scale, stream)

    def pack(self, rank: int, shards, gathered, stream=None) -> None:
        _t.tide_ag_pack_bf16(self.handle, rank, shards, gathered, stream)

    def stage(self, grads, slot, stream=None) -> None:
        _t.tide_rs_stage_bf16(self.handle, grads, slot, stream)

    def reduce_scatter_staged(self, slots, shards, scale: float, stream=None) -> None:
        _t.tide_rs_staged_bf16_to_fp32(self.handle, slots, shards, scale, stream)

    def place(self, gathered, params, stream=None) -> None:
        _t.tide_ag_place(self.handle, gathered, params, stream)

    def place_ranks(self, gathered, params, stream=None) -> None:
        _t.tide_ag_place_ranks(self.handle, gathered, params, stream)

    # -------- lifetime
    def close(self) -> None:
        if getattr(self, "handle", None):
            _t.tide_layout_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
