"""ctypes binding of libtide.so (declared in include/tide.h).

Argument marshalling only: every step of the reduce-scatter and placement
runs in the library's CUDA kernels (or, for copy-engine placement, in CUDA
copies the library enqueues).  There is no Python or CPU fallback: if the
library is missing, importing this module raises.

Pointer arguments accept ints (raw device addresses), objects with a
``data_ptr()`` method (e.g. torch tensors), or a prebuilt ``PointerTable``.
Streams accept ints (cudaStream_t values), objects with a ``cuda_stream``
attribute (e.g. torch.cuda.Stream), or None for the legacy default stream.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# TIDE_LIBRARY=debug loads the build whose kernels range-check every tile
# (libtide_debug.so); anything else loads the release library.
LIB_PATH = os.path.join(_HERE, "libtide_debug.so" if os.environ.get("TIDE_LIBRARY") == "debug" else "libtide.so")

TIDE_OK = 0
TIDE_ERR_INVALID_ARG = 1
TIDE_ERR_MISALIGNED = 2
TIDE_ERR_UNSUPPORTED = 3
TIDE_ERR_CUDA = 4
TIDE_ERR_TIMEOUT = 5
TIDE_ERR_OUT_OF_MEMORY = 6
TIDE_ERR_RANGE = 7

TIDE_MODE_UNCAPPED = 0
TIDE_MODE_CAPPED = 1
TIDE_MODE_COPY_ENGINE = 2
TIDE_MODE_BULK = 3

TIDE_OP_RS = 0
TIDE_OP_AG = 1
TIDE_OP_PACK = 2
TIDE_OP_STAGE = 3
TIDE_OP_STAGED_RS = 4

TIDE_MAX_RANKS = 4096
TIDE_IPC_HANDLE_BYTES = 64
TIDE_NOALLOC_SCRATCH_BYTES = 4 << 20

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python __graft_entry__.py` "
                      "(the CUDA library is required; there is no fallback)")

_lib = ctypes.CDLL(LIB_PATH)
_vp = ctypes.c_void_p
_st = ctypes.c_int
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("tide_layout_create", _st, ctypes.c_int32, _vp, _vp, ctypes.c_int32, ctypes.POINTER(_vp))
_sig("tide_layout_create_ex", _st, ctypes.c_int32, _vp, _vp, ctypes.c_int32, ctypes.c_int64,
     ctypes.POINTER(_vp))
_sig("tide_layout_destroy", None, _vp)
_sig("tide_layout_num_params", _st, _vp, _i32p)
_sig("tide_layout_num_ranks", _st, _vp, _i32p)
_sig("tide_layout_rank_block_numel", _st, _vp, _i64p)
_sig("tide_layout_shard_numel", _st, _vp, ctypes.c_int32, _i64p)
_sig("tide_layout_param_offset", _st, _vp, ctypes.c_int32, _i64p)
_sig("tide_layout_valid_rows", _st, _vp, ctypes.c_int32, ctypes.c_int32, _i64p)
_sig("tide_layout_chunk_rows", _st, _vp, ctypes.c_int32, _i64p)
_sig("tide_layout_set_mode", _st, _vp, ctypes.c_int, ctypes.c_int32)
_sig("tide_layout_get_mode", _st, _vp, _i32p, _i32p)
_sig("tide_layout_launch_shape", _st, _vp, ctypes.c_int, _i32p, _i32p)
_sig("tide_layout_tiles", _st, _vp, ctypes.c_int, _vp, ctypes.c_int64, _i64p)
_sig("tide_rs_bf16_to_fp32", _st, _vp, _vp, _vp, ctypes.c_float, _vp)
_sig("tide_ag_place", _st, _vp, _vp, _vp, _vp)
_sig("tide_rs_bf16_to_fp32_noalloc", _st, _vp, _vp, _vp, ctypes.c_float, _vp)
_sig("tide_rs_bf16_to_fp32_rank", _st, _vp, ctypes.c_int32, _vp, _vp, ctypes.c_float, _vp)
_sig("tide_ag_place_ranks", _st, _vp, _vp, _vp, _vp)
_sig("tide_ag_pack_bf16", _st, _vp, ctypes.c_int32, _vp, _vp, _vp)
_sig("tide_rs_stage_bf16", _st, _vp, _vp, _vp, _vp)
_sig("tide_rs_staged_bf16_to_fp32", _st, _vp, _vp, _vp, ctypes.c_float, _vp)
_sig("tide_layout_check_device", _st, _vp)
_sig("tide_layout_set_test_stall", _st, _vp, ctypes.c_int64)
_sig("tide_ipc_export", _st, _vp, _vp, ctypes.POINTER(ctypes.c_uint64))
_sig("tide_ipc_open", _st, _vp, ctypes.POINTER(_vp))
_sig("tide_ipc_close", _st, _vp)
_sig("tide_layout_check_tiles", _st, _vp, ctypes.c_int, _vp, ctypes.c_int64, _i64p)
_sig("tide_build_info", ctypes.c_char_p)
_sig("tide_status_string", ctypes.c_char_p, _st)
_sig("tide_last_error", ctypes.c_char_p)


class TideError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.tide_last_error().decode(errors="replace")
        super().__init__(f"{where}: {tide_status_string(status)}" + (f" — {msg}" if msg else ""))


def _check(status: int, where: str) -> None:
    if status != TIDE_OK:
        raise TideError(status, where)


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int:
    if s is None:
        return 0
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


class PointerTable:
    """A host array of device pointers, built once and reused across calls."""

    def __init__(self, items):
        addrs = [_addr(x) for x in items]
        self.n = len(addrs)
        self.array = (ctypes.c_void_p * max(1, self.n))(*addrs)
        self.keep = list(items)  # keep tensors alive while the table exists

    @property
    def ptr(self) -> int:
        return ctypes.addressof(self.array)


def _table(x) -> PointerTable | None:
    """A PointerTable for x; the caller keeps it referenced across the C call
    so the host array outlives the library's read of it."""
    if x is None:
        return None
    return x if isinstance(x, PointerTable) else PointerTable(x)


def _tptr(t: PointerTable | None) -> int:
    return t.ptr if t is not None and t.n else 0


def tide_layout_check_device(layout) -> None:
    """Raises TideError(TIDE_ERR_TIMEOUT) if a bounded device wait ran out."""
    _check(_lib.tide_layout_check_device(layout), "tide_layout_check_device")


def tide_layout_set_test_stall(layout, ns: int) -> None:
    _check(_lib.tide_layout_set_test_stall(layout, ns), "tide_layout_set_test_stall")


def tide_layout_check_tiles(layout, op: int, rows) -> int:
    """Index of the first tile of `rows` ((n, 6) int64, as tide_layout_tiles
    returns) that fails the kernels' range test, or -1."""
    r = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 6)
    bad = ctypes.c_int64(0)
    _check(_lib.tide_layout_check_tiles(layout, op, r.ctypes.data if r.size else 0, r.shape[0],
                                        ctypes.byref(bad)), "tide_layout_check_tiles")
    return bad.value


def tide_ipc_export(ptr) -> tuple[bytes, int]:
    """(IPC handle of the allocation holding ptr, byte offset of ptr in it)."""
    h = (ctypes.c_uint8 * TIDE_IPC_HANDLE_BYTES)()
    off = ctypes.c_uint64(0)
    _check(_lib.tide_ipc_export(_addr(ptr), h, ctypes.byref(off)), "tide_ipc_export")
    return bytes(h), off.value


def tide_ipc_open(handle: bytes) -> int:
    """Base address of a peer's exported allocation mapped into this process."""
    if len(handle) != TIDE_IPC_HANDLE_BYTES:
        raise ValueError("an IPC handle is 64 bytes")
    h = (ctypes.c_uint8 * TIDE_IPC_HANDLE_BYTES).from_buffer_copy(handle)
    base = ctypes.c_void_p(0)
    _check(_lib.tide_ipc_open(h, ctypes.byref(base)), "tide_ipc_open")
    return base.value


def tide_ipc_close(base: int) -> None:
    _check(_lib.tide_ipc_close(base), "tide_ipc_close")


def tide_build_info() -> str:
    return _lib.tide_build_info().decode()


def tide_status_string(status: int) -> str:
    return _lib.tide_status_string(status).decode()


def tide_last_error() -> str:
    return _lib.tide_last_error().decode(errors="replace")


def _shape_arrays(shapes):
    nd = np.asarray([len(s) for s in shapes], dtype=np.int32)
    flat = np.asarray([int(d) for s in shapes for d in s], dtype=np.int64)
    return nd, flat


def tide_layout_create(shapes, num_ranks: int, align_elems: int | None = None) -> int:
    """Layout handle for parameters of the given shapes over num_ranks ranks."""
    nd, flat = _shape_arrays(shapes)
    out = ctypes.c_void_p(0)
    nd_p = nd.ctypes.data if nd.size else 0
    fl_p = flat.ctypes.data if flat.size else 0
    if align_elems is None:
        st = _lib.tide_layout_create(len(shapes), nd_p, fl_p, num_ranks, ctypes.byref(out))
    else:
        st = _lib.tide_layout_create_ex(len(shapes), nd_p, fl_p, num_ranks, align_elems,
                                        ctypes.byref(out))
    _check(st, "tide_layout_create")
    return out.value


def tide_layout_destroy(layout: int) -> None:
    _lib.tide_layout_destroy(layout)


def _q64(fn, *args):
    v = ctypes.c_int64(0)
    _check(getattr(_lib, fn)(*args, ctypes.byref(v)), fn)
    return v.value


def _q32(fn, *args):
    v = ctypes.c_int32(0)
    _check(getattr(_lib, fn)(*args, ctypes.byref(v)), fn)
    return v.value


def tide_layout_num_params(layout) -> int:
    return _q32("tide_layout_num_params", layout)


def tide_layout_num_ranks(layout) -> int:
    return _q32("tide_layout_num_ranks", layout)


def tide_layout_rank_block_numel(layout) -> int:
    return _q64("tide_layout_rank_block_numel", layout)


def tide_layout_shard_numel(layout, p: int) -> int:
    return _q64("tide_layout_shard_numel", layout, p)


def tide_layout_param_offset(layout, p: int) -> int:
    return _q64("tide_layout_param_offset", layout, p)


def tide_layout_valid_rows(layout, p: int, r: int) -> int:
    return _q64("tide_layout_valid_rows", layout, p, r)


def tide_layout_chunk_rows(layout, p: int) -> int:
    return _q64("tide_layout_chunk_rows", layout, p)


def tide_layout_set_mode(layout, mode: int, cta_cap: int = 0) -> None:
    _check(_lib.tide_layout_set_mode(layout, mode, cta_cap), "tide_layout_set_mode")


def tide_layout_get_mode(layout):
    """(mode, cta_cap) of the layout."""
    m, c = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(_lib.tide_layout_get_mode(layout, ctypes.byref(m), ctypes.byref(c)), "tide_layout_get_mode")
    return m.value, c.value


def tide_layout_launch_shape(layout, op: int):
    g, b = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(_lib.tide_layout_launch_shape(layout, op, ctypes.byref(g), ctypes.byref(b)),
           "tide_layout_launch_shape")
    return g.value, b.value


def tide_layout_tiles(layout, op: int) -> np.ndarray:
    """(count, 6) int64 array: param, rank, src_offset, dst_offset, length, flags."""
    n = ctypes.c_int64(0)
    _check(_lib.tide_layout_tiles(layout, op, 0, 0, ctypes.byref(n)), "tide_layout_tiles")
    rows = np.zeros((max(1, n.value), 6), dtype=np.int64)
    _check(_lib.tide_layout_tiles(layout, op, rows.ctypes.data, n.value, ctypes.byref(n)),
           "tide_layout_tiles")
    return rows[: n.value]


def tide_rs_bf16_to_fp32(layout, grads, shards, scale: float, stream=None) -> None:
    """grads: N*P rank-major bf16 gradient pointers; shards: N*P fp32 shard pointers."""
    g, s = _table(grads), _table(shards)
    _check(_lib.tide_rs_bf16_to_fp32(layout, _tptr(g), _tptr(s), scale, _stream(stream)),
           "tide_rs_bf16_to_fp32")


def tide_rs_bf16_to_fp32_noalloc(layout, grads, shards, scale: float, stream=None) -> None:
    """As tide_rs_bf16_to_fp32, for callers that cannot allocate device memory:
    the kernel's tables go into the library's fixed 4 MiB device array."""
    g, s = _table(grads), _table(shards)
    _check(_lib.tide_rs_bf16_to_fp32_noalloc(layout, _tptr(g), _tptr(s), scale, _stream(stream)),
           "tide_rs_bf16_to_fp32_noalloc")


def tide_rs_bf16_to_fp32_rank(layout, rank: int, grads, shards, scale: float, stream=None) -> None:
    """grads: N*P rank-major pointers; shards: the P fp32 shards of rank `rank`."""
    g, s = _table(grads), _table(shards)
    _check(_lib.tide_rs_bf16_to_fp32_rank(layout, rank, _tptr(g), _tptr(s), scale, _stream(stream)),
           "tide_rs_bf16_to_fp32_rank")


def tide_ag_pack_bf16(layout, rank: int, shards, gathered, stream=None) -> None:
    """rank >= 0: shards = that rank's P fp32 shards; rank == -1: all N*P."""
    s = _table(shards)
    _check(_lib.tide_ag_pack_bf16(layout, rank, _tptr(s), _addr(gathered), _stream(stream)),
           "tide_ag_pack_bf16")


def tide_rs_stage_bf16(layout, grads, slot, stream=None) -> None:
    """grads: one rank's P bf16 gradients; slot: that rank's N*S bf16 buffer."""
    g = _table(grads)
    _check(_lib.tide_rs_stage_bf16(layout, _tptr(g), _addr(slot), _stream(stream)),
           "tide_rs_stage_bf16")


def tide_rs_staged_bf16_to_fp32(layout, slots, shards, scale: float, stream=None) -> None:
    """slots: N staged slot buffers; shards: N*P fp32 shard pointers."""
    a, b = _table(slots), _table(shards)
    _check(_lib.tide_rs_staged_bf16_to_fp32(layout, _tptr(a), _tptr(b), scale, _stream(stream)),
           "tide_rs_staged_bf16_to_fp32")


def tide_ag_place(layout, gathered, params, stream=None) -> None:
    """gathered: N*S bf16 rank-major buffer; params: P bf16 parameter pointers."""
    t = _table(params)
    _check(_lib.tide_ag_place(layout, _addr(gathered), _tptr(t), _stream(stream)), "tide_ag_place")


def tide_ag_place_ranks(layout, gathered, params, stream=None) -> None:
    """gathered: N rank-major bf16 buffers (block k read from buffer k); params: P pointers."""
    g, t = _table(gathered), _table(params)
    _check(_lib.tide_ag_place_ranks(layout, _tptr(g), _tptr(t), _stream(stream)), "tide_ag_place_ranks")


def exported_symbols():
    """Names of the ABI functions this binding resolved (for load checks)."""
    return [n for n in dir(_lib) if n.startswith("tide_")]
