"""ctypes wrapper of the CPU oracle (liboracle.so, built from tide_oracle.c).

TEST INFRASTRUCTURE.  Only tests/, the smoke check and the benchmark's
CPU-baseline / reference leg may import this package.  The product library
and its Python binding never import it and never fall back to it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboracle.so")
MAX_RANKS = 4096
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.oracle_chunk_rows.restype = ctypes.c_int64
        L.oracle_chunk_rows.argtypes = [ctypes.c_int64, ctypes.c_int32]
        L.oracle_valid_rows.restype = ctypes.c_int64
        L.oracle_valid_rows.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
        L.oracle_layout.restype = ctypes.c_int
        L.oracle_layout.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, _i64p]
        L.oracle_rs_element.restype = ctypes.c_float
        L.oracle_rs_element.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_float]
        L.oracle_rs.restype = ctypes.c_int
        L.oracle_rs.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float]
        L.oracle_ag_place.restype = None
        L.oracle_ag_place.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_ag_source_index.restype = ctypes.c_int64
        L.oracle_ag_source_index.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int64]
        L.oracle_rs_rank.restype = ctypes.c_int
        L.oracle_rs_rank.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_float, ctypes.c_int32]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_ag_pack.restype = None
        L.oracle_ag_pack.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                     ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_rs_stage.restype = None
        L.oracle_rs_stage.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_rs_staged.restype = ctypes.c_int
        L.oracle_rs_staged.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float]
        _lib = L
    return _lib


def _dims(shapes):
    d0, inner = [], []
    for s in shapes:
        if len(s) == 0:
            d0.append(1)
            inner.append(1)
            continue
        n = 1
        for d in s[1:]:
            n *= int(d)
        d0.append(int(s[0]))
        inner.append(n)
    return np.asarray(d0, dtype=np.int64), np.asarray(inner, dtype=np.int64)


def _check_ranks(num_ranks: int) -> None:
    """The C oracle gathers one element's N inputs into a 4096-entry stack
    array and refuses larger N; refuse here too, with a clear message."""
    if not 1 <= num_ranks <= MAX_RANKS:
        raise ValueError(f"oracle supports 1 .. {MAX_RANKS} ranks, got {num_ranks}")


def _rc(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"{what} refused its arguments")


def _ptrs(arrays):
    return np.asarray([a.ctypes.data for a in arrays], dtype=np.uint64)


def chunk_rows(d0: int, n: int) -> int:
    return lib().oracle_chunk_rows(d0, n)


def valid_rows(d0: int, n: int, r: int) -> int:
    return lib().oracle_valid_rows(d0, n, r)


def layout(shapes, num_ranks: int, align: int = 8):
    """(offsets[P], S) of the rank-major block layout."""
    d0, inner = _dims(shapes)
    offs = np.zeros(max(len(shapes), 1), dtype=np.int64)
    S = ctypes.c_int64(0)
    rc = lib().oracle_layout(len(shapes), d0.ctypes.data, inner.ctypes.data, num_ranks, align,
                             offs.ctypes.data, ctypes.byref(S))
    if rc:
        raise ValueError("oracle_layout rejected its arguments")
    return offs[: len(shapes)].copy(), S.value


def shard_numel(shape, num_ranks: int) -> int:
    d0, inner = _dims([shape])
    return chunk_rows(int(d0[0]), num_ranks) * int(inner[0])


def rs_element(vals_bf16: np.ndarray, scale: float) -> float:
    v = np.ascontiguousarray(vals_bf16, dtype=np.uint16)
    return lib().oracle_rs_element(v.size, v.ctypes.data, scale)


def rs(shapes, num_ranks: int, grads, scale: float):
    """grads[k][p]: uint16 arrays (bf16 bits).  Returns shards[r][p] fp32 arrays."""
    _check_ranks(num_ranks)
    P = len(shapes)
    d0, inner = _dims(shapes)
    g = [np.ascontiguousarray(grads[k][p], dtype=np.uint16)
         for k in range(num_ranks) for p in range(P)]
    shards = [[np.empty(chunk_rows(int(d0[p]), num_ranks) * int(inner[p]), dtype=np.float32)
               for p in range(P)] for _ in range(num_ranks)]
    flat_out = [shards[r][p] for r in range(num_ranks) for p in range(P)]
    gp, op = _ptrs(g), _ptrs(flat_out)
    _rc(lib().oracle_rs(num_ranks, P, d0.ctypes.data, inner.ctypes.data, gp.ctypes.data,
                        op.ctypes.data, scale), "oracle_rs")
    return shards


def ag_place(shapes, num_ranks: int, gathered: np.ndarray, offsets, block_numel: int):
    """Returns params[p] (uint16 bf16 bits) placed from the rank-major buffer."""
    P = len(shapes)
    d0, inner = _dims(shapes)
    buf = np.ascontiguousarray(gathered, dtype=np.uint16)
    assert buf.size >= num_ranks * block_numel
    offs = np.ascontiguousarray(offsets, dtype=np.int64)
    params = [np.empty(int(d0[p]) * int(inner[p]), dtype=np.uint16) for p in range(P)]
    pp = _ptrs(params)
    lib().oracle_ag_place(num_ranks, P, d0.ctypes.data, inner.ctypes.data, offs.ctypes.data,
                          block_numel, buf.ctypes.data, pp.ctypes.data)
    return params


def ag_source_index(num_ranks, shape, offset, block_numel, i, j) -> int:
    d0, inner = _dims([shape])
    return lib().oracle_ag_source_index(num_ranks, int(d0[0]), int(inner[0]), offset,
                                        block_numel, i, j)


def rs_rank(shapes, num_ranks: int, grads, scale: float, r: int):
    """Rank r's shards only: list of P fp32 arrays."""
    _check_ranks(num_ranks)
    if not 0 <= r < num_ranks:
        raise ValueError(f"rank {r} out of range")
    P = len(shapes)
    d0, inner = _dims(shapes)
    g = [np.ascontiguousarray(grads[k][p], dtype=np.uint16)
         for k in range(num_ranks) for p in range(P)]
    out = [np.empty(chunk_rows(int(d0[p]), num_ranks) * int(inner[p]), dtype=np.float32)
           for p in range(P)]
    gp, op = _ptrs(g), _ptrs(out)
    _rc(lib().oracle_rs_rank(num_ranks, P, d0.ctypes.data, inner.ctypes.data, gp.ctypes.data,
                             op.ctypes.data, scale, r), "oracle_rs_rank")
    return out


def f32_to_bf16(x) -> np.ndarray:
    """Element-wise fp32 -> bf16 bits by the oracle's rounding."""
    bits = np.ascontiguousarray(x, dtype=np.float32).ravel().view(np.uint32)
    f = lib().oracle_f32_to_bf16
    # pass the exact fp32 bits (a round trip through a Python float would
    # quieten signalling NaNs before the oracle sees them)
    return np.array([f(ctypes.c_float.from_buffer_copy(int(b).to_bytes(4, "little")))
                     for b in bits], dtype=np.uint16)


def ag_pack(shapes, num_ranks: int, offsets, block_numel: int, r: int, shards_r, gathered):
    """Writes rank r's block of `gathered` (uint16 array, modified in place)."""
    P = len(shapes)
    d0, inner = _dims(shapes)
    src = [np.ascontiguousarray(shards_r[p], dtype=np.float32) for p in range(P)]
    offs = np.ascontiguousarray(offsets, dtype=np.int64)
    assert gathered.dtype == np.uint16 and gathered.flags.c_contiguous
    sp = _ptrs(src)
    lib().oracle_ag_pack(num_ranks, P, d0.ctypes.data, inner.ctypes.data, offs.ctypes.data,
                         block_numel, r, sp.ctypes.data, gathered.ctypes.data)
    return gathered


def rs_stage(shapes, num_ranks: int, offsets, block_numel: int, grads_k, slot):
    """Writes rank k's gradients into `slot` (uint16, N*S, modified in place)."""
    P = len(shapes)
    d0, inner = _dims(shapes)
    g = [np.ascontiguousarray(grads_k[p], dtype=np.uint16) for p in range(P)]
    offs = np.ascontiguousarray(offsets, dtype=np.int64)
    assert slot.dtype == np.uint16 and slot.flags.c_contiguous
    gp = _ptrs(g)
    lib().oracle_rs_stage(num_ranks, P, d0.ctypes.data, inner.ctypes.data, offs.ctypes.data,
                          block_numel, gp.ctypes.data, slot.ctypes.data)
    return slot


def rs_staged(shapes, num_ranks: int, offsets, block_numel: int, slots, scale: float):
    """Reduce-scatter from N staged slots; returns shards[r][p]."""
    _check_ranks(num_ranks)
    P = len(shapes)
    d0, inner = _dims(shapes)
    sl = [np.ascontiguousarray(x, dtype=np.uint16) for x in slots]
    offs = np.ascontiguousarray(offsets, dtype=np.int64)
    shards = [[np.empty(chunk_rows(int(d0[p]), num_ranks) * int(inner[p]), dtype=np.float32)
               for p in range(P)] for _ in range(num_ranks)]
    flat = [shards[r][p] for r in range(num_ranks) for p in range(P)]
    sp, op = _ptrs(sl), _ptrs(flat)
    _rc(lib().oracle_rs_staged(num_ranks, P, d0.ctypes.data, inner.ctypes.data, offs.ctypes.data,
                               block_numel, sp.ctypes.data, op.ctypes.data, scale), "oracle_rs_staged")
    return shards
