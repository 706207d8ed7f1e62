"""C ABI on the CPU: the library loads and exports every declared symbol, the
host layout descriptor agrees with the oracle, the tile lists partition the
outputs exactly, and invalid arguments come back as error codes.  No call
here launches device work."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import layout_aware_collectives_gb300 as tide
from layout_aware_collectives_gb300 import tide as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"^TIDE_API [^(]*?\b(tide_\w+)\(", src, re.M))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 17, names
    lib = ctypes.CDLL(T.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    for st in range(7):
        assert tide.tide_status_string(st).startswith("TIDE_")
    assert "unknown" in tide.tide_status_string(99)


def _rand_shapes(rng, k):
    shapes = []
    for _ in range(k):
        nd = int(rng.integers(0, 4))
        shapes.append(tuple(int(rng.integers(0, 40)) for _ in range(nd)))
    return shapes


@pytest.mark.parametrize("seed", range(8))
def test_layout_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.choice([1, 2, 3, 4, 7, 8, 16, 64]))
    align = int(rng.choice([1, 2, 8, 16]))
    shapes = _rand_shapes(rng, int(rng.integers(0, 12)))
    offs, S = oracle.layout(shapes, n, align)
    with tide.Layout(shapes, n, align_elems=align) as lay:
        assert lay.num_params == len(shapes) and lay.num_ranks == n
        assert lay.block_numel == S
        for p, s in enumerate(shapes):
            d0 = s[0] if s else 1
            assert lay.param_offset(p) == offs[p]
            assert lay.chunk_rows(p) == oracle.chunk_rows(d0, n)
            assert lay.shard_numel(p) == oracle.shard_numel(s, n)
            for r in range(n):
                assert lay.valid_rows(p, r) == oracle.valid_rows(d0, n, r)


def _dims(s):
    if not s:
        return 1, 1
    inner = 1
    for d in s[1:]:
        inner *= d
    return s[0], inner


@pytest.mark.parametrize("n,shapes,align", [
    (4, [(256, 256), (704, 256), (256, 704), (250,)], 8),
    (3, [(5, 3), (1,), (), (0, 4), (17, 9)], 1),
    (16, [(100000, 3)], 8),
    (64, [(1000, 4096), (63, 4096)], 8),
    (8, [(70000, 1)], 2),
])
def test_tiles_partition_outputs(n, shapes, align):
    offs, S = oracle.layout(shapes, n, align)
    with tide.Layout(shapes, n, align_elems=align) as lay:
        rs = lay.tiles(tide.TIDE_OP_RS)
        ag = lay.tiles(tide.TIDE_OP_AG)
    # reduce-scatter: every shard element written by exactly one tile, reading
    # the same element offset of the full gradient; padding by zero tiles
    cover = {}
    for p, r, src, dst, ln, flags in rs:
        d0, inner = _dims(shapes[p])
        c = oracle.chunk_rows(d0, n)
        cnt = cover.setdefault((p, r), np.zeros(c * inner, dtype=np.int64))
        cnt[dst: dst + ln] += 1
        v = oracle.valid_rows(d0, n, r) * inner
        if flags & 1:
            assert dst >= v and dst + ln <= c * inner
        else:
            assert dst + ln <= v and src == r * c * inner + dst
            if flags & 2:
                assert src % 8 == 0 and dst % 4 == 0
        assert ln > 0
    for p, s in enumerate(shapes):
        d0, inner = _dims(s)
        c = oracle.chunk_rows(d0, n)
        for r in range(n):
            if c * inner:
                assert np.all(cover[(p, r)] == 1), (p, r)
    # placement: every parameter element written once, from the oracle's source index
    seen = [np.zeros(_dims(s)[0] * _dims(s)[1], dtype=np.int64) for s in shapes]
    for p, r, src, dst, ln, flags in ag:
        d0, inner = _dims(shapes[p])
        seen[p][dst: dst + ln] += 1
        for e in (dst, dst + ln - 1):
            assert src + (e - dst) == oracle.ag_source_index(n, shapes[p], offs[p], S,
                                                             e // inner, e % inner)
        if flags & 2:
            assert src % 8 == 0 and dst % 8 == 0
    for p in range(len(shapes)):
        assert np.all(seen[p] == 1), p


def _st(fn, *args):
    return getattr(T._lib, fn)(*args)


def test_create_rejects_bad_arguments():
    out = ctypes.c_void_p(0)
    nd = (ctypes.c_int32 * 1)(2)
    dims = (ctypes.c_int64 * 2)(4, 4)
    INV = tide.TIDE_ERR_INVALID_ARG
    assert _st("tide_layout_create", 1, nd, dims, 0, ctypes.byref(out)) == INV
    assert _st("tide_layout_create", 1, nd, dims, 4097, ctypes.byref(out)) == INV
    assert _st("tide_layout_create", -1, nd, dims, 4, ctypes.byref(out)) == INV
    assert _st("tide_layout_create", 1, None, dims, 4, ctypes.byref(out)) == INV
    assert _st("tide_layout_create", 1, nd, None, 4, ctypes.byref(out)) == INV
    assert _st("tide_layout_create", 1, nd, dims, 4, None) == INV
    neg = (ctypes.c_int64 * 2)(4, -1)
    assert _st("tide_layout_create", 1, nd, neg, 4, ctypes.byref(out)) == INV
    big = (ctypes.c_int64 * 2)(1 << 40, 1 << 40)
    assert _st("tide_layout_create", 1, nd, big, 4, ctypes.byref(out)) == INV
    assert "overflow" in tide.tide_last_error()
    for a in (0, 3, 8192):
        assert _st("tide_layout_create_ex", 1, nd, dims, 4, a, ctypes.byref(out)) == INV
    assert out.value is None


def test_queries_and_modes_reject_bad_arguments():
    INV = tide.TIDE_ERR_INVALID_ARG
    v = ctypes.c_int64(0)
    with tide.Layout([(8, 2)], 4) as lay:
        h = lay.handle
        assert _st("tide_layout_shard_numel", h, 1, ctypes.byref(v)) == INV
        assert _st("tide_layout_shard_numel", h, -1, ctypes.byref(v)) == INV
        assert _st("tide_layout_valid_rows", h, 0, 4, ctypes.byref(v)) == INV
        assert _st("tide_layout_param_offset", h, 0, None) == INV
        assert _st("tide_layout_set_mode", h, 7, 0) == INV
        assert _st("tide_layout_set_mode", h, tide.TIDE_MODE_CAPPED, 0) == INV
        assert _st("tide_layout_set_mode", h, tide.TIDE_MODE_CAPPED, 3) == tide.TIDE_OK
    assert _st("tide_layout_rank_block_numel", None, ctypes.byref(v)) == INV
    T._lib.tide_layout_destroy(None)  # no-op


def test_compute_calls_validate_before_touching_the_device():
    """Null and misaligned pointers are refused on the host, before any CUDA
    call, so these run without a GPU (addresses are never dereferenced)."""
    shapes = [(8, 2), (5,)]
    with tide.Layout(shapes, 2) as lay:
        good = 0x10000
        grads = [good + 0x1000 * i for i in range(4)]
        shards = [good + 0x8000 + 0x1000 * i for i in range(4)]
        with pytest.raises(tide.TideError) as e:
            lay.reduce_scatter(grads[:3] + [good + 2], shards, 0.5)
        assert e.value.status == tide.TIDE_ERR_MISALIGNED
        with pytest.raises(tide.TideError) as e:
            lay.reduce_scatter(grads, shards[:1] + [0] + shards[2:], 0.5)
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
        with pytest.raises(tide.TideError) as e:
            lay.place(good + 8, [good, good], None)
        assert e.value.status == tide.TIDE_ERR_MISALIGNED
        with pytest.raises(tide.TideError) as e:
            lay.place(good, [good, None], None)
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
        lay.set_mode(tide.TIDE_MODE_COPY_ENGINE)
        with pytest.raises(tide.TideError) as e:
            lay.reduce_scatter(grads, shards, 0.5)
        assert e.value.status == tide.TIDE_ERR_UNSUPPORTED
    assert _st("tide_rs_bf16_to_fp32", None, None, None, ctypes.c_float(1.0), None) == \
        tide.TIDE_ERR_INVALID_ARG
    assert _st("tide_ag_place", None, None, None, None) == tide.TIDE_ERR_INVALID_ARG


def test_empty_layout_calls_are_noops_without_a_device():
    with tide.Layout([], 3) as lay:
        assert lay.block_numel == 0
        lay.reduce_scatter([], [], 1.0)
        lay.place(None, [])
        assert len(lay.tiles(tide.TIDE_OP_RS)) == 0


@pytest.mark.parametrize("n,shapes,align", [
    (4, [(256, 256), (704, 256), (256, 704), (250,)], 8),
    (3, [(5, 3), (1,), (), (0, 4), (17, 9)], 1),
    (64, [(1000, 4096), (63, 4096)], 8),
])
def test_pack_tiles_partition_and_rank_order(n, shapes, align):
    """Pack tiles cover every element of every padded shard exactly once at
    r*S + o_p + e; RS and pack lists are rank-major (single-rank calls use a
    contiguous sub-range)."""
    offs, S = oracle.layout(shapes, n, align)
    with tide.Layout(shapes, n, align_elems=align) as lay:
        pk = lay.tiles(tide.TIDE_OP_PACK)
        rs = lay.tiles(tide.TIDE_OP_RS)
    for lst in (pk, rs):
        if len(lst):
            assert np.all(np.diff(lst[:, 1]) >= 0)
    cover = {}
    for p, r, src, dst, ln, flags in pk:
        d0, inner = _dims(shapes[p])
        c = oracle.chunk_rows(d0, n)
        cnt = cover.setdefault((p, r), np.zeros(c * inner, dtype=np.int64))
        cnt[src: src + ln] += 1
        assert dst == r * S + offs[p] + src
        if flags & 2:
            assert src % 4 == 0 and dst % 8 == 0
    for p, s in enumerate(shapes):
        d0, inner = _dims(s)
        if oracle.chunk_rows(d0, n) * inner:
            for r in range(n):
                assert np.all(cover[(p, r)] == 1), (p, r)


def test_rank_and_pack_calls_validate_on_the_host():
    shapes = [(8, 2), (5,)]
    good = 0x10000
    with tide.Layout(shapes, 2) as lay:
        grads = [good + 0x1000 * i for i in range(4)]
        mine = [good + 0x8000, good + 0x9000]
        for bad_rank in (-1, 2):
            with pytest.raises(tide.TideError) as e:
                lay.reduce_scatter_rank(bad_rank, grads, mine, 0.5)
            assert e.value.status == tide.TIDE_ERR_INVALID_ARG
        with pytest.raises(tide.TideError) as e:
            lay.pack(2, mine, good)
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
        with pytest.raises(tide.TideError) as e:
            lay.pack(0, [good + 4, good], good)
        assert e.value.status == tide.TIDE_ERR_MISALIGNED
        with pytest.raises(tide.TideError) as e:
            lay.pack(-1, mine + [None, good], good)  # all-rank form: N*P pointers, one NULL
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
        lay.set_mode(tide.TIDE_MODE_COPY_ENGINE)
        with pytest.raises(tide.TideError) as e:
            lay.pack(0, mine, good)
        assert e.value.status == tide.TIDE_ERR_UNSUPPORTED
        with pytest.raises(tide.TideError) as e:
            lay.reduce_scatter_rank(0, grads, mine, 0.5)
        assert e.value.status == tide.TIDE_ERR_UNSUPPORTED


@pytest.mark.parametrize("n,shapes,align", [
    (4, [(256, 256), (704, 256), (256, 704), (250,)], 8),
    (3, [(5, 3), (1,), (), (0, 4), (17, 9)], 1),
])
def test_staged_tiles_read_slot_offsets(n, shapes, align):
    """Staged RS tiles write the same shard runs as the RS tiles and read
    them at r*S + o_p + e of every slot."""
    offs, S = oracle.layout(shapes, n, align)
    with tide.Layout(shapes, n, align_elems=align) as lay:
        rs = lay.tiles(tide.TIDE_OP_RS)
        st = lay.tiles(tide.TIDE_OP_STAGED_RS)
    assert np.array_equal(rs[:, [0, 1, 3, 4, 5]] & ~2, st[:, [0, 1, 3, 4, 5]] & ~2)
    for p, r, src, dst, ln, flags in st:
        if not flags & 1:
            assert src == r * S + offs[p] + dst


def test_environment_overrides(monkeypatch):
    """TIDE_MODE / TIDE_CTA_CAP set a new layout's mode; TIDE_TILE_BYTES its
    reduce-scatter tile size; invalid values leave the defaults."""
    shapes = [(65536, 512)]  # large enough that small-layout tile shrinking stays out of it
    with tide.Layout(shapes, 8) as lay:
        assert lay.get_mode() == (tide.TIDE_MODE_UNCAPPED, 0)
        base = len(lay.tiles(tide.TIDE_OP_RS))
    monkeypatch.setenv("TIDE_MODE", "capped")
    monkeypatch.setenv("TIDE_CTA_CAP", "12")
    monkeypatch.setenv("TIDE_TILE_BYTES", str(64 * 1024))
    with tide.Layout(shapes, 8) as lay:
        assert lay.get_mode() == (tide.TIDE_MODE_CAPPED, 12)
        assert len(lay.tiles(tide.TIDE_OP_RS)) == 4 * base
    monkeypatch.setenv("TIDE_MODE", "bulk")
    monkeypatch.setenv("TIDE_CTA_CAP", "0")
    with tide.Layout(shapes, 8) as lay:
        assert lay.get_mode() == (tide.TIDE_MODE_BULK, 0)
    monkeypatch.setenv("TIDE_MODE", "capped")
    monkeypatch.setenv("TIDE_CTA_CAP", "0")  # invalid cap: default mode
    monkeypatch.setenv("TIDE_TILE_BYTES", "12")  # out of range: default tiles
    with tide.Layout(shapes, 8) as lay:
        assert lay.get_mode() == (tide.TIDE_MODE_UNCAPPED, 0)
        assert len(lay.tiles(tide.TIDE_OP_RS)) == base


def test_small_layouts_spread_over_the_gpu():
    """A small layout gets tiles of one CTA pass (4096 elements: 512 threads
    x 8), at least one per SM of a 152-SM GPU; a large one keeps the
    full-size tiles."""
    import synth

    with tide.Layout(synth.tiny().shapes, 4) as lay:
        for op in (tide.TIDE_OP_RS, tide.TIDE_OP_AG, tide.TIDE_OP_PACK):
            t = lay.tiles(op)
            assert len(t) >= 152
            assert t[:, 4].max() == 4096
    with tide.Layout([(8192, 8192)], 8) as lay:
        t = lay.tiles(tide.TIDE_OP_RS)
        assert t[:, 4].max() == 16384  # 256 KiB of bf16 reads over 8 ranks


def test_place_ranks_and_ipc_validate_on_the_host():
    """The per-rank placement checks its N buffer pointers and P parameter
    pointers before anything touches a device; the IPC calls refuse NULL
    arguments and malformed handles."""
    shapes = [(8, 2), (5,)]
    good = 0x10000
    with tide.Layout(shapes, 2) as lay:
        params = [good + 0x1000, good + 0x2000]
        for bufs, status in (([good, None], tide.TIDE_ERR_INVALID_ARG),
                             ([good, good + 8], tide.TIDE_ERR_MISALIGNED)):
            with pytest.raises(tide.TideError) as e:
                lay.place_ranks(bufs, params)
            assert e.value.status == status
        with pytest.raises(tide.TideError) as e:
            lay.place_ranks([good, good], [good + 2, good])
        assert e.value.status == tide.TIDE_ERR_MISALIGNED
        with pytest.raises(tide.TideError) as e:
            tide.tide_ag_place_ranks(lay.handle, None, params)
        assert e.value.status == tide.TIDE_ERR_INVALID_ARG
    from layout_aware_collectives_gb300 import tide as T

    for call in (lambda: T._lib.tide_ipc_export(None, None, None),
                 lambda: T._lib.tide_ipc_open(None, None),
                 lambda: T._lib.tide_ipc_close(None)):
        assert call() == tide.TIDE_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        tide.tide_ipc_open(b"short")
