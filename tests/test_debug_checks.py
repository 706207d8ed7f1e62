"""The range test the kernels of the debug build apply to every tile they
fetch, run on the host through tide_layout_check_tiles (no GPU): every tile
of every real list passes, a tile that ends exactly at its buffer's end
passes, and each planted corruption of a single tile is caught at its index.
The GPU tests only ever give the debug build valid tile lists."""
import numpy as np
import pytest

import layout_aware_collectives_gb300 as tide

OPS = {"rs": tide.TIDE_OP_RS, "ag": tide.TIDE_OP_AG, "pack": tide.TIDE_OP_PACK,
       "stage": tide.TIDE_OP_STAGE, "staged_rs": tide.TIDE_OP_STAGED_RS}


def _layouts():
    rng = np.random.default_rng(21)
    cases = [("tiny", 4, [(256, 256)] * 4 + [(704, 256), (704, 256), (256, 704), (250,)], 8)]
    for n in (1, 3, 5, 13, 64):
        shapes = [(int(rng.integers(1, 3 * n + 5)), int(rng.integers(1, 40))) for _ in range(3)]
        shapes += [(max(1, n - 1), 24), (3 * n + 1,), (), (0, 16), (2 * n, 3, 5)]
        for align in (8, 1):
            cases.append((f"ragged_n{n}_a{align}", n, shapes, align))
    return cases


LAYOUTS = _layouts()


def _extents(lay, shapes, op):
    """(source extent, destination extent, source alignment, destination
    alignment) of parameter p for `op`, from the layout's own queries."""
    N, S = lay.num_ranks, lay.block_numel
    numel = [int(np.prod(s)) if len(s) else 1 for s in shapes]
    shard = [lay.shard_numel(p) for p in range(len(shapes))]
    buf = N * S

    def ext(p):
        if op == tide.TIDE_OP_RS:
            return numel[p], shard[p], 8, 4
        if op == tide.TIDE_OP_STAGED_RS:
            return buf, shard[p], 8, 4
        if op == tide.TIDE_OP_PACK:
            return shard[p], buf, 4, 8
        return buf, numel[p], 8, 8  # placement, and staging (the placement list run backwards)
    return ext


@pytest.mark.parametrize("case", LAYOUTS, ids=[c[0] for c in LAYOUTS])
def test_every_real_tile_passes(case):
    name, n, shapes, align = case
    with tide.Layout(shapes, n, align_elems=align) as lay:
        for op in OPS.values():
            rows = lay.tiles(op)
            assert lay.check_tiles(op, rows) == -1, op
            assert lay.check_tiles(op, rows[:0]) == -1


def _corruptions(row, op, ext, P, N):
    """(what, corrupted row) pairs for one valid tile; each must fail."""
    p, r, src, dst, ln, flags = (int(x) for x in row)
    src_n, dst_n, src_al, dst_al = ext(p)
    zero = bool(flags & 1)
    vec = bool(flags & 2)
    out = []

    def put(what, **kw):
        x = dict(p=p, r=r, src=src, dst=dst, ln=ln, flags=flags)
        x.update(kw)
        out.append((what, [x["p"], x["r"], x["src"], x["dst"], x["ln"], x["flags"]]))

    put("parameter past the last", p=P)
    put("negative parameter", p=-1)
    put("rank past the last", r=N)
    put("negative rank", r=-1)
    put("negative length", ln=-1)
    put("negative destination", dst=-8)
    put("destination run past its buffer", dst=dst_n - ln + 1 if ln else dst_n + 1)
    put("length past the destination", ln=dst_n - dst + 1)
    put("unknown flag", flags=flags | 4)
    if not zero:
        put("negative source", src=-8)
        put("source run past its buffer", src=src_n - ln + 1 if ln else src_n + 1)
    if op not in (tide.TIDE_OP_RS, tide.TIDE_OP_STAGED_RS):
        put("zero-fill tile outside a reduce-scatter list", flags=flags | 1)
    if vec and ln >= 2:
        if not zero:
            put("vector tile with a misaligned source", src=src + 1, ln=ln - 1)
        put("vector tile with a misaligned destination", dst=dst + 1, ln=ln - 1)
    return out


@pytest.mark.parametrize("case", LAYOUTS[:1] + LAYOUTS[3:5] + LAYOUTS[-2:], ids=lambda c: c[0])
def test_planted_corruptions_are_caught(case):
    name, n, shapes, align = case
    P = len(shapes)
    with tide.Layout(shapes, n, align_elems=align) as lay:
        for opname, op in OPS.items():
            rows = lay.tiles(op)
            if rows.shape[0] == 0:
                continue
            ext = _extents(lay, shapes, op)
            picks = sorted({0, rows.shape[0] // 2, rows.shape[0] - 1})
            picks += [i for i in range(rows.shape[0]) if rows[i, 5] & 1][:1]  # a zero-fill tile
            picks += [i for i in range(rows.shape[0]) if rows[i, 5] & 2][:1]  # a vector tile
            tried = 0
            for i in picks:
                for what, bad in _corruptions(rows[i], op, ext, P, n):
                    corrupted = rows.copy()
                    corrupted[i] = bad
                    got = lay.check_tiles(op, corrupted)
                    assert got == i, f"{opname} tile {i}: '{what}' not caught ({bad})"
                    tried += 1
            assert tried > 0


@pytest.mark.parametrize("case", LAYOUTS[:1] + LAYOUTS[-2:], ids=lambda c: c[0])
def test_a_tile_ending_at_its_buffer_end_passes(case):
    name, n, shapes, align = case
    with tide.Layout(shapes, n, align_elems=align) as lay:
        for op in OPS.values():
            rows = lay.tiles(op)
            ext = _extents(lay, shapes, op)
            for i in range(min(rows.shape[0], 40)):
                p, r, src, dst, ln, flags = (int(x) for x in rows[i])
                src_n, dst_n, _, _ = ext(p)
                moved = rows.copy()
                # last possible destination (vector flag dropped so only the extent is tested)
                moved[i, 3] = dst_n - ln
                moved[i, 5] = flags & ~2
                if not flags & 1:
                    moved[i, 2] = src_n - ln
                assert lay.check_tiles(op, moved) == -1, (op, i)


def test_check_tiles_rejects_bad_arguments():
    with tide.Layout([(8, 8)], 2) as lay:
        with pytest.raises(tide.TideError):
            tide.tide_layout_check_tiles(lay.handle, 99, np.zeros((1, 6), np.int64))
    assert tide.tide_build_info() in ("release", "debug: device range checks")
