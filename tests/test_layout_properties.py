"""Property tests of the host layout descriptor (no GPU): for random shapes,
rank counts and alignments, the layout matches the oracle and every tile
list covers its outputs exactly once, reading from the right place.  With
hypothesis installed the cases are drawn (and shrunk) by it; without it,
150 seeded random cases of the same distribution run instead."""
import numpy as np
import pytest

import oracle
import layout_aware_collectives_gb300 as tide

try:
    from hypothesis import given, settings, strategies as st
except ImportError:  # the property still runs, on seeded cases
    given = None


def _dims(s):
    if not s:
        return 1, 1
    inner = 1
    for d in s[1:]:
        inner *= d
    return s[0], inner


ALIGNS = [1, 2, 4, 8, 16, 64]


def check_layout_and_tiles(shapes, n, align):
    offs, S = oracle.layout(shapes, n, align)
    with tide.Layout(shapes, n, align_elems=align) as lay:
        assert lay.block_numel == S
        assert [lay.param_offset(p) for p in range(len(shapes))] == list(offs)
        rs = lay.tiles(tide.TIDE_OP_RS)
        ag = lay.tiles(tide.TIDE_OP_AG)
        pk = lay.tiles(tide.TIDE_OP_PACK)
        sr = lay.tiles(tide.TIDE_OP_STAGED_RS)
    shard = {}
    packed = {}
    for p, s in enumerate(shapes):
        d0, inner = _dims(s)
        c = oracle.chunk_rows(d0, n)
        for r in range(n):
            shard[(p, r)] = np.zeros(c * inner, np.int64)
            packed[(p, r)] = np.zeros(c * inner, np.int64)
    for lst, staged in ((rs, False), (sr, True)):
        cover = {k: v.copy() for k, v in shard.items()}
        for p, r, src, dst, ln, fl in lst:
            d0, inner = _dims(shapes[p])
            c = oracle.chunk_rows(d0, n)
            v = oracle.valid_rows(d0, n, r) * inner
            cover[(p, r)][dst: dst + ln] += 1
            if not fl & 1:
                assert dst + ln <= v
                want = r * S + offs[p] + dst if staged else r * c * inner + dst
                assert src == want
        assert all(np.all(x == 1) for x in cover.values())
    params = [np.zeros(_dims(s)[0] * _dims(s)[1], np.int64) for s in shapes]
    for p, r, src, dst, ln, fl in ag:
        params[p][dst: dst + ln] += 1
        d0, inner = _dims(shapes[p])
        assert src == oracle.ag_source_index(n, shapes[p], offs[p], S, dst // inner, dst % inner)
    assert all(np.all(x == 1) for x in params)
    for p, r, src, dst, ln, fl in pk:
        packed[(p, r)][src: src + ln] += 1
        assert dst == r * S + offs[p] + src
    assert all(np.all(x == 1) for x in packed.values())


if given is not None:
    shapes_st = st.lists(st.lists(st.integers(0, 40), min_size=0, max_size=3).map(tuple),
                         min_size=0, max_size=7)

    @settings(max_examples=150, deadline=None)
    @given(shapes=shapes_st, n=st.integers(1, 70), align=st.sampled_from(ALIGNS))
    def test_layout_and_tiles(shapes, n, align):
        check_layout_and_tiles(shapes, n, align)
else:
    def _seeded_cases(count=150, seed=41):
        rng = np.random.default_rng(seed)
        cases = []
        for _ in range(count):
            shapes = [tuple(int(d) for d in rng.integers(0, 41, size=int(rng.integers(0, 4))))
                      for _ in range(int(rng.integers(0, 8)))]
            cases.append((shapes, int(rng.integers(1, 71)), ALIGNS[int(rng.integers(0, len(ALIGNS)))]))
        return cases

    @pytest.mark.parametrize("case", _seeded_cases())
    def test_layout_and_tiles(case):
        check_layout_and_tiles(*case)
