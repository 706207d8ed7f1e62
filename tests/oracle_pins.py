"""Checks that pin the CPU oracle to facts other than itself.

Each check raises AssertionError on a mismatch.  test_oracle.py runs them
against the oracle; test_oracle_mutants.py runs them against copies of the
oracle with one planted mistake each and requires that some check fails.

Pins used (the pages print no worked numbers, so nothing comes from them):
  - hand-derived golden fixtures in tests/golden/ (each cites its source);
  - torch.chunk, the dim-0 split FSDP2 uses, for the chunk rule;
  - whole-array numpy arithmetic followed by a torch.chunk split (brute force);
  - exact integer sums (order-free: any correct summation gives them);
  - N identical inputs averaged with scale 1/N (exact for power-of-two N);
  - the recursive-summation error bound against an fp64 sum;
  - placement identity with sentinels in every padding slot, and the
    composition reduce-scatter -> bf16 -> rank-major pack -> placement.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
SENTINEL = 0x7FC1
U = 2.0 ** -24


# ---------------------------------------------------------------- helpers
def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """bf16 bits of fp32 values via torch's own rounding (RNE)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def dims(shape):
    if len(shape) == 0:
        return 1, 1
    inner = 1
    for d in shape[1:]:
        inner *= d
    return shape[0], inner


def torch_chunks(d0, inner, n, data=None):
    """FSDP2-style dim-0 split: torch.chunk, padded with empty chunks to n."""
    t = torch.arange(d0 * inner).reshape(d0, inner) if data is None else data
    chunks = list(torch.chunk(t, n, dim=0)) if d0 > 0 else []
    while len(chunks) < n:
        chunks.append(t[d0:])
    return chunks


def random_bf16(rng, n, scale=1.0):
    x = (rng.standard_normal(n) * scale).astype(np.float32)
    return f32_to_bf16_rne(x)


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def fp32_bits(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).view(np.uint32)


# ---------------------------------------------------------------- chunking
def check_chunking_golden():
    for row in load_golden("chunking.txt"):
        d0, n, c = int(row[0]), int(row[1]), int(row[2])
        valid = [int(v) for v in row[3].split(",")]
        assert oracle.chunk_rows(d0, n) == c, (d0, n)
        assert [oracle.valid_rows(d0, n, r) for r in range(n)] == valid, (d0, n)


def check_chunking_vs_torch():
    for n in range(1, 9):
        for d0 in range(0, 18):
            chunks = torch_chunks(d0, 1, n)
            c = chunks[0].shape[0] if d0 else 0
            assert oracle.chunk_rows(d0, n) == c, (d0, n)
            for r in range(n):
                assert oracle.valid_rows(d0, n, r) == chunks[r].shape[0], (d0, n, r)
                # the rows rank r owns are exactly torch.chunk's rows
                if chunks[r].shape[0]:
                    assert int(chunks[r][0, 0]) == r * c


# ---------------------------------------------------------------- layout
def check_layout_golden():
    rows = load_golden("tiny_layout.txt")
    shapes, offs = [], []
    for row in rows:
        if row[0] == "S":
            S = int(row[1])
        elif row[0] == "S_dense":
            S_dense = int(row[1])
        else:
            d0, inner = int(row[1]), int(row[2])
            shapes.append((d0, inner) if inner > 1 else (d0,))
            assert oracle.chunk_rows(d0, 4) == int(row[3])
            assert oracle.shard_numel(shapes[-1], 4) == int(row[4])
            offs.append(int(row[5]))
    o, s = oracle.layout(shapes, 4, 8)
    assert list(o) == offs and s == S, (list(o), s)
    o1, s1 = oracle.layout(shapes, 4, 1)
    assert list(o1) == offs and s1 == S_dense, (list(o1), s1)


def check_layout_properties(seed=1):
    rng = np.random.default_rng(seed)
    for trial in range(60):
        n = int(rng.integers(1, 12))
        align = int(rng.choice([1, 2, 4, 8, 16]))
        shapes = []
        for _ in range(int(rng.integers(0, 7))):
            nd = int(rng.integers(0, 4))
            shapes.append(tuple(int(rng.integers(0, 9)) for _ in range(nd)))
        offs, S = oracle.layout(shapes, n, align)
        end = 0
        for p, s in enumerate(shapes):
            d0, inner = dims(s)
            sn = -(-d0 // n) * inner
            assert offs[p] % align == 0
            assert offs[p] >= end  # no overlap with the previous shard
            assert offs[p] - end < align  # and no gap beyond the alignment
            end = offs[p] + sn
        assert S % align == 0 and S >= end and S - end < align


# ---------------------------------------------------------------- reduce-scatter
def _parse_rs_cases():
    cases, cur = [], None
    for row in load_golden("rs_hand.txt"):
        if row[0] == "case":
            d0, inner = (int(v) for v in row[5].split("x"))
            cur = dict(name=row[1], n=int(row[3]), d0=d0, inner=inner, scale=float(row[7]),
                       grads={}, shards={})
            cases.append(cur)
        elif row[0] == "grad":
            cur["grads"][int(row[1])] = np.array([int(h, 16) for h in row[2:]], dtype=np.uint16)
        elif row[0] == "shard":
            cur["shards"][int(row[1])] = np.array([int(h, 16) for h in row[2:]], dtype=np.uint32)
    return cases


def check_rs_golden():
    for cs in _parse_rs_cases():
        shape = (cs["d0"], cs["inner"])
        grads = [[cs["grads"][k]] for k in range(cs["n"])]
        out = oracle.rs([shape], cs["n"], grads, cs["scale"])
        for r in range(cs["n"]):
            got = fp32_bits(out[r][0])
            assert np.array_equal(got, cs["shards"][r]), (cs["name"], r, got, cs["shards"][r])


def brute_force_rs(shapes, n, grads, scale):
    """Whole-array fp32 sums in rank order, then a torch.chunk split + zero pad."""
    out = [[None] * len(shapes) for _ in range(n)]
    for p, s in enumerate(shapes):
        d0, inner = dims(s)
        full = np.zeros(d0 * inner, dtype=np.float32)
        for k in range(n):
            full = full + bf16_to_f32(grads[k][p])
        full = full * np.float32(scale)
        chunks = torch_chunks(d0, inner, n, torch.from_numpy(full.reshape(d0, inner)))
        c = -(-d0 // n)
        for r in range(n):
            ch = chunks[r].numpy().reshape(-1, inner)
            pad = np.zeros((c - ch.shape[0], inner), dtype=np.float32)
            out[r][p] = np.concatenate([ch, pad]).ravel()
    return out


def check_rs_brute_force(seed=2):
    rng = np.random.default_rng(seed)
    for n in (1, 2, 3, 4, 5, 8):
        for d0 in range(1, 18):
            shapes = [(d0, 3), (d0,), (2, d0)]
            grads = [[random_bf16(rng, d0 * 3), random_bf16(rng, d0), random_bf16(rng, 2 * d0)]
                     for _ in range(n)]
            scale = float(rng.choice([1.0 / n, 0.3, -2.0]))
            got = oracle.rs(shapes, n, grads, scale)
            want = brute_force_rs(shapes, n, grads, scale)
            for r in range(n):
                for p in range(len(shapes)):
                    assert np.array_equal(fp32_bits(got[r][p]), fp32_bits(want[r][p])), \
                        (n, d0, r, p)


def check_rs_integer_exact(seed=3):
    """Small integers sum exactly in any order: compare with Python ints."""
    rng = np.random.default_rng(seed)
    for n in (1, 2, 3, 7, 16, 64):
        shapes = [(11, 5), (4,), (3, 2, 2)]
        ints = [[rng.integers(-128, 129, size=int(np.prod(s))) for s in shapes] for _ in range(n)]
        grads = [[f32_to_bf16_rne(a.astype(np.float32)) for a in row] for row in ints]
        scale = 0.25
        got = oracle.rs(shapes, n, grads, scale)
        for p, s in enumerate(shapes):
            d0, inner = dims(s)
            total = [sum(int(ints[k][p][e]) for k in range(n)) for e in range(d0 * inner)]
            c = -(-d0 // n)
            for r in range(n):
                for ii in range(c):
                    for j in range(inner):
                        i = r * c + ii
                        want = total[i * inner + j] * scale if i < d0 else 0.0
                        assert got[r][p][ii * inner + j] == want, (n, p, r, ii, j)


def check_rs_identical_inputs(seed=4):
    """N copies of the same bf16 gradient averaged with 1/N give it back exactly."""
    rng = np.random.default_rng(seed)
    for n in (1, 2, 4, 8, 16, 32, 64):
        shape = (2 * n + 3, 7)
        g = random_bf16(rng, shape[0] * shape[1])
        out = oracle.rs([shape], n, [[g] for _ in range(n)], 1.0 / n)
        full = np.concatenate([out[r][0] for r in range(n)])[: g.size]
        assert np.array_equal(fp32_bits(full), fp32_bits(bf16_to_f32(g))), n


def check_rs_f64_bound(seed=5):
    """|fp32 result - fp64 result| <= gamma_{N-1} |scale| sum|g| + u |result|."""
    rng = np.random.default_rng(seed)
    for n in (2, 3, 8, 16, 64):
        shape = (n + 1, 33)
        m = shape[0] * shape[1]
        grads = [[random_bf16(rng, m, scale=float(rng.choice([1e-3, 1.0, 1e3])))]
                 for _ in range(n)]
        scale = 1.0 / 3.0
        out = oracle.rs([shape], n, grads, scale)
        full = np.concatenate([out[r][0] for r in range(n)])[:m].astype(np.float64)
        vals = np.stack([bf16_to_f32(grads[k][0]).astype(np.float64) for k in range(n)])
        exact = vals.sum(axis=0) * np.float64(np.float32(scale))
        gamma = (n - 1) * U / (1 - (n - 1) * U)
        bound = gamma * abs(float(np.float32(scale))) * np.abs(vals).sum(axis=0) + U * np.abs(exact)
        assert np.all(np.abs(full - exact) <= bound + 1e-45), n
        # and the sum is not trivially zero
        assert np.count_nonzero(full) > m // 2


def check_rs_special_values():
    inf, ninf, nan, one = 0x7F80, 0xFF80, 0x7FC0, 0x3F80
    shape = (1, 4)
    grads = [[np.array([inf, inf, nan, one], dtype=np.uint16)],
             [np.array([one, ninf, one, ninf], dtype=np.uint16)]]
    out = oracle.rs([shape], 2, grads, 1.0)[0][0]
    assert out[0] == np.inf
    assert np.isnan(out[1]) and np.isnan(out[2])
    assert out[3] == -np.inf


# ---------------------------------------------------------------- placement
def check_ag_golden():
    rows = load_golden("ag_hand.txt")
    kv = {r[0]: r[1:] for r in rows if r[0] not in ("shape", "param")}
    n, align = int(kv["N"][0]), int(kv["align"][0])
    shapes, params = {}, {}
    for r in rows:
        if r[0] == "shape":
            d0, inner = (int(v) for v in r[2].split("x"))
            shapes[int(r[1])] = (d0, inner)
        elif r[0] == "param":
            params[int(r[1])] = np.array([int(h, 16) for h in r[2:]], dtype=np.uint16)
    shp = [shapes[p] for p in sorted(shapes)]
    offs, S = oracle.layout(shp, n, align)
    assert list(offs) == [int(v) for v in kv["offsets"]] and S == int(kv["S"][0])
    buf = np.array([int(h, 16) for h in kv["gathered"]], dtype=np.uint16)
    got = oracle.ag_place(shp, n, buf, offs, S)
    for p in range(len(shp)):
        assert np.array_equal(got[p], params[p]), p


def pack_rank_major(shapes, n, full_bits, offs, S, fill=SENTINEL):
    """Test-side packing of each parameter's padded dim-0 shards, rank-major."""
    buf = np.full(n * S, fill, dtype=np.uint16)
    for p, s in enumerate(shapes):
        d0, inner = dims(s)
        chunks = torch_chunks(d0, inner, n,
                              torch.from_numpy(full_bits[p].view(np.int16).reshape(d0, inner)))
        for r in range(n):
            v = chunks[r].numpy().view(np.uint16).ravel()
            buf[r * S + offs[p]: r * S + offs[p] + v.size] = v
    return buf


def check_ag_identity(seed=6):
    rng = np.random.default_rng(seed)
    for n in (1, 2, 3, 4, 7, 8):
        for align in (1, 8):
            shapes = [(int(rng.integers(1, 20)), int(rng.integers(1, 6))) for _ in range(3)]
            shapes += [(int(rng.integers(1, 13)),), (1,)]
            full = [random_bf16(rng, dims(s)[0] * dims(s)[1]) for s in shapes]
            for f in full:
                f[f == SENTINEL] = 0x3F80
            offs, S = oracle.layout(shapes, n, align)
            buf = pack_rank_major(shapes, n, full, offs, S)
            got = oracle.ag_place(shapes, n, buf, offs, S)
            for p in range(len(shapes)):
                assert np.array_equal(got[p], full[p]), (n, align, p)
                assert not np.any(got[p] == SENTINEL)


def check_rs_ag_composition(seed=7):
    """RS -> RNE bf16 -> rank-major pack -> placement == bf16(full reduced tensor)."""
    rng = np.random.default_rng(seed)
    for n in (2, 4, 5):
        shapes = [(9, 4), (13,), (4, 6)]
        grads = [[random_bf16(rng, dims(s)[0] * dims(s)[1]) for s in shapes] for _ in range(n)]
        shards = oracle.rs(shapes, n, grads, 1.0 / n)
        offs, S = oracle.layout(shapes, n, 8)
        buf = np.full(n * S, SENTINEL, dtype=np.uint16)
        for r in range(n):
            for p in range(len(shapes)):
                d0, inner = dims(s := shapes[p])
                v = oracle.valid_rows(d0, n, r) * inner
                buf[r * S + offs[p]: r * S + offs[p] + v] = f32_to_bf16_rne(shards[r][p][:v])
        placed = oracle.ag_place(shapes, n, buf, offs, S)
        want = brute_force_rs(shapes, n, grads, 1.0 / n)
        for p, s in enumerate(shapes):
            d0, inner = dims(s)
            full = np.concatenate([want[r][p] for r in range(n)])[: d0 * inner]
            assert np.array_equal(placed[p], f32_to_bf16_rne(full)), (n, p)


ALL_CHECKS = [
    check_chunking_golden, check_chunking_vs_torch, check_layout_golden, check_layout_properties,
    check_rs_golden, check_rs_brute_force, check_rs_integer_exact, check_rs_identical_inputs,
    check_rs_f64_bound, check_rs_special_values, check_ag_golden, check_ag_identity,
    check_rs_ag_composition,
]


# ---------------------------------------------------------------- single-rank RS and AG input pack
def check_bf16_rounding_golden():
    for row in load_golden("bf16_rounding.txt"):
        f = np.array([int(row[0], 16)], dtype=np.uint32).view(np.float32)
        got = int(oracle.f32_to_bf16(f)[0])
        assert got == int(row[1], 16), (row[0], hex(got), row[1])


def check_bf16_rounding_vs_torch(seed=8):
    """Finite values against torch's own fp32 -> bfloat16 conversion."""
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    x = np.concatenate([x, (rng.standard_normal(5000) * 1e-3).astype(np.float32)])
    assert np.array_equal(oracle.f32_to_bf16(x), f32_to_bf16_rne(x))


def check_rs_rank_matches_full(seed=9):
    rng = np.random.default_rng(seed)
    for n in (1, 3, 4, 8):
        shapes = [(2 * n + 1, 3), (n - 1 if n > 1 else 1,), (5, 2, 2)]
        grads = [[random_bf16(rng, dims(s)[0] * dims(s)[1]) for s in shapes] for _ in range(n)]
        full = oracle.rs(shapes, n, grads, 0.5)
        for r in range(n):
            one = oracle.rs_rank(shapes, n, grads, 0.5, r)
            for p in range(len(shapes)):
                assert np.array_equal(fp32_bits(one[p]), fp32_bits(full[r][p])), (n, r, p)


def check_pack_then_place(seed=10):
    """Every rank packs its fp32 shards; placement of the result gives the
    bf16 (torch rounding) of the full reduced tensor; padding slots of each
    shard carry bf16 +0 and alignment gaps keep the sentinel."""
    rng = np.random.default_rng(seed)
    for n in (2, 3, 4):
        shapes = [(7, 5), (11,), (3, 4)]
        grads = [[random_bf16(rng, dims(s)[0] * dims(s)[1]) for s in shapes] for _ in range(n)]
        shards = oracle.rs(shapes, n, grads, 1.0 / n)
        offs, S = oracle.layout(shapes, n, 8)
        buf = np.full(n * S, SENTINEL, dtype=np.uint16)
        for r in range(n):
            oracle.ag_pack(shapes, n, offs, S, r, shards[r], buf)
        placed = oracle.ag_place(shapes, n, buf, offs, S)
        want = brute_force_rs(shapes, n, grads, 1.0 / n)
        written = np.zeros(n * S, dtype=bool)
        for p, s in enumerate(shapes):
            d0, inner = dims(s)
            full = np.concatenate([want[r][p] for r in range(n)])[: d0 * inner]
            assert np.array_equal(placed[p], f32_to_bf16_rne(full)), (n, p)
            c = oracle.chunk_rows(d0, n)
            for r in range(n):
                v = oracle.valid_rows(d0, n, r) * inner
                blk = buf[r * S + offs[p]: r * S + offs[p] + c * inner]
                assert np.all(blk[v:] == 0)  # padding rows: bf16(+0.0)
                written[r * S + offs[p]: r * S + offs[p] + c * inner] = True
        assert np.all(buf[~written] == SENTINEL)


ALL_CHECKS += [check_bf16_rounding_golden, check_bf16_rounding_vs_torch, check_rs_rank_matches_full,
               check_pack_then_place]


# ---------------------------------------------------------------- Slot-Reuse staged reduce-scatter
def check_stage_is_inverse_of_placement(seed=11):
    """Staging a full gradient into the rank-major slot and placing the slot
    back gives the gradient (bit for bit); every padding slot keeps the
    sentinel."""
    rng = np.random.default_rng(seed)
    for n in (1, 2, 3, 5):
        for align in (1, 8):
            shapes = [(int(rng.integers(1, 3 * n + 4)), int(rng.integers(1, 6))) for _ in range(3)]
            shapes += [(n - 1 if n > 1 else 1,), (4, 2, 3)]
            g = [random_bf16(rng, dims(s)[0] * dims(s)[1]) for s in shapes]
            for x in g:
                x[x == SENTINEL] = 0x3F80
            offs, S = oracle.layout(shapes, n, align)
            slot = np.full(n * S, SENTINEL, dtype=np.uint16)
            oracle.rs_stage(shapes, n, offs, S, g, slot)
            # the slot is exactly the rank-major packing of the gradient
            assert np.array_equal(slot, pack_rank_major(shapes, n, g, offs, S))
            back = oracle.ag_place(shapes, n, slot, offs, S)
            for p in range(len(shapes)):
                assert np.array_equal(back[p], g[p]), (n, align, p)


def check_staged_rs_equals_rs(seed=12):
    """Reduce-scatter from the staged slots equals the brute-force reduce-
    scatter of the per-parameter gradients, bit for bit."""
    rng = np.random.default_rng(seed)
    for n in (1, 2, 4, 5, 8):
        shapes = [(2 * n + 3, 4), (n + 1,), (3, 3, 2), (1, 7)]
        grads = [[random_bf16(rng, dims(s)[0] * dims(s)[1]) for s in shapes] for _ in range(n)]
        offs, S = oracle.layout(shapes, n, 8)
        slots = []
        for k in range(n):
            slot = np.full(n * S, SENTINEL, dtype=np.uint16)  # padding is never read
            slots.append(oracle.rs_stage(shapes, n, offs, S, grads[k], slot))
        got = oracle.rs_staged(shapes, n, offs, S, slots, 1.0 / n)
        want = brute_force_rs(shapes, n, grads, 1.0 / n)
        for r in range(n):
            for p in range(len(shapes)):
                assert np.array_equal(fp32_bits(got[r][p]), fp32_bits(want[r][p])), (n, r, p)


ALL_CHECKS += [check_stage_is_inverse_of_placement, check_staged_rs_equals_rs]


def check_rs_rank_limit():
    """The reduce-scatter functions gather one element's N inputs into a
    4096-entry array: N = 4096 is computed (and equals the exact integer
    sum), N = 4097 and N = 0 are refused before anything is read or written,
    through the wrapper and through the C entry points themselves."""
    import ctypes

    one = 0x3F80  # bf16 1.0
    n = 4096
    grads = [[np.array([one], dtype=np.uint16)] for _ in range(n)]
    out = oracle.rs([(1,)], n, grads, 1.0)
    assert out[0][0][0] == np.float32(n) and all(out[r][0].size == 1 and out[r][0][0] == 0 for r in range(1, n))
    assert oracle.rs_rank([(1,)], n, grads, 1.0, 0)[0][0] == np.float32(n)
    for bad in (n + 1, 0):
        for call in (lambda: oracle.rs([(1,)], bad, grads, 1.0),
                     lambda: oracle.rs_rank([(1,)], bad, grads, 1.0, 0),
                     lambda: oracle.rs_staged([(1,)], bad, [0], 8, [], 1.0)):
            try:
                call()
            except ValueError:
                continue
            raise AssertionError(f"oracle accepted {bad} ranks")
    # the C functions refuse on their own (the wrapper is not the only guard)
    L = oracle.lib()
    n = 4097
    d0 = np.ones(1, dtype=np.int64)
    inner = np.ones(1, dtype=np.int64)
    src = np.array([one], dtype=np.uint16)
    gp = np.full(n, src.ctypes.data, dtype=np.uint64)
    outs = [np.full(1, 7.0, dtype=np.float32) for _ in range(n)]
    op = np.asarray([o.ctypes.data for o in outs], dtype=np.uint64)
    offs = np.zeros(1, dtype=np.int64)
    assert L.oracle_rs(n, 1, d0.ctypes.data, inner.ctypes.data, gp.ctypes.data, op.ctypes.data,
                       ctypes.c_float(1.0)) == 1
    assert L.oracle_rs_rank(n, 1, d0.ctypes.data, inner.ctypes.data, gp.ctypes.data, op.ctypes.data,
                            ctypes.c_float(1.0), 0) == 1
    assert L.oracle_rs_staged(n, 1, d0.ctypes.data, inner.ctypes.data, offs.ctypes.data, 8,
                              gp.ctypes.data, op.ctypes.data, ctypes.c_float(1.0)) == 1
    assert L.oracle_rs_rank(4, 1, d0.ctypes.data, inner.ctypes.data, gp.ctypes.data, op.ctypes.data,
                            ctypes.c_float(1.0), 4) == 1
    assert all(o[0] == 7.0 for o in outs), "a refused call wrote an output"


ALL_CHECKS += [check_rs_rank_limit]


def check_rs_ieee_closed_forms():
    """Every special-value case of ieee_cases against its closed form, derived
    by hand from the sequential fp32 sum: subnormal sums kept (no flush),
    -0 inputs giving +0, infinities and NaNs propagated, overflow to
    infinity, and the cases whose result depends on ascending rank order."""
    import math

    import ieee_cases

    for n in (1, 2, 3, 4, 5, 8, 13, 64, 100):
        names = [c[0] for c in ieee_cases.cases(n)]
        cols = np.array([v for _, v in ieee_cases.cases(n)], dtype=np.uint16).T  # [N][C]
        grads = [[np.ascontiguousarray(cols[k])] for k in range(n)]
        for scale in (1.0, 0.25, 2.0 ** -6):
            got = oracle.rs([(1, len(names))], n, grads, scale)[0][0]
            for j, name in enumerate(names):
                want = ieee_cases.expected(name, n, scale)
                g = float(got[j])
                if math.isnan(want):
                    assert math.isnan(g), (name, n, scale, g)
                else:
                    assert g == want and math.copysign(1, g) == math.copysign(1, want), (name, n, scale, g, want)


ALL_CHECKS += [check_rs_ieee_closed_forms]
