"""Checks of device results against the CPU oracle (and, at full size, a
plain PyTorch fp32 reference that covers every element).

Oracle inputs are regenerated on the host from the seeded generator; nothing
the CUDA path produced is fed to the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from synth import SENTINEL_BF16


def _bits32(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int32).cpu().numpy().view(np.uint32)


def _bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def check_layout(job):
    offs, S = oracle.layout(job.wl.shapes, job.N, job.align)
    assert S == job.layout.block_numel, (S, job.layout.block_numel)
    for p in range(job.P):
        assert offs[p] == job.layout.param_offset(p), p
    return offs, S


def full_check_rs(job, scale=None):
    """Every shard element (padding included) bit-exact against the oracle."""
    wl = job.wl
    scale = wl.scale if scale is None else scale
    grads = [[wl.host_grad(k, p) for p in range(job.P)] for k in range(job.N)]
    want = oracle.rs(wl.shapes, job.N, grads, scale)
    for r in range(job.N):
        for p in range(job.P):
            got = _bits32(job.shards[r][p])
            exp = want[r][p].view(np.uint32)
            if not np.array_equal(got, exp):
                bad = np.flatnonzero(got != exp)
                raise AssertionError(f"RS mismatch rank {r} param {p}: {bad.size} elements, first "
                                     f"at {bad[0]}: got {got[bad[0]]:08x} want {exp[bad[0]]:08x}")


def host_gathered(job):
    """The rank-major buffer rebuilt on the host with the oracle's layout."""
    wl = job.wl
    offs, S = oracle.layout(wl.shapes, job.N, job.align)
    buf = np.full(job.N * S, SENTINEL_BF16, dtype=np.uint16)
    for p in range(job.P):
        full = wl.host_param_value(p)
        d0, inner = job.dims[p]
        c = oracle.chunk_rows(d0, job.N)
        for r in range(job.N):
            v = oracle.valid_rows(d0, job.N, r) * inner
            buf[r * S + offs[p]: r * S + offs[p] + v] = full[r * c * inner: r * c * inner + v]
    return buf, offs, S


def full_check_ag(job):
    """Every parameter element bit-exact against the oracle's placement."""
    buf, offs, S = host_gathered(job)
    assert S == job.layout.block_numel
    assert np.array_equal(_bits16(job.gathered), buf), "device and host generators disagree"
    want = oracle.ag_place(job.wl.shapes, job.N, buf, offs, S)
    for p in range(job.P):
        got = _bits16(job.params[p])
        assert np.array_equal(got, want[p]), f"placement mismatch in param {p}"
        assert not np.any(got == SENTINEL_BF16), f"padding slot reached param {p}"


def sample_indices(rng, job, p, r, per=6):
    """Shard-local sample positions of (p, r): edges of the valid rows, random
    interior points and padding positions."""
    d0, inner = job.dims[p]
    c = job.chunk[p]
    v = oracle.valid_rows(d0, job.N, r)
    n = c * inner
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    pts = {0, n - 1}
    if v:
        pts |= {v * inner - 1, (v - 1) * inner, min(inner, v * inner - 1)}
        pts |= set(int(x) for x in rng.integers(0, v * inner, size=per))
    if v < c:
        pts |= {v * inner, n - 1}
        pts |= set(int(x) for x in rng.integers(v * inner, n, size=2))
    return np.array(sorted(pts), dtype=np.int64)


def sampled_check_rs(job, seed=0, per=6, scale=None, ranks=None, outputs=None):
    """Sampled shard elements of every (rank, param) against the oracle, one
    element at a time from host-regenerated inputs.  `ranks` restricts the
    check to some ranks; `outputs[r]` (P tensors) replaces job.shards[r],
    e.g. the output of a single-rank reduce-scatter."""
    wl = job.wl
    scale = wl.scale if scale is None else scale
    ranks = list(range(job.N)) if ranks is None else list(ranks)
    outputs = {} if outputs is None else outputs
    rng = np.random.default_rng(seed)
    checked = 0
    for p in range(job.P):
        d0, inner = job.dims[p]
        c = job.chunk[p]
        per_rank = [sample_indices(rng, job, p, r, per) for r in ranks]
        rows = [r * c * inner + idx for r, idx in zip(ranks, per_rank)]
        # source index of every sample in the full gradient
        src = np.concatenate(rows) if rows else np.zeros(0, np.int64)
        valid = src < d0 * inner
        vals = np.stack([wl.host_grad_at(k, p, np.where(valid, src, 0)) for k in range(job.N)])
        pos = 0
        for r, idx in zip(ranks, per_rank):
            if idx.size == 0:
                continue
            shard = outputs[r][p] if r in outputs else job.shards[r][p]
            got = _bits32(shard[torch.from_numpy(idx).to(job.device)])
            for t, e in enumerate(idx):
                if valid[pos + t]:
                    want = np.float32(oracle.rs_element(vals[:, pos + t], scale))
                else:
                    want = np.float32(0.0)
                assert got[t] == want.view(np.uint32), \
                    f"RS param {p} rank {r} elem {e}: got {got[t]:08x} want {want.view(np.uint32):08x}"
            pos += idx.size
            checked += idx.size
    return checked


def sampled_check_ag(job, seed=0, per=16):
    """Sampled parameter elements: value == the generator's full-parameter
    value (all-gather + placement is the identity), and the oracle's source
    index of that element in the rank-major buffer holds the same bits."""
    wl = job.wl
    rng = np.random.default_rng(seed)
    offs, S = oracle.layout(wl.shapes, job.N, job.align)
    checked = 0
    for p in range(job.P):
        d0, inner = job.dims[p]
        n = d0 * inner
        if n == 0:
            continue
        c = job.chunk[p]
        idx = {0, n - 1} | set(int(x) for x in rng.integers(0, n, size=per))
        idx |= {min(n - 1, r * c * inner) for r in range(job.N)}  # first element of each chunk
        idx = np.array(sorted(idx), dtype=np.int64)
        got = _bits16(job.params[p][torch.from_numpy(idx).to(job.device)])
        want = wl.host_param_value_at(p, idx)
        assert np.array_equal(got, want), f"placement param {p}"
        srcs = np.array([oracle.ag_source_index(job.N, wl.shapes[p], offs[p], S, e // inner, e % inner)
                         for e in idx], dtype=np.int64)
        buf_vals = _bits16(job.gathered[torch.from_numpy(srcs).to(job.device)])
        assert np.array_equal(buf_vals, want), f"oracle source index, param {p}"
        checked += idx.size
    return checked


def torch_check_rs(job, scale=None):
    """Every element against a plain PyTorch fp32 reference on the GPU: the
    same rank-order fp32 sum and multiply, then the dim-0 split with padding."""
    wl = job.wl
    scale = wl.scale if scale is None else scale
    for p in range(job.P):
        d0, inner = job.dims[p]
        c = job.chunk[p]
        acc = torch.zeros(d0 * inner, dtype=torch.float32, device=job.device)
        for k in range(job.N):
            acc += job.grads[k][p].view(torch.bfloat16).float()
        acc *= scale
        for r in range(job.N):
            v = max(0, min(c, d0 - r * c)) * inner
            sh = job.shards[r][p]
            assert torch.equal(sh[:v].view(torch.int32), acc[r * c * inner: r * c * inner + v].view(torch.int32)), \
                f"RS vs torch: param {p} rank {r}"
            if sh.numel() > v:
                assert bool((sh[v:].view(torch.int32) == 0).all()), f"padding of param {p} rank {r}"
        del acc


def torch_check_ag(job):
    """Every parameter element against a PyTorch gather of its chunks."""
    for p in range(job.P):
        d0, inner = job.dims[p]
        c = job.chunk[p]
        o = job.layout.param_offset(p)
        parts = []
        for r in range(job.N):
            v = max(0, min(c, d0 - r * c)) * inner
            parts.append(job.gathered[r * job.S + o: r * job.S + o + v])
        want = torch.cat(parts) if parts else job.params[p][:0]
        assert torch.equal(job.params[p], want), f"placement vs torch: param {p}"


# ---------------------------------------------------------------- single-rank RS and AG input pack
def guarded(n, dtype, device, canary):
    """A device buffer of n elements inside 256-byte canary bands."""
    g = 256 // torch.tensor([], dtype=dtype).element_size()
    buf = torch.full((n + 2 * g,), canary, dtype=dtype, device=device)
    return buf, buf[g: g + n], g


def check_rank_rs(job, rank, outs, scale=None):
    """Rank `rank`'s shards bit-exact against the oracle's single-rank RS."""
    wl = job.wl
    scale = wl.scale if scale is None else scale
    grads = [[wl.host_grad(k, p) for p in range(job.P)] for k in range(job.N)]
    want = oracle.rs_rank(wl.shapes, job.N, grads, scale, rank)
    for p in range(job.P):
        got = _bits32(outs[p])
        assert np.array_equal(got, want[p].view(np.uint32)), f"rank RS: rank {rank} param {p}"


def host_pack(job, ranks):
    """The oracle's pack of host-regenerated fp32 shards into a sentinel buffer."""
    wl = job.wl
    offs, S = oracle.layout(wl.shapes, job.N, job.align)
    buf = np.full(job.N * S, SENTINEL_BF16, dtype=np.uint16)
    for r in ranks:
        src = [wl.host_shard_f32(r, p, job.shard_numel[p]) for p in range(job.P)]
        oracle.ag_pack(wl.shapes, job.N, offs, S, r, src, buf)
    return buf


def check_pack(job, ranks):
    got = _bits16(job.packed)
    want = host_pack(job, ranks)
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        raise AssertionError(f"pack mismatch at {bad.size} slots, first {bad[0]}: "
                             f"got {got[bad[0]]:04x} want {want[bad[0]]:04x}")


def sampled_check_pack(job, seed=0, per=16):
    """Sampled slots of every (rank, param) block against the oracle rounding."""
    wl = job.wl
    rng = np.random.default_rng(seed)
    offs, S = oracle.layout(wl.shapes, job.N, job.align)
    checked = 0
    for p in range(job.P):
        n = job.shard_numel[p]
        if n == 0:
            continue
        for r in range(job.N):
            idx = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, size=per)]))
            src = wl.host_shard_f32(r, p, int(idx.max()) + 1)[idx]
            want = oracle.f32_to_bf16(src)
            pos = torch.from_numpy(r * S + offs[p] + idx).to(job.device)
            got = _bits16(job.packed[pos])
            assert np.array_equal(got, want), f"pack param {p} rank {r}"
            checked += idx.size
    return checked
