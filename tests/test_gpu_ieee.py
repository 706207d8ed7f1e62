"""IEEE special values and every rank count of the TMA-staged reduce-scatter,
through the C ABI, against the CPU oracle.

- Reduce-scatter (all four entry points: all ranks, one rank, from staged
  slots, and the no-allocation form) in every mode, on gradients holding
  subnormals, signed zeros, infinities, NaNs with payloads, values whose
  fp32 sum overflows and cancellations whose result depends on ascending
  rank order.  Every shard element is compared bit for bit with the oracle;
  a NaN matches a NaN (payloads differ between CPU and GPU arithmetic).
  A build that flushed subnormals, started the sum from -0.0f, fused the
  scale into an add or summed in another order fails here.
- Placement and Slot-Reuse staging (bit copies) in every mode, copy engines
  included, on uniformly random 16-bit patterns: every NaN payload must
  arrive unchanged.
- The TMA-staged reduce-scatter at N = 100, 257 and 512 (the largest N it
  takes), capped and over every SM.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gpu_checks  # noqa: E402
import ieee_cases  # noqa: E402
import oracle  # noqa: E402
from synth import SENTINEL_BF16  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only hosts
    pytest.skip("no CUDA device", allow_module_level=True)

import layout_aware_collectives_gb300 as tide  # noqa: E402

RS_MODES = [("uncapped", tide.TIDE_MODE_UNCAPPED, 0), ("capped1", tide.TIDE_MODE_CAPPED, 1),
            ("capped7", tide.TIDE_MODE_CAPPED, 7), ("bulk_cap3", tide.TIDE_MODE_BULK, 3),
            ("bulk", tide.TIDE_MODE_BULK, 0)]
COPY_MODES = [("uncapped", tide.TIDE_MODE_UNCAPPED, 0), ("capped2", tide.TIDE_MODE_CAPPED, 2),
              ("bulk", tide.TIDE_MODE_BULK, 0), ("bulk_cap3", tide.TIDE_MODE_BULK, 3),
              ("copy_engine", tide.TIDE_MODE_COPY_ENGINE, 0)]
CANARY32 = -0x5A5A5A5B
CANARY16 = 0x7FA5  # fits in int16 as is


def dev_u16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16).copy()).cuda()


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


class Outputs:
    """Guarded fp32 outputs (canary bands on both sides of each)."""

    def __init__(self, sizes):
        self.bufs = [gpu_checks.guarded(n, torch.int32, "cuda", CANARY32) for n in sizes]
        self.t = [b[1].view(torch.float32) for b in self.bufs]

    def intact(self) -> bool:
        return all(bool((buf[:g] == CANARY32).all()) and bool((buf[g + v.numel():] == CANARY32).all())
                   for buf, v, g in self.bufs)


def compare_f32(got_t: torch.Tensor, want: np.ndarray, where: str) -> None:
    """Bit-exact, except that any NaN matches any NaN."""
    got = got_t.view(torch.int32).cpu().numpy().view(np.uint32)
    exp = np.ascontiguousarray(want, dtype=np.float32).view(np.uint32)
    assert got.shape == exp.shape, where
    ok = (got == exp) | (np.isnan(got.view(np.float32)) & np.isnan(exp.view(np.float32)))
    if not ok.all():
        i = int(np.flatnonzero(~ok)[0])
        raise AssertionError(f"{where}: {int((~ok).sum())} elements differ, first at {i}: "
                             f"got {got[i]:08x} want {exp[i]:08x}")


def _all_forms(lay, align, n, shps, host, grads_dev, scale, modes, ranks=None):
    """Every reduce-scatter entry point in every mode against the oracle."""
    P = len(shps)
    shard_n = [lay.shard_numel(p) for p in range(P)]
    offs, S = oracle.layout(shps, n, align)
    assert S == lay.block_numel
    want = oracle.rs(shps, n, host, scale)
    gptrs = [grads_dev[k][p] for k in range(n) for p in range(P)]
    ranks = sorted({0, n - 1}) if ranks is None else ranks
    want_slots = []
    for k in range(n):
        slot = np.full(n * S, SENTINEL_BF16, dtype=np.uint16)
        want_slots.append(oracle.rs_stage(shps, n, offs, S, host[k], slot))
    for name, mode, cap in modes:
        lay.set_mode(mode, cap)
        tag = f"N={n} scale={scale} mode={name}"
        # all ranks, and the no-allocation form of the same call
        for form in ("rs", "noalloc"):
            out = Outputs([shard_n[p] for _ in range(n) for p in range(P)])
            call = lay.reduce_scatter if form == "rs" else lay.reduce_scatter_noalloc
            call(gptrs, out.t, scale)
            torch.cuda.synchronize()
            for r in range(n):
                for p in range(P):
                    compare_f32(out.t[r * P + p], want[r][p], f"{tag} {form} rank {r} param {p}")
            assert out.intact(), f"{tag} {form}: write outside a shard"
        # one rank
        for r in ranks:
            out = Outputs(shard_n)
            lay.reduce_scatter_rank(r, gptrs, out.t, scale)
            torch.cuda.synchronize()
            for p in range(P):
                compare_f32(out.t[p], want[r][p], f"{tag} single rank {r} param {p}")
            assert out.intact(), f"{tag} single rank {r}: write outside a shard"
        # Slot-Reuse staging (a bit copy: NaN payloads kept), then the staged RS
        slots = [torch.full((n * S,), SENTINEL_BF16, dtype=torch.int16, device="cuda")
                 for _ in range(n)]
        for k in range(n):
            lay.stage([grads_dev[k][p] for p in range(P)], slots[k])
        torch.cuda.synchronize()
        for k in range(n):
            assert np.array_equal(bits16(slots[k]), want_slots[k]), f"{tag} staging of rank {k}"
        out = Outputs([shard_n[p] for _ in range(n) for p in range(P)])
        lay.reduce_scatter_staged(slots, out.t, scale)
        torch.cuda.synchronize()
        for r in range(n):
            for p in range(P):
                compare_f32(out.t[r * P + p], want[r][p], f"{tag} staged rank {r} param {p}")
        assert out.intact(), f"{tag} staged: write outside a shard"
        lay.check_device()


@pytest.mark.parametrize("align", [8, 1])
@pytest.mark.parametrize("n", [1, 3, 4, 8, 13, 16, 64, 100])
def test_rs_special_values(n, align):
    shps = ieee_cases.shapes(n)
    host = ieee_cases.grads(n, shps)
    with tide.Layout(shps, n, align_elems=align) as lay:
        grads_dev = [[dev_u16(host[k][p]) for p in range(len(shps))] for k in range(n)]
        # 1/N and a scale whose products round (0.3 is not a power of two)
        for scale in (1.0 / n, 0.3):
            _all_forms(lay, align, n, shps, host, grads_dev, scale, RS_MODES)
        # a negative scale turns the +0 of all-(-0) columns into -0 on both sides
        _all_forms(lay, align, n, shps, host, grads_dev, -1.0, RS_MODES[:1])
        # the staging copy in copy-engine mode moves the special values bit for bit
        lay.set_mode(tide.TIDE_MODE_COPY_ENGINE)
        offs, S = oracle.layout(shps, n, align)
        for k in (0, n - 1):
            slot = torch.full((n * S,), SENTINEL_BF16, dtype=torch.int16, device="cuda")
            lay.stage(grads_dev[k], slot)
            torch.cuda.synchronize()
            want = oracle.rs_stage(shps, n, offs, S, host[k], np.full(n * S, SENTINEL_BF16, np.uint16))
            assert np.array_equal(bits16(slot), want), f"copy-engine staging of rank {k}"


@pytest.mark.parametrize("align", [8, 1])
@pytest.mark.parametrize("n", [1, 4, 13, 64])
def test_placement_and_staging_keep_nan_payloads(n, align):
    """Random 16-bit patterns (all NaN payloads, signalling NaNs,
    subnormals, infinities) through placement and staging in every mode."""
    rng = np.random.default_rng(100 + n)
    shps = ieee_cases.shapes(n) + [(0, 8), (2 * n, 3, 5)]
    P = len(shps)
    offs, S = oracle.layout(shps, n, align)
    buf = np.full(n * S, SENTINEL_BF16, dtype=np.uint16)
    for p, s in enumerate(shps):
        d0 = s[0] if len(s) else 1
        inner = int(np.prod(s[1:])) if len(s) > 1 else 1
        for r in range(n):
            v = oracle.valid_rows(d0, n, r) * inner
            buf[r * S + offs[p]: r * S + offs[p] + v] = ieee_cases.random_bits(rng, v, SENTINEL_BF16)
    want = oracle.ag_place(shps, n, buf, offs, S)
    grad_host = [ieee_cases.random_bits(rng, int(np.prod(s)) if len(s) else 1, SENTINEL_BF16) for s in shps]
    want_slot = oracle.rs_stage(shps, n, offs, S, grad_host, np.full(n * S, SENTINEL_BF16, np.uint16))
    with tide.Layout(shps, n, align_elems=align) as lay:
        assert lay.block_numel == S
        gathered = dev_u16(buf)
        grads = [dev_u16(g) for g in grad_host]
        g16 = 128
        for name, mode, cap in COPY_MODES:
            lay.set_mode(mode, cap)
            bufs = [torch.full((w.size + 2 * g16,), CANARY16, dtype=torch.int16, device="cuda") for w in want]
            params = [b[g16: g16 + w.size] for b, w in zip(bufs, want)]
            lay.place(gathered, params)
            slot = torch.full((n * S,), SENTINEL_BF16, dtype=torch.int16, device="cuda")
            lay.stage(grads, slot)
            torch.cuda.synchronize()
            lay.check_device()
            for p in range(P):
                got = bits16(params[p])
                assert np.array_equal(got, want[p]), f"{name}: placement of param {p}"
                assert not np.any(got == SENTINEL_BF16), f"{name}: padding reached param {p}"
                assert bool((bufs[p][:g16] == CANARY16).all()) and bool((bufs[p][g16 + want[p].size:] == CANARY16).all())
            assert np.array_equal(bits16(slot), want_slot), f"{name}: staging"


@pytest.mark.parametrize("align", [8, 1])
@pytest.mark.parametrize("n", [100, 257, 512])
def test_tma_staged_rs_many_ranks(n, align):
    """The TMA-staged reduce-scatter at N = 100, 257 (odd, not a power of
    two) and 512, its largest N (96-element rank slices, a two-stage ring),
    capped and over every SM: every element of every form against the oracle."""
    rng = np.random.default_rng(n)
    shps = [(n + 3, 16), (2 * n - 1, 8), (7,), (3 * n, 24), (n // 2, 40)]
    host = [[(rng.standard_normal(int(np.prod(s))).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
             for s in shps] for _ in range(n)]
    with tide.Layout(shps, n, align_elems=align) as lay:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        lay.set_mode(tide.TIDE_MODE_BULK, 0)
        tiles = len(lay.tiles(tide.TIDE_OP_RS))
        assert lay.launch_shape(tide.TIDE_OP_RS) == (min(sms, tiles), 288), "TMA-staged kernel not selected"
        grads_dev = [[dev_u16(host[k][p]) for p in range(len(shps))] for k in range(n)]
        _all_forms(lay, align, n, shps, host, grads_dev, 1.0 / n,
                   [("bulk", tide.TIDE_MODE_BULK, 0), ("bulk_cap5", tide.TIDE_MODE_BULK, 5)],
                   ranks=[0, n // 2, n - 1])
