"""CUDA path (through the C ABI) against the CPU oracle.

Small jobs are compared element by element over every output; full-size
workloads on sampled outputs the oracle computes one by one, plus a PyTorch
fp32 reference over every element.  Reduce-scatter is summed in rank order
on both sides, so every comparison is bit-exact.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gpu_checks  # noqa: E402
import synth  # noqa: E402
from synth.device import DeviceJob  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU-only hosts
    pytest.skip("no CUDA device", allow_module_level=True)

import layout_aware_collectives_gb300 as tide  # noqa: E402

MODES = [("uncapped", tide.TIDE_MODE_UNCAPPED, 0)] + [
    (f"capped{c}", tide.TIDE_MODE_CAPPED, c) for c in (1, 2, 7, 8, 32, 120)] + [
    ("bulk_cap3", tide.TIDE_MODE_BULK, 3), ("bulk", tide.TIDE_MODE_BULK, 0)]


def run(job, rs_mode=None, ag_mode=None, scale=None):
    lay = job.layout
    if rs_mode is not None:
        lay.set_mode(*rs_mode)
    lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), job.wl.scale if scale is None else scale)
    if ag_mode is not None:
        lay.set_mode(*ag_mode)
    lay.place(job.gathered, job.param_ptrs())
    torch.cuda.synchronize()


@pytest.fixture
def tiny_job():
    wl = synth.tiny()
    lay = tide.Layout(wl.shapes, wl.num_ranks)
    job = DeviceJob(wl, lay)
    yield job
    lay.close()


def test_device_generator_matches_host(tiny_job):
    job = tiny_job
    for k in range(job.N):
        for p in range(job.P):
            got = job.grads[k][p].cpu().numpy().view(np.uint16)
            assert np.array_equal(got, job.wl.host_grad(k, p)), (k, p)


@pytest.mark.parametrize("mode", MODES, ids=[m[0] for m in MODES])
def test_tiny_full_parity(tiny_job, mode):
    job = tiny_job
    gpu_checks.check_layout(job)
    run(job, rs_mode=mode[1:], ag_mode=mode[1:])
    gpu_checks.full_check_rs(job)
    gpu_checks.full_check_ag(job)
    assert job.guards_intact()


def test_tiny_copy_engine_placement(tiny_job):
    job = tiny_job
    job.layout.set_mode(tide.TIDE_MODE_COPY_ENGINE)
    job.layout.place(job.gathered, job.param_ptrs())
    torch.cuda.synchronize()
    gpu_checks.full_check_ag(job)
    assert job.guards_intact()
    with pytest.raises(tide.TideError) as e:
        job.layout.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), 0.25)
    assert e.value.status == tide.TIDE_ERR_UNSUPPORTED


def test_repeated_calls_and_pointer_cache(tiny_job):
    """Same buffers (cache hit), fresh outputs (miss) and more distinct
    pointer sets than cache slots (eviction) all give the oracle's result."""
    job = tiny_job
    for _ in range(3):
        job.reset_outputs()
        run(job)
        gpu_checks.full_check_rs(job)
    wl = job.wl
    jobs = [DeviceJob(wl, job.layout, fill=False) for _ in range(10)]
    for j in jobs:
        j.grads = job.grads
        j.gathered = job.gathered
        run(j)
    for j in jobs[::3]:
        gpu_checks.full_check_rs(j)
        gpu_checks.full_check_ag(j)


def test_other_stream(tiny_job):
    job = tiny_job
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    job.layout.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), job.wl.scale, stream=s)
    job.layout.place(job.gathered, job.param_ptrs(), stream=s)
    s.synchronize()
    gpu_checks.full_check_rs(job)
    gpu_checks.full_check_ag(job)


@pytest.mark.parametrize("mode", MODES[:2] + [("bulk", tide.TIDE_MODE_BULK, 0)], ids=lambda m: m[0])
def test_low_priority_stream_next_to_gemm(tiny_job, mode):
    """The step on a low-priority stream while bf16 GEMMs run on a
    high-priority one (the arrangement that keeps the GEMM's slowdown small):
    same bits as the oracle."""
    job = tiny_job
    job.layout.set_mode(*mode[1:])
    least, greatest = torch.cuda.Stream.priority_range()
    s_lo = torch.cuda.Stream(priority=least)
    s_hi = torch.cuda.Stream(priority=greatest)
    a = torch.randn(2048, 2048, dtype=torch.bfloat16, device="cuda")
    c = torch.empty_like(a)
    torch.cuda.synchronize()
    with torch.cuda.stream(s_hi):
        for _ in range(4):
            torch.matmul(a, a, out=c)
    for _ in range(3):
        job.layout.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), job.wl.scale, stream=s_lo)
        job.layout.place(job.gathered, job.param_ptrs(), stream=s_lo)
    torch.cuda.synchronize()
    job.layout.check_device()
    gpu_checks.full_check_rs(job)
    gpu_checks.full_check_ag(job)


def _ragged_cases():
    rng = np.random.default_rng(11)
    cases = []
    for n in (1, 2, 3, 5, 8, 13, 16, 64):
        shapes = [(int(rng.integers(1, 3 * n + 5)), int(rng.integers(1, 40)))
                  for _ in range(4)]
        shapes += [(n - 1 if n > 1 else 1, 24), (3 * n + 1,), (), (0, 16), (7, 0, 3),
                   (2 * n, 3, 5)]
        cases.append((n, shapes))
    return cases


@pytest.mark.parametrize("align", [8, 1])
@pytest.mark.parametrize("case", _ragged_cases(), ids=lambda c: f"N{c[0]}")
def test_ragged_shapes_full_parity(case, align):
    """d0 < N (empty ranks), d0 not a multiple of N, inner not a multiple of
    8, 0-dim scalars, zero-size tensors, 3-D tensors, unaligned offsets."""
    n, shapes = case
    wl = synth.custom(f"ragged{n}", n, shapes, sigma=0.5, seed=n)
    with tide.Layout(wl.shapes, n, align_elems=align) as lay:
        job = DeviceJob(wl, lay, align=align)
        gpu_checks.check_layout(job)
        for mode in MODES[:3] + MODES[-1:]:
            job.reset_outputs()
            run(job, rs_mode=mode[1:], ag_mode=mode[1:], scale=0.3)
            gpu_checks.full_check_rs(job, scale=0.3)
            gpu_checks.full_check_ag(job)
            assert job.guards_intact()
        # copy-engine placement: 2-D copies for the ranks with a full chunk, one
        # copy for a partial chunk, nothing for empty ranks or zero-size tensors
        lay.set_mode(tide.TIDE_MODE_COPY_ENGINE)
        job.reset_outputs()
        lay.place(job.gathered, job.param_ptrs())
        torch.cuda.synchronize()
        gpu_checks.full_check_ag(job)
        assert job.guards_intact()


def _rank_rs_and_pack(job, modes, scale=None):
    scale = job.wl.scale if scale is None else scale
    job.make_pack_inputs()
    for mode in modes:
        job.layout.set_mode(*mode[1:])
        for r in range(job.N):
            bufs = [gpu_checks.guarded(n, torch.int32, job.device, -0x5A5A5A5B)
                    for n in job.shard_numel]
            outs = [b[1].view(torch.float32) for b in bufs]
            job.layout.reduce_scatter_rank(r, job.grad_ptrs(), outs, scale)
            torch.cuda.synchronize()
            gpu_checks.check_rank_rs(job, r, outs, scale)
            for buf, view, g in bufs:
                assert bool((buf[:g] == -0x5A5A5A5B).all()) and bool((buf[g + view.numel():] == -0x5A5A5A5B).all())
        # pack rank by rank (each call writes only its own block), then all at once
        job.packed.fill_(0x7FC1)
        for r in range(job.N):
            job.layout.pack(r, job.pack_src_ptrs(r), job.packed)
            torch.cuda.synchronize()
            gpu_checks.check_pack(job, range(r + 1))
        job.packed.fill_(0x7FC1)
        job.layout.pack(-1, job.pack_src_ptrs(), job.packed)
        torch.cuda.synchronize()
        gpu_checks.check_pack(job, range(job.N))


@pytest.mark.parametrize("mode", MODES, ids=[m[0] for m in MODES])
def test_tiny_rank_rs_and_pack(tiny_job, mode):
    _rank_rs_and_pack(tiny_job, [mode])


@pytest.mark.parametrize("align", [8, 1])
@pytest.mark.parametrize("case", _ragged_cases(), ids=lambda c: f"N{c[0]}")
def test_ragged_rank_rs_and_pack(case, align):
    n, shapes = case
    wl = synth.custom(f"ragged{n}", n, shapes, sigma=0.5, seed=n)
    with tide.Layout(wl.shapes, n, align_elems=align) as lay:
        job = DeviceJob(wl, lay, align=align)
        _rank_rs_and_pack(job, MODES[:2], scale=0.3)


def _staged(job, modes, scale=None):
    """Stage every rank's gradients into its slot, reduce-scatter from the
    slots: slots equal the oracle's staging, shards the oracle's RS."""
    import oracle

    wl = job.wl
    scale = wl.scale if scale is None else scale
    offs, S = oracle.layout(wl.shapes, job.N, job.align)
    job.make_slots()
    for mode in modes:
        lay = job.layout
        lay.set_mode(*mode[1:])
        for k in range(job.N):
            job.slots[k].fill_(0x7FC1)
            lay.stage([job.grads[k][p] for p in range(job.P)], job.slots[k])
        torch.cuda.synchronize()
        for k in range(job.N):
            want = np.full(job.N * S, 0x7FC1, dtype=np.uint16)
            oracle.rs_stage(wl.shapes, job.N, offs, S, [wl.host_grad(k, p) for p in range(job.P)], want)
            assert np.array_equal(job.slots[k].cpu().numpy().view(np.uint16), want), (mode[0], k)
        if mode[1] == tide.TIDE_MODE_COPY_ENGINE:
            continue
        job.reset_outputs()
        lay.reduce_scatter_staged(job.slots, job.shard_ptrs(), scale)
        torch.cuda.synchronize()
        gpu_checks.full_check_rs(job, scale=scale)
        assert job.guards_intact()


def test_capped_forms_on_both_sides_of_half_the_sms(tiny_job):
    """Capped grids of at most half the SMs hand tiles to single warps and
    larger ones to whole CTAs: caps just below, at and above that boundary,
    and one CTA per SM, give the oracle's results in every capped operation
    (reduce-scatter, placement, pack, staging, staged reduce-scatter).  The
    tiny block's lists hold more tiles than any cap here, so each cap is the
    launched grid."""
    job = tiny_job
    lay = job.layout
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    half = sms // 2
    for op in (tide.TIDE_OP_RS, tide.TIDE_OP_AG, tide.TIDE_OP_PACK, tide.TIDE_OP_STAGE, tide.TIDE_OP_STAGED_RS):
        assert len(lay.tiles(op)) > sms, op
    caps = [(f"capped{c}", tide.TIDE_MODE_CAPPED, c) for c in (half - 1, half, half + 1, sms)]
    for mode in caps:
        lay.set_mode(*mode[1:])
        assert lay.launch_shape(tide.TIDE_OP_RS) == (mode[2], 1024)
        job.reset_outputs()
        run(job)
        gpu_checks.full_check_rs(job)
        gpu_checks.full_check_ag(job)
        assert job.guards_intact()
    _rank_rs_and_pack(job, caps[1:3])
    _staged(job, caps[1:3])


STAGE_MODES = MODES[:3] + [("bulk", tide.TIDE_MODE_BULK, 0),
                           ("copy_engine", tide.TIDE_MODE_COPY_ENGINE, 0)]


@pytest.mark.parametrize("mode", STAGE_MODES, ids=[m[0] for m in STAGE_MODES])
def test_tiny_staged_rs(tiny_job, mode):
    _staged(tiny_job, [mode])


@pytest.mark.parametrize("align", [8, 1])
@pytest.mark.parametrize("case", _ragged_cases(), ids=lambda c: f"N{c[0]}")
def test_ragged_staged_rs(case, align):
    n, shapes = case
    wl = synth.custom(f"ragged{n}", n, shapes, sigma=0.5, seed=n)
    with tide.Layout(wl.shapes, n, align_elems=align) as lay:
        job = DeviceJob(wl, lay, align=align)
        _staged(job, [MODES[0], MODES[1], STAGE_MODES[-2], STAGE_MODES[-1]], scale=0.3)


def test_pack_special_values():
    """Ties, overflow, subnormals, infinities and NaNs through the device pack."""
    bits = np.array([0x3F800000, 0x3F808000, 0x3F818000, 0x3F808001, 0x3F807FFF, 0xBF818000,
                     0x7F7FFFFF, 0x7F7F7FFF, 0x80000000, 0x00000001, 0x00008000, 0x00018000,
                     0x7F800000, 0xFF800000, 0x7FC00000, 0x7F800001, 0xFFC00001, 0x00000000],
                    dtype=np.uint32)
    n = bits.size
    with tide.Layout([(n,)], 1) as lay:
        src = torch.from_numpy(bits.view(np.int32).copy()).cuda().view(torch.float32)
        out = torch.zeros(lay.block_numel, dtype=torch.int16, device="cuda")
        lay.pack(0, [src], out)
        torch.cuda.synchronize()
        got = out[:n].cpu().numpy().view(np.uint16)
        import oracle
        assert np.array_equal(got, oracle.f32_to_bf16(bits.view(np.float32)))


def test_empty_layout():
    with tide.Layout([], 4) as lay:
        lay.reduce_scatter([], [], 0.25)
        lay.place(None, [])
        torch.cuda.synchronize()
    with tide.Layout([(0, 8)], 4) as lay:
        lay.reduce_scatter([None] * 4, [None] * 4, 0.25)
        lay.place(None, [None])
        torch.cuda.synchronize()


FULL = ["llama8b", "llama70b", "moe", "sweep16", "sweep32", "sweep64"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_parity(name):
    """Full-size workloads in the bench's launch configuration (uncapped):
    sampled elements of every (rank, param) against the oracle, every element
    against a PyTorch fp32 reference.  Then every other form and mode on the
    same inputs, each against the oracle (sampled) and the PyTorch reference:
    single-rank RS, pack, Slot-Reuse staging + staged RS, CTA-capped 64,
    TMA-staged / TMA-copy modes capped and over every SM, and copy-engine
    placement."""
    wl = synth.WORKLOADS[name]()
    with tide.Layout(wl.shapes, wl.num_ranks) as lay:
        job = DeviceJob(wl, lay, guard=False)
        gpu_checks.check_layout(job)
        run(job)
        assert gpu_checks.sampled_check_rs(job) > 0
        assert gpu_checks.sampled_check_ag(job) > 0
        gpu_checks.torch_check_rs(job)
        gpu_checks.torch_check_ag(job)
        for r in (0, job.N - 1):
            outs = [torch.full((n,), float("nan"), dtype=torch.float32, device="cuda") for n in job.shard_numel]
            lay.reduce_scatter_rank(r, job.grad_ptrs(), outs, wl.scale)
            torch.cuda.synchronize()
            assert gpu_checks.sampled_check_rs(job, seed=10 + r, ranks=[r], outputs={r: outs}) > 0
            for p in range(job.P):
                assert torch.equal(outs[p].view(torch.int32), job.shards[r][p].view(torch.int32)), (r, p)
            del outs
        job.make_pack_inputs()
        lay.pack(-1, job.pack_src_ptrs(), job.packed)
        torch.cuda.synchronize()
        assert gpu_checks.sampled_check_pack(job) > 0
        del job.pack_src, job.packed

        def clear_outputs():
            for row in job.shards:
                for s in row:
                    s.fill_(float("nan"))
            for prm in job.params:
                prm.fill_(0x7FA5)  # a bf16 NaN pattern the placement never writes

        # Slot-Reuse: stage every rank, reduce-scatter from the slots
        job.make_slots()
        for k in range(job.N):
            lay.stage([job.grads[k][p] for p in range(job.P)], job.slots[k])
        clear_outputs()
        lay.reduce_scatter_staged(job.slots, job.shard_ptrs(), wl.scale)
        torch.cuda.synchronize()
        assert gpu_checks.sampled_check_rs(job, seed=1) > 0
        gpu_checks.torch_check_rs(job)
        del job.slots

        # capped grids of at most half the SMs hand tiles to single warps; larger ones to whole CTAs
        for cap in (64, 152):
            lay.set_mode(tide.TIDE_MODE_CAPPED, cap)
            clear_outputs()
            run(job)
            assert gpu_checks.sampled_check_rs(job, seed=cap) > 0
            assert gpu_checks.sampled_check_ag(job, seed=cap) > 0
            gpu_checks.torch_check_rs(job)
            gpu_checks.torch_check_ag(job)
        # TMA bulk-staged reduce-scatter and bulk-copy placement, capped and over every SM
        for cap in (16, 0):
            lay.set_mode(tide.TIDE_MODE_BULK, cap)
            clear_outputs()
            run(job)
            lay.check_device()
            assert gpu_checks.sampled_check_rs(job, seed=3 + cap) > 0
            assert gpu_checks.sampled_check_ag(job, seed=3 + cap) > 0
            gpu_checks.torch_check_rs(job)
            gpu_checks.torch_check_ag(job)
        # copy-engine placement
        lay.set_mode(tide.TIDE_MODE_COPY_ENGINE)
        clear_outputs()
        lay.place(job.gathered, job.param_ptrs())
        torch.cuda.synchronize()
        assert gpu_checks.sampled_check_ag(job, seed=5) > 0
        gpu_checks.torch_check_ag(job)
        del job
        torch.cuda.empty_cache()


def test_int64_offsets():
    """A parameter of more than 2^31 elements: offsets past 32-bit range."""
    d0 = (1 << 31) // 4096 + 17
    wl = synth.custom("huge", 2, [(d0, 4096), (5,)], sigma=1e-3, seed=3)
    with tide.Layout(wl.shapes, 2) as lay:
        job = DeviceJob(wl, lay, guard=False)
        run(job)
        assert gpu_checks.sampled_check_rs(job, per=32) > 0
        assert gpu_checks.sampled_check_ag(job, per=64) > 0
        del job
        torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", [MODES[0], MODES[1], ("bulk", tide.TIDE_MODE_BULK, 0)], ids=lambda m: m[0])
def test_max_ranks(mode):
    """N = 4096, the most ranks a layout takes: the runtime-N reduce-scatter
    stages 2*N source pointers in 64 KiB of shared memory (above the 48 KiB
    launch default), most ranks own padding only, and the bulk mode falls
    back to the load/store kernel above 512 ranks.  Every element against
    the oracle, guard bands intact."""
    n = 4096
    wl = synth.custom("max_ranks", n, [(n + 3, 8), (5,), (2 * n, 3)], sigma=1e-2, seed=5)
    with tide.Layout(wl.shapes, n) as lay:
        lay.set_mode(*mode[1:])
        job = DeviceJob(wl, lay)
        run(job)
        lay.check_device()
        gpu_checks.full_check_rs(job)
        gpu_checks.full_check_ag(job)
        assert job.guards_intact()
        del job
        torch.cuda.empty_cache()


def test_zero_copy_host_buffers(tiny_job):
    """Inputs and outputs in pinned host memory, read and written by the
    kernels directly: same bits as the oracle."""
    import bench

    job = tiny_job
    h_g = [[g.cpu().pin_memory() for g in row] for row in job.grads]
    h_buf = job.gathered.cpu().pin_memory()
    h_s = [[torch.full_like(s.cpu(), float("nan")).pin_memory() for s in row] for row in job.shards]
    h_p = [torch.zeros_like(p.cpu()).pin_memory() for p in job.params]
    flat = [t for row in h_g for t in row] + [t for row in h_s for t in row] + h_p + [h_buf]
    if not bench._host_mapped(flat):
        pytest.skip("pinned host memory is not device-mapped here")
    job.layout.reduce_scatter([t for row in h_g for t in row], [t for row in h_s for t in row],
                              job.wl.scale)
    job.layout.place(h_buf, h_p)
    torch.cuda.synchronize()
    job.shards = h_s
    job.params = h_p
    job.gathered = h_buf
    gpu_checks.full_check_rs(job)
    gpu_checks.full_check_ag(job)


def test_launch_shapes(tiny_job):
    """Uncapped: one CTA of 512 threads per tile of each list.  Capped: `cap`
    CTAs of 1024 threads (fewer if the list is shorter).  Copy engine: no
    kernel for placement.  Bulk: one 32-thread placement CTA per tile and
    one 288-thread reduce-scatter CTA per SM, or `cap` of either."""
    lay = tiny_job.layout
    ops = (tide.TIDE_OP_RS, tide.TIDE_OP_AG, tide.TIDE_OP_PACK, tide.TIDE_OP_STAGE,
           tide.TIDE_OP_STAGED_RS)
    for op in ops:
        n = len(lay.tiles(op))
        assert n > 16
        assert lay.launch_shape(op) == (n, 512), op
    lay.set_mode(tide.TIDE_MODE_CAPPED, 16)
    for op in ops:
        assert lay.launch_shape(op) == (16, 1024), op
    lay.set_mode(tide.TIDE_MODE_CAPPED, 1 << 20)
    for op in ops:
        assert lay.launch_shape(op) == (len(lay.tiles(op)), 1024), op
    lay.set_mode(tide.TIDE_MODE_COPY_ENGINE)
    assert lay.launch_shape(tide.TIDE_OP_AG)[0] == 0
    lay.set_mode(tide.TIDE_MODE_BULK)
    assert lay.launch_shape(tide.TIDE_OP_AG) == (len(lay.tiles(tide.TIDE_OP_AG)), 32)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert lay.launch_shape(tide.TIDE_OP_RS) == (min(sms, len(lay.tiles(tide.TIDE_OP_RS))), 288)
    lay.set_mode(tide.TIDE_MODE_BULK, 3)
    assert lay.launch_shape(tide.TIDE_OP_AG) == (3, 32)
    assert lay.launch_shape(tide.TIDE_OP_RS) == (3, 288)
    lay.set_mode(tide.TIDE_MODE_UNCAPPED)


def test_bounded_wait_timeout_is_reported(tiny_job):
    """The bulk-copy kernel's waits are bounded: with the test hook set, its
    wait on a barrier nothing arrives on runs out after 1 ms, the kernel
    returns, and the host reads TIDE_ERR_TIMEOUT; the next call (hook off)
    completes and matches the oracle."""
    job = tiny_job
    lay = job.layout
    lay.set_mode(tide.TIDE_MODE_BULK)
    assert lay.launch_shape(tide.TIDE_OP_AG)[1] == 32
    lay.set_test_stall(1_000_000)
    lay.place(job.gathered, job.param_ptrs())
    with pytest.raises(tide.TideError) as e:
        lay.check_device()
    assert e.value.status == tide.TIDE_ERR_TIMEOUT
    lay.check_device()  # cleared
    # the bulk-staged reduce-scatter's waits too
    lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), job.wl.scale)
    with pytest.raises(tide.TideError) as e:
        lay.check_device()
    assert e.value.status == tide.TIDE_ERR_TIMEOUT
    lay.set_test_stall(0)
    job.reset_outputs()
    lay.place(job.gathered, job.param_ptrs())
    lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), job.wl.scale)
    lay.check_device()
    gpu_checks.full_check_ag(job)
    gpu_checks.full_check_rs(job)


def test_two_host_threads_share_a_layout(tiny_job):
    """Calls from two host threads on two streams with their own outputs
    (the layout serialises the host side; the streams run independently)."""
    import threading

    job = tiny_job
    other = DeviceJob(job.wl, job.layout, fill=False)
    other.grads, other.gathered = job.grads, job.gathered
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    errors = []

    def work(j, s):
        try:
            for _ in range(20):
                j.layout.reduce_scatter(j.grad_ptrs(), j.shard_ptrs(), j.wl.scale, stream=s)
                j.layout.place(j.gathered, j.param_ptrs(), stream=s)
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    ts = [threading.Thread(target=work, args=(j, s)) for j, s in zip((job, other), streams)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for j in (job, other):
        gpu_checks.full_check_rs(j)
        gpu_checks.full_check_ag(j)


def test_cuda_graph_capture_of_the_step(tiny_job):
    """After a first call (which sets the layout up on the device), the
    reduce-scatter and placement calls can be captured into a CUDA graph and
    replayed; the replay gives the oracle's result."""
    job = tiny_job
    lay = job.layout
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g_ptrs, s_ptrs, p_ptrs = (tide.PointerTable(job.grad_ptrs()), tide.PointerTable(job.shard_ptrs()),
                              tide.PointerTable(job.param_ptrs()))
    lay.reduce_scatter(g_ptrs, s_ptrs, job.wl.scale, stream=s)
    lay.place(job.gathered, p_ptrs, stream=s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        lay.reduce_scatter(g_ptrs, s_ptrs, job.wl.scale, stream=s)
        lay.place(job.gathered, p_ptrs, stream=s)
    torch.cuda.synchronize()
    for _ in range(2):
        job.reset_outputs()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        gpu_checks.full_check_rs(job)
        gpu_checks.full_check_ag(job)
        assert job.guards_intact()
    # more pointer sets than cache slots after the capture: the tables the
    # graph reads stay put, so its replay is still right
    others = [DeviceJob(job.wl, lay, fill=False) for _ in range(10)]
    for o in others:
        o.grads, o.gathered = job.grads, job.gathered
        lay.reduce_scatter(o.grad_ptrs(), o.shard_ptrs(), job.wl.scale)
        lay.place(o.gathered, o.param_ptrs())
    gpu_checks.full_check_rs(others[-1])
    job.reset_outputs()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    gpu_checks.full_check_rs(job)
    gpu_checks.full_check_ag(job)
    # a pointer set never used before cannot be first seen inside a capture
    fresh = DeviceJob(job.wl, lay, fill=False)
    g2 = torch.cuda.CUDAGraph()
    import warnings

    with warnings.catch_warnings():
        warnings.simplefilter("ignore")  # the refused call leaves the capture empty
        with torch.cuda.graph(g2, stream=s):
            with pytest.raises(tide.TideError) as e:
                lay.reduce_scatter(fresh.grad_ptrs(), fresh.shard_ptrs(), job.wl.scale, stream=s)
    assert e.value.status == tide.TIDE_ERR_UNSUPPORTED
    del graph, g2
    lay.close()
    torch.zeros(1, device="cuda").add_(1)  # no CUDA error left behind by the library
    torch.cuda.synchronize()


def test_first_call_does_not_wait_for_the_stream():
    """A layout's first compute calls (device set-up, tile-list and pointer-
    table uploads) enqueue their copies on the caller's stream and return
    while that stream is still busy; the results then match the oracle."""
    import time

    wl = synth.tiny()
    with tide.Layout(wl.shapes, wl.num_ranks) as lay:
        job = DeviceJob(wl, lay)
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            torch.cuda._sleep(3_000_000_000)  # ~1.5 s of device time on s
        t0 = time.perf_counter()
        lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), wl.scale, stream=s)
        lay.place(job.gathered, job.param_ptrs(), stream=s)
        host_s = time.perf_counter() - t0
        busy = not s.query()
        s.synchronize()
        assert busy, "the stream finished before the calls returned; the check says nothing"
        assert host_s < 0.5, f"first calls held the host for {host_s:.3f} s"
        gpu_checks.full_check_rs(job)
        gpu_checks.full_check_ag(job)
        # a second stream is ordered after the upload made on the first
        other = DeviceJob(wl, lay, fill=False)
        other.grads, other.gathered = job.grads, job.gathered
        s2 = torch.cuda.Stream()
        lay.reduce_scatter(other.grad_ptrs(), other.shard_ptrs(), wl.scale, stream=s2)
        s2.synchronize()
        gpu_checks.full_check_rs(other)


def test_first_call_inside_capture_is_refused():
    """Setting a layout up on the device cannot be captured: the call is
    refused before it enqueues anything, the capture stays usable, and the
    same call outside the capture then works."""
    import warnings

    wl = synth.tiny()
    with tide.Layout(wl.shapes, wl.num_ranks) as lay:
        job = DeviceJob(wl, lay)
        x = torch.zeros(16, device="cuda")
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            with torch.cuda.graph(g, stream=s):
                x.add_(1.0)
                with pytest.raises(tide.TideError) as e:
                    lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), wl.scale, stream=s)
        assert e.value.status == tide.TIDE_ERR_UNSUPPORTED
        g.replay()
        torch.cuda.synchronize()
        assert float(x[0]) == 1.0
        lay.reduce_scatter(job.grad_ptrs(), job.shard_ptrs(), wl.scale, stream=s)
        s.synchronize()
        gpu_checks.full_check_rs(job)
