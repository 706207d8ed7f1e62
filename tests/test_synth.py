"""Input generator checks (no GPU): distribution, structure and workload shapes."""
import numpy as np
import pytest

import synth
from oracle_pins import bf16_to_f32


def test_splitmix64_reference_values():
    # splitmix64 seeded at 0 (state advanced by the golden gamma before mixing):
    # first outputs published with the algorithm's reference implementation.
    assert synth.hash64(0, 0) == 0xE220A8397B1DCDAF
    assert synth.hash64(0, 1) == 0x6E789E6AA1B965F4
    assert synth.hash64(0, 2) == 0x06C45D188009454F


def test_normal_moments():
    w = synth.custom("m", 1, [(1 << 20,)], sigma=1e-3)
    x = bf16_to_f32(w.host_grad(0, 0)).astype(np.float64)
    assert abs(x.mean()) < 1e-5
    assert abs(x.std() / 1e-3 - 1) < 0.01
    # Irwin-Hall(4) is bounded by sqrt(12) sigma and has excess kurtosis -0.3
    assert np.abs(x).max() <= 1e-3 * np.sqrt(12) * 1.01
    k = ((x - x.mean()) ** 4).mean() / x.var() ** 2 - 3
    assert -0.4 < k < -0.2


def test_outlier_fraction():
    w = synth.llama70b()
    x = bf16_to_f32(w.host_grad_at(0, 0, np.arange(1 << 20))).astype(np.float64)
    frac = np.mean(np.abs(x) > 1e-3 * np.sqrt(12) * 1.01)
    # 1% of elements are x100; the few that land near 0 stay below the bound
    assert 0.008 < frac < 0.0105


def test_zero_expert_fraction():
    w = synth.moe()
    zeros = [w.zero_grad(k, g[0]) for k in range(w.num_ranks) for g in w.zero_groups]
    assert 0.25 < np.mean(zeros) < 0.35
    # gate, up and down of one expert on one rank go together
    for k in range(4):
        for g in w.zero_groups[:16]:
            assert len({w.zero_grad(k, p) for p in g}) == 1
    assert not w.zero_grad(0, 0)  # attention weights are always routed
    g = w.zero_groups[0]
    k = next(k for k in range(w.num_ranks) if w.zero_grad(k, g[0]))
    assert not np.any(w.host_grad(k, g[0]))


@pytest.mark.parametrize("n", [16, 32, 64])
def test_sweep_shapes(n):
    w = synth.sweep(n)
    rows = sum(-(-s[0] // n) for s in w.shapes)
    assert rows == 2048  # per-rank fp32 shard = 2048 * 4096 = 2^23 elements
    for s in w.shapes[:-1]:
        assert 512 <= s[0] <= 16384 and s[0] % n != 0 and s[1] == 4096
    assert w.shapes[-1][0] % n == n - 1


def test_workload_sizes():
    assert synth.tiny().psi == 803066
    assert synth.llama8b().psi == 218112000
    assert synth.llama70b().psi == 855654400
    m = synth.moe()
    assert m.num_params == 391 and m.psi == 623120384
    assert synth.llama70b().rs_bytes() == 2 * 8 * 855654400 + 4 * 855654400


def test_host_fill_matches_gather():
    w = synth.tiny()
    full = w.host_grad(2, 7)
    idx = np.array([0, 17, 249])
    assert np.array_equal(w.host_grad_at(2, 7, idx), full[idx])


def test_device_generator_library_exports():
    import ctypes

    lib = ctypes.CDLL(synth.DEVICE_LIB)
    assert hasattr(lib, "synth_fill_bf16_device") and hasattr(lib, "synth_set_u16_device")
