"""Host-side pieces of the benchmark (no GPU): the HBM-mix probe library
exports its entry points, the read:write ratio follows the reduce-scatter's
2N bytes read per 4 written, and the per-mode interference summary stays
short enough to sit at the end of the one JSON line."""
import ctypes
import json
import os

import bench


def test_hbm_probe_library_exports_its_entry_points():
    lib = ctypes.CDLL(bench.HBM_LIB)
    for name in ("hbm_read", "hbm_write", "hbm_mix", "hbm_sm_stream"):
        assert hasattr(lib, name), name


def test_mix_ratio_follows_the_reduce_scatter():
    # 2N bf16 bytes read per 4 fp32 bytes written
    assert [bench.mix_ratio(n) for n in (1, 2, 4, 8, 16, 32, 64)] == [1, 1, 2, 4, 8, 16, 16]


def test_interference_summary_is_compact():
    modes = []
    names = (["uncapped", "uncapped_lowprio"] + [f"capped{c}" for c in (8, 16, 32, 64)]
             + [f"bulk_tma_capped{c}" for c in (8, 16, 32, 64)] + ["bulk_tma_uncapped", "bulk_tma_uncapped_lowprio"])
    for name in names:
        modes.append({"op": "rs", "mode": name, "grid": 52240, "gemm_slowdown_pct": 266.25,
                      "gemm_slowdown_pct_range": [261.12, 270.31], "gemm_slowdown_cycles_pct": 259.91,
                      "op_GB/s_during_gemm": 4268.3,
                      "clocks": {"sm_mhz_concurrent": 2062.0, "sm_mhz_alone": 1980.0, "samples": 31,
                                 "reasons": ["sw_power_cap"]}})
    for name in ("uncapped", "uncapped_lowprio", "bulk_tma", "bulk_tma_lowprio", "capped16", "copy_engine"):
        modes.append(dict(modes[0], op="ag", mode=name))
    s = bench.interference_summary({"gemm_ms_alone": 0.55, "modes": modes})
    assert len(s["rows"]) == len(names) + 2  # every RS mode, two placement modes
    assert len(json.dumps(s)) < 2000
    assert all(r[-1] == "pcap" for r in s["rows"])


def test_bench_hbm_source_sits_beside_the_bench():
    assert os.path.exists(os.path.join(bench.ROOT, "bench_hbm.cu"))
