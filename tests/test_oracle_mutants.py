"""Plant one plausible mistake at a time in a copy of the CPU oracle and check
that at least one pin in oracle_pins fails for it.  Each mutant is compiled
with gcc into a temporary directory and exercised in a child process, so a
mutant can never affect the real oracle or this test process."""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "tide_oracle.c")

MUTANTS = {
    "dropped_last_rank": ("k < num_ranks; ++k) acc = acc +", "k < num_ranks - 1; ++k) acc = acc +"),
    "wrong_sign": ("acc = acc + bf16_to_f32", "acc = acc - bf16_to_f32"),
    "reversed_rank_order": ("for (int32_t k = 0; k < num_ranks; ++k) acc = acc +",
                            "for (int32_t k = num_ranks - 1; k >= 0; --k) acc = acc +"),
    "scale_dropped": ("return acc * scale;", "return acc;"),
    "acc_starts_neg_zero": ("float acc = 0.0f;", "float acc = -0.0f;"),
    "flush_subnormal_results": ("return acc * scale;",
                                "return (acc * scale > -1.17549435e-38f && acc * scale < 1.17549435e-38f) "
                                "? 0.0f : acc * scale;"),
    "floor_chunk": ("return (d0 + num_ranks - 1) / num_ranks;",
                    "return d0 > 0 && d0 < num_ranks ? 1 : d0 / num_ranks;"),
    "row_off_by_one": ("const int64_t i = (int64_t)r * c + ii; /* row of the full tensor */",
                       "const int64_t i = (int64_t)r * c + ii + (ii + 1 < c ? 1 : 0);"),
    "transposed_rank_param": ("grads[(int64_t)k * num_params + p]",
                              "grads[(int64_t)p * num_ranks + k]"),
    "nonzero_padding": ("out[ii * inner[p] + j] = 0.0f;", "out[ii * inner[p] + j] = -0.0f;"),
    "offset_dropped": ("return r * block_numel + offset +", "return r * block_numel +"),
    "bf16_truncation": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0u;"),
    "bf16_ties_away": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    "nan_to_inf": ("return (uint16_t)((u >> 16) | 0x0040u); /* NaN */", "return (uint16_t)(u >> 16); /* NaN */"),
    "pack_wrong_block": ("gathered[(int64_t)r * block_numel + offsets[p] + e]",
                         "gathered[(int64_t)r * block_numel + offsets[p] + e - (e > 0 ? 1 : 0)]"),
    "rank_rs_wrong_row": ("const int64_t i = (int64_t)r * c + ii;\n      for (int64_t j = 0; j < inner[p]; ++j) {\n        if (i < d0[p]) {\n          for (int32_t k = 0; k < num_ranks; ++k)\n            vals[k] = grads[(int64_t)k * num_params + p][i * inner[p] + j];\n          shards_r",
                          "const int64_t i = (int64_t)r * c + ii + (ii + 1 < c ? 1 : 0);\n      for (int64_t j = 0; j < inner[p]; ++j) {\n        if (i < d0[p]) {\n          for (int32_t k = 0; k < num_ranks; ++k)\n            vals[k] = grads[(int64_t)k * num_params + p][i * inner[p] + j];\n          shards_r"),
    "stage_wrong_source_row": ("slot[(int64_t)r * block_numel + offsets[p] + e] = grads_k[p][(int64_t)r * c * inner[p] + e];",
                               "slot[(int64_t)r * block_numel + offsets[p] + e] = grads_k[p][(int64_t)r * n + e];"),
    "staged_rs_reads_padding": ("        if (e < n) {\n          for (int32_t k = 0; k < num_ranks; ++k)\n            vals[k] = slots[k]",
                                "        if (e < c * inner[p]) {\n          for (int32_t k = 0; k < num_ranks; ++k)\n            vals[k] = slots[k]"),
    "unaligned_offsets": ("o = roundup(o + oracle_chunk_rows(d0[p], num_ranks) * inner[p], align);",
                          "o = o + oracle_chunk_rows(d0[p], num_ranks) * inner[p];"),
}

CHILD = textwrap.dedent("""
    import sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import oracle
    oracle.LIB_PATH = {lib!r}
    import oracle_pins
    failed = []
    for chk in oracle_pins.ALL_CHECKS:
        try:
            chk()
        except Exception as e:  # a planted mistake may also raise elsewhere
            failed.append(chk.__name__)
    print("FAILED:" + ",".join(failed))
""")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mdir = tmp_path / "oracle_mutant"
    mdir.mkdir()
    (mdir / "tide_oracle.c").write_text(src.replace(old, new, 1))  # first occurrence
    (mdir / "tide_oracle.h").write_text(open(os.path.join(ROOT, "oracle", "tide_oracle.h")).read())
    lib = str(mdir / "liboracle_mutant.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    str(mdir / "tide_oracle.c"), "-o", lib], check=True)
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    line = [ln for ln in res.stdout.splitlines() if ln.startswith("FAILED:")]
    # a crash of the child also counts as caught, but say so
    caught = (line and line[0] != "FAILED:") or res.returncode != 0
    assert caught, f"mutant {name} passed every pin:\n{res.stdout}\n{res.stderr}"
