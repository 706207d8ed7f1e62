"""The C ABI from plain C: the header compiles as C99 and C++17, and a C
program (tests/c_driver) links libtide.so, the CUDA runtime and the oracle,
runs both operations and checks them bit for bit (GPU part)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")
CUDA_INC = "/usr/local/cuda/include"
CUDA_LIB = "/usr/local/cuda/lib64"
SRC = os.path.join(ROOT, "tests", "c_driver", "tide_c_driver.c")
RESET_SRC = os.path.join(ROOT, "tests", "c_driver", "noalloc_reset.c")


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_header_compiles(lang, tmp_path):
    src = tmp_path / ("t.c" if lang == "c" else "t.cpp")
    src.write_text('#include "tide.h"\nint main(void) { tide_layout_t l = 0; (void)l; return 0; }\n')
    cc = "gcc" if lang == "c" else "g++"
    std = "-std=c99" if lang == "c" else "-std=c++17"
    subprocess.run([cc, std, "-Wall", "-Werror", "-I", INC, "-I", CUDA_INC, "-c", str(src), "-o",
                    str(tmp_path / "t.o")], check=True)


def build_driver(out):
    lib_dirs = [os.path.join(ROOT, "layout_aware_collectives_gb300"), os.path.join(ROOT, "oracle"), CUDA_LIB]
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-I", INC, "-I", CUDA_INC, SRC, "-o", str(out)]
    for d in lib_dirs:
        cmd += ["-L", d, "-Wl,-rpath," + d]
    cmd += ["-ltide", "-l:liboracle.so", "-lcudart"]
    subprocess.run(cmd, check=True)


def build_reset_driver(out):
    """The no-allocation entry point across a device reset (needs only
    libtide and the CUDA runtime)."""
    d = os.path.join(ROOT, "layout_aware_collectives_gb300")
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-I", INC, "-I", CUDA_INC, RESET_SRC, "-o", str(out),
                    "-L", d, "-Wl,-rpath," + d, "-L", CUDA_LIB, "-Wl,-rpath," + CUDA_LIB, "-ltide", "-lcudart"],
                   check=True)


def test_driver_builds(tmp_path):
    if not shutil.which("gcc"):
        pytest.skip("no C compiler")
    build_driver(tmp_path / "driver")
    build_reset_driver(tmp_path / "reset_driver")


@pytest.mark.gpu
def test_driver_runs_bit_exact(tmp_path):
    exe = tmp_path / "driver"
    build_driver(exe)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert res.stdout.startswith("ok:")
