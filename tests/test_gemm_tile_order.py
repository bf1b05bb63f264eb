"""The GEMM's tile order, checked on the host: the device function that maps
a CTA pair's round-robin index to its output tile is compiled into a host
program (tests/gemm_tile_order_check.cu) and run over ~700k shapes.  It must
be a bijection onto the tiles, keep each round's tiles those of row order
when it balances half-width tiles, and never load a pair more than row order
does.  Needs nvcc (no GPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="needs nvcc")
def test_tile_order_is_a_balanced_bijection(tmp_path):
    exe = str(tmp_path / "tile_order_check")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "nvfp4_int8_mixed_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "gemm_tile_order_check.cu"), "-o", exe],
                   check=True, capture_output=True, timeout=600)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok:"), r.stdout
