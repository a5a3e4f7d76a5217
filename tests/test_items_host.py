"""The prefill kernel's work decomposition checked on the host (no GPU): tests/host_items_check.cu
includes the kernel's own item and range functions (csrc/fa_items.cuh), walks every CTA's item
list for some fifteen thousand problem shapes (dense with Nq != Nk, per-sequence lengths, packed
sequences; causal, windows, grouped heads; persistent and one-CTA-per-item grids) and checks that
every output row belongs to exactly one Q tile, that the softmax warps and the MMA issuer make the
same number of P handoffs (the count the named-barrier handoff relies on), and that a tile the
kernel leaves unmasked holds only keys each of its rows may see."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_work_decomposition_on_host(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "items_check")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(ROOT, "flashattention_forward_fa_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "host_items_check.cu"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and out.stdout.strip().startswith("ok"), out.stdout[-2000:]
