"""Host logic of the attention kernels' work order.  tests/c/order_check.cpp runs the kernels'
own order function (chunked_order from csrc/pg_internal.h, compiled for the host) over every item
index of many launches and checks that each (tile, head) pair comes out exactly once, chunk by
chunk of heads.  Needs no GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")


def test_work_order_is_a_bijection(tmp_path):
    if shutil.which("g++") is None or not os.path.isdir(CUDA_INC):
        pytest.skip("g++ or the CUDA headers not available")
    exe = str(tmp_path / "order_check")
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CUDA_INC,
                    "-I", os.path.join(ROOT, "shared_prefix_grouped_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "c", "order_check.cpp"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout
