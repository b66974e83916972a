"""The persistent decode's work split, checked on the host: tests/mega_split_check.cu compiles
the kernel header's split_of and warp cursors for the host (they are __host__ __device__) and
walks them for seven model shapes over ten grid sizes -- every (pair, slot) of a CTA visited
exactly once, slots on 256-column boundaries inside their rows, the CTAs' pair ranges a
partition, the split-pair scratch large enough wherever the shape is accepted.  These are the
index facts the weight stream's tensor copies depend on; no GPU is needed."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "layer_range_stage_gb300", "csrc")


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    pytest.skip("nvcc not found")


def test_split_covers_every_pair_and_slot_once(tmp_path):
    exe = str(tmp_path / "mega_split_check")
    subprocess.run([nvcc(), "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC, "-o", exe,
                    os.path.join(ROOT, "tests", "mega_split_check.cu")], check=True, capture_output=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout[-4000:]
    assert "0 failures" in out.stdout
