"""CPU check of the SYRK unit schedule and the kernels' index guards.

`schedule_check.cu` is compiled with nvcc as host code. It calls the schedule functions the kernels
use (`csrc/schedule.cuh`) for several thousand flush shapes and checks four things:
- every unit lies inside the upper triangle and the flush;
- every (tile, k-block) is summed exactly once: slabs, the last wave split in halves, and pairs of
  SMs;
- the pair kernel stores every upper tile once and nothing below the diagonal;
- the tile layout is one to one.

It runs here, without a GPU. A planted mistake in a copy of the schedule must make it fail.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gptq_qqq_calibration_gb300", "csrc")
SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "schedule_check.cu")


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    pytest.skip("nvcc not found")


def _build_and_run(tmp_path, csrc_dir):
    exe = str(tmp_path / "schedule_check")
    cmd = [_nvcc(), "-std=c++17", "-O1", "-I", csrc_dir, "-I", os.path.join(ROOT, "include"), SRC, "-o", exe]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, timeout=300)
    assert r.returncode == 0, r.stdout.decode(errors="replace")
    return subprocess.run([exe], stdout=subprocess.PIPE, stderr=subprocess.STDOUT, timeout=300)


def test_schedule_covers_every_tile_and_k_block_once(tmp_path):
    r = _build_and_run(tmp_path, CSRC)
    out = r.stdout.decode(errors="replace")
    assert r.returncode == 0, out
    assert out.startswith("schedule ok"), out


@pytest.mark.parametrize("mistake", [
    # the second half of a split tile starting one k-block late
    ("const int mid = p.total_kb >> 1;\n            un.k0 = (v & 1) ? mid : 0;",
     "const int mid = p.total_kb >> 1;\n            un.k0 = (v & 1) ? mid + 1 : 0;"),
    # slabs rounded the wrong way at their ends
    ("un.k1 = static_cast<int>(static_cast<long long>(slab + 1) * p.total_kb / p.n_slabs);\n    }",
     "un.k1 = static_cast<int>(static_cast<long long>(slab + 1) * p.total_kb / p.n_slabs) - (slab & 1);\n    }"),
    # the pair kernel's odd CTA storing the tile below the diagonal
    ("return (rb < T && rb <= un.J) ? tile_index(rb, un.J, T) : -1;",
     "return (rb < T && rb <= un.J + 1) ? tile_index(rb < un.J ? rb : un.J, un.J, T) : -1;"),
])
def test_planted_schedule_mistakes_fail(tmp_path, mistake):
    old, new = mistake
    d = tmp_path / "csrc"
    shutil.copytree(CSRC, d)
    p = d / "schedule.cuh"
    s = p.read_text()
    assert s.count(old) == 1, old
    p.write_text(s.replace(old, new))
    r = _build_and_run(tmp_path, str(d))
    assert r.returncode != 0, r.stdout.decode(errors="replace")
