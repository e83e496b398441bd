"""The persistent launcher's host-side scheduling and layout, checked on the host (CPU only).

Two small programs compile the scheduling sources as they are and check their properties;
only host functions run, no GPU is needed:

* `tests/host/persist_host_check.cu` -- the kernel's shared-memory layout for every instance,
  ring depth, vectors per pass and activation length up to 65,536 (alignment of every region,
  no overlap, the configuration picked within the 227 KB budget whenever one fits), and the
  stage partition over 35,100 random stages on grids of 1 to 160 CTAs: every unit owned
  exactly once, non-empty ranges, the barrier flag on each CTA's first item of a stage, one
  unit set per CTA between barriers, the byte share without barriers, and CTA 0 without units
  in chained stages;
* `tests/host/quant_jobs_check.cu` -- the first phase's job placement: whole rounds of the
  grid, every vector once as a one-vector job, the longest-processing-time bound, and on the
  8B-shaped batch-1 step at 152 CTAs one wide vector or at most two narrow ones per CTA.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "packed_weight_gemv_gb300", "_lib")


@pytest.mark.parametrize("name,min_cases", [("persist_host_check", 40000), ("quant_jobs_check", 2000)])
def test_host_scheduling_properties(name, min_cases, tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    if not os.path.exists(os.path.join(LIBDIR, "libnt.so")):
        pytest.skip("libnt.so not built")
    exe = str(tmp_path / name)
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "--expt-relaxed-constexpr",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "packed_weight_gemv_gb300", "csrc"),
           os.path.join(ROOT, "tests", "host", name + ".cu"), "-o", exe,
           "-Xlinker", "-rpath", "-Xlinker", LIBDIR, "-L", LIBDIR, "-lnt"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok "), r.stdout + r.stderr
    assert int(r.stdout.split()[1]) >= min_cases
