"""The GPU tests' CUDA probes (tests/csrc/*.cu) compile against the library's
current headers.  They are built only by the GPU tests that run them, so a
header change that breaks one would otherwise show up on a GPU machine alone.
Compile-only (nvcc cross-compiles for sm_103a without a GPU)."""
import glob
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PROBES = sorted(glob.glob(os.path.join(HERE, "csrc", "*.cu")))


@pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not installed")
@pytest.mark.parametrize("src", PROBES, ids=[os.path.basename(p) for p in PROBES])
def test_probe_compiles(src, tmp_path):
    out = tmp_path / (os.path.basename(src) + ".o")
    r = subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                        "-std=c++17", "-Xcompiler", "-fPIC", "-c",
                        "-I", os.path.join(ROOT, "gated_deltanet_linear_chunk_gb300", "csrc"),
                        "-I", os.path.join(ROOT, "include"), src, "-o", str(out)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]


def test_probes_found():
    assert len(PROBES) >= 2, PROBES
