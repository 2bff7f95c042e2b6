"""The register FFT codelets of the CUDA library, compiled as host code and
checked on the CPU against a brute-force DFT (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def output(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("codelets") / "check")
    src = os.path.join(ROOT, "tests", "host", "codelets_check.cu")
    inc = os.path.join(ROOT, "fft_gemm_ifft_gb300", "csrc")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-I", inc, src, "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return [ln.split() for ln in out.strip().splitlines()]


def test_codelets_match_brute_force(output):
    assert len(output) == 19
    for name, err, scale in output:
        # float32 arithmetic: a few ulps of the largest bin per stage
        assert float(err) <= 4e-6 * max(1.0, float(scale)), (name, err, scale)


def test_constexpr_twiddles_are_double_accurate(output):
    tw = [r for r in output if r[0] == "twiddles"][0]
    assert float(tw[1]) < 1e-14


def test_gelu_erf_within_its_published_bound():
    # erf by Abramowitz & Stegun 7.1.26 (|error| <= 1.5e-7): the GELU error is at
    # most |v|/2 of that plus float rounding, far inside the float32 tolerance
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    import tempfile
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "gelu")
        src = os.path.join(ROOT, "tests", "host", "gelu_check.cu")
        inc = os.path.join(ROOT, "fft_gemm_ifft_gb300", "csrc")
        subprocess.run([nvcc, "-std=c++17", "-O2", "-I", inc, src, "-o", exe], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split()
    worst, worst_rel, n = float(out[0]), float(out[1]), int(out[2])
    assert n > 2000000
    assert worst_rel <= 2.5e-7, (worst, worst_rel)
