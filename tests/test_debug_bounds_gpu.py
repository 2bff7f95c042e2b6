"""The index-checking build (libfno_bounds.so, compiled with FNO_DEBUG_BOUNDS)
on the GPU: every checked global-memory index of the separate-kernels path,
the padded path and the 16-bit 256x256 fused path stays in range on small
cases (no FNO_ERR_DEVICE_BOUNDS), and the results still match the oracle.  The
checks run in a child process that loads the variant (FNO_LIBRARY=bounds), so
the rest of the suite keeps the normal library."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, numpy as np, torch
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import oracle
from fft_gemm_ifft_gb300 import SpectralConv, capi, workloads
from parity_util import assert_close, to_dev
assert capi.library_path().endswith("libfno_bounds.so"), capi.library_path()
cases = [
    # (n, modes, batch, cin, cout, dtype, flags, pad)
    ((12,), (7,), 2, 3, 4, "f32", capi.FNO_PLAN_UNFUSED, None),
    ((6, 10, 14), (2, 3, 4), 1, 2, 3, "f32", capi.FNO_PLAN_UNFUSED, None),
    ((24, 40), (5, 9), 2, 4, 3, "f16", capi.FNO_PLAN_UNFUSED, None),
    ((6, 10), (2, 6), 2, 3, 2, "f32", 0, (2, 6)),
    ((256, 256), (32, 32), 2, 64, 64, "f16", capi.FNO_PLAN_PACKED_WEIGHTS, None),
    ((256, 256), (32, 32), 3, 5, 7, "bf16", 0, None),
]
for n, modes, b, ci, co, dt, flags, pad in cases:
    L = tuple(a + p for a, p in zip(n, pad)) if pad else n
    case = workloads.small_case(n, modes, b, ci, co, dt, index=11)
    x = workloads.make_x(case, seed=71)
    w = workloads.make_w(workloads.small_case(L, modes, b, ci, co, dt), seed=72)
    conv = SpectralConv(n, modes, b, ci, co, dt, flags, pad=pad)
    W = to_dev(w, dt)
    if flags & capi.FNO_PLAN_PACKED_WEIGHTS:
        W = conv.pack_weights(W)
    y = conv(to_dev(x, dt), W)
    torch.cuda.synchronize()
    st = conv.device_error()
    assert st == capi.FNO_OK, (n, capi.fno_status_string(st))
    ref = (oracle.spectral_conv_padded(x.astype(np.float64), workloads.as_complex(w), modes, pad)
           if pad else oracle.spectral_conv(x.astype(np.float64), workloads.as_complex(w), modes))
    assert_close(y.float().cpu().numpy(), ref, dt, f"bounds build {n}")
    conv.close()
print("bounds build ok:", len(cases), "cases")
'''


def test_index_checked_build_runs_clean(fno, oracle_mod):
    from fft_gemm_ifft_gb300 import build
    build.build(debug_bounds=True)
    env = dict(os.environ, FNO_LIBRARY="bounds")
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHILD], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "bounds build ok" in r.stdout
