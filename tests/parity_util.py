"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and the float64 oracle on the same seeded inputs, then compare."""
import numpy as np
import torch

import oracle
from fft_gemm_ifft_gb300 import SpectralConv, workloads

# Bars from the specification of the layer: relative L2 error against the
# float64 oracle <= 1e-5 for float32 storage and arithmetic, <= 1e-2 for
# half storage with float32 accumulation.  The element-wise bound catches a
# few wrong elements that a norm over a large tensor would average away:
# float32 allows 1e-4 of the largest output magnitude; half storage allows
# 1e-2 of it (the output rounding alone is 2^-11 of each element).
REL_L2 = {"f32": 1e-5, "f16": 1e-2, "bf16": 1e-2}
ELEMWISE = {"f32": 1e-4, "f16": 1e-2, "bf16": 1e-2}


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_close(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    r = rel_l2(got, ref)
    assert r <= REL_L2[dtype], f"{what}: rel-L2 {r:.3e} > {REL_L2[dtype]}"
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    e = float(np.max(np.abs(got - ref))) / scale
    assert e <= ELEMWISE[dtype], f"{what}: max |err| / max |ref| = {e:.3e}"
    return r


def to_dev(a: np.ndarray, dtype: str = "") -> torch.Tensor:
    """Host array -> device tensor; dtype "bf16" casts the (exactly
    representable) float32 values to bfloat16 storage."""
    if dtype == "bf16":
        return workloads.to_torch_storage(a, dtype).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gpu(case, x_np, w_np, flags=0):
    conv = SpectralConv(case.n, case.modes, x_np.shape[0], case.cin, case.cout, case.dtype,
                        flags)
    y = conv(to_dev(x_np, case.dtype), to_dev(w_np, case.dtype))
    torch.cuda.synchronize()
    assert conv.device_error() == 0
    out = y.float().cpu().numpy()
    kernels = conv.kernel_count
    conv.close()
    return out, kernels


def run_oracle(case, x_np, w_np):
    return oracle.spectral_conv(x_np.astype(np.float64), workloads.as_complex(w_np), case.modes)
