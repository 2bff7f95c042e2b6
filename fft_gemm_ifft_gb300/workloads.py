"""Synthetic workloads and seeded input generators.

This module is shared by the tests, the benchmark and the smoke check, on both
sides of the parity comparison (the CUDA library and the float64 oracle).  It
holds no transform, mixing or activation arithmetic: only shapes, random draws
(``torch.Generator`` on the CPU, drawn in float64 then rounded once to the
storage dtype) and the coordinate channels of the FNO input.

The five workloads are the synthetic stand-ins for the application tasks of the
TurboFNO article (gsyq.cn/news/457482, §5.1: CFD, weather, EM, materials and
finance fields on 128x128 grids; §1: a 64^3 three-dimensional flow field).
Those data sets are not available, so each workload draws N(0,1) fields of the
same spatial scale:

=========  ====  =====================================================  =====
name       dim   shape                                                  dtype
=========  ====  =====================================================  =====
1d_f32     1     B=4, C=16, N=256, modes 16                             f32
2d_f32     2     B=8, C=32, 128x128, modes 16x16 (2 blocks)             f32
2d_f16     2     B=32, C=64, 256x256, modes 32x32 (2 blocks)            f16
2d_bf16    2     the 2d_f16 problem with bfloat16 storage               bf16
3d_f32     3     B=4, C=32, 64^3, modes 16^3 (4 blocks)                 f32
fno2d_f32  2     B=16, 3 -> 64 -> 4 layers -> 128 -> 1, 128x128, 16x16  f32
=========  ====  =====================================================  =====

Seeds: the input field of workload ``c`` (index 0..4 in the table) uses seed
1000+c, its spectral weights seed 2000+c and (FNO only) its 1x1 linear weights
seed 3000+c.  Spectral weights draw re and im from U[0,1) and scale them by
1/(Cin*Cout); 1x1 linear weights are Kaiming-uniform U(-sqrt(6/fan_in),
+sqrt(6/fan_in)) with biases U(-1/sqrt(fan_in), +1/sqrt(fan_in)).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class SpectralConvCase:
    """One spectral-convolution problem."""
    name: str
    n: Tuple[int, ...]          # spatial extents N_0..N_{d-1}
    modes: Tuple[int, ...]      # m_a per axis (per block on full axes)
    batch: int
    cin: int
    cout: int
    dtype: str                  # "f32", "f16" or "bf16" (storage; accumulation is fp32)
    index: int = 0              # workload index used for the seeds

    @property
    def ndim(self) -> int:
        return len(self.n)

    @property
    def nblk(self) -> int:
        return 2 ** (self.ndim - 1)

    @property
    def weight_shape(self) -> Tuple[int, ...]:
        return (self.nblk, self.cin, self.cout) + tuple(self.modes)

    @property
    def x_shape(self) -> Tuple[int, ...]:
        return (self.batch, self.cin) + tuple(self.n)

    @property
    def y_shape(self) -> Tuple[int, ...]:
        return (self.batch, self.cout) + tuple(self.n)

    @property
    def np_dtype(self):
        """Host array dtype: bfloat16 values are held exactly in float32."""
        return np.float16 if self.dtype == "f16" else np.float32

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def algorithmic_bytes(self) -> int:
        """Read x once, read the weights once, write y once."""
        nx = math.prod(self.x_shape)
        ny = math.prod(self.y_shape)
        nw = math.prod(self.weight_shape) * 2
        return (nx + ny + nw) * self.elem_bytes

    def with_batch(self, batch: int) -> "SpectralConvCase":
        return dataclasses.replace(self, batch=batch)


@dataclasses.dataclass(frozen=True)
class FnoCase:
    """The 2-D FNO forward stack."""
    name: str
    batch: int = 16
    cin_lift: int = 3
    width: int = 64
    nlayers: int = 4
    h: int = 128
    w: int = 128
    modes: Tuple[int, int] = (16, 16)
    hidden: int = 128
    cout: int = 1
    index: int = 4

    @property
    def spectral(self) -> SpectralConvCase:
        return SpectralConvCase(self.name + "/spectral", (self.h, self.w), self.modes,
                                self.batch, self.width, self.width, "f32", self.index)

    def algorithmic_bytes(self) -> int:
        """Float32 bytes of the least traffic a forward of the stack can have
        with two passes per layer: each layer reads its input twice (for the
        forward transform, then for the pointwise term beside the inverse) and
        writes its output once; the lift is recomputed from the 3-channel x
        where the first layer reads, the head is taken where the last layer
        writes (so only the 1-channel output is stored); every parameter is
        read once."""
        pix = self.batch * self.h * self.w
        act = pix * self.width * 4
        total = 0
        for l in range(self.nlayers):
            reads = pix * self.cin_lift * 4 if l == 0 else act
            writes = pix * self.cout * 4 if l == self.nlayers - 1 else act
            total += 2 * reads + writes
        nblk = 2
        spec = self.nlayers * nblk * self.width * self.width * math.prod(self.modes) * 8
        lin = (self.width * (self.cin_lift + 1)
               + self.nlayers * self.width * (self.width + 1)
               + self.hidden * (self.width + 1) + self.cout * (self.hidden + 1)) * 4
        return total + spec + lin


CASES: Dict[str, SpectralConvCase] = {
    "1d_f32": SpectralConvCase("1d_f32", (256,), (16,), 4, 16, 16, "f32", 0),
    "2d_f32": SpectralConvCase("2d_f32", (128, 128), (16, 16), 8, 32, 32, "f32", 1),
    "2d_f16": SpectralConvCase("2d_f16", (256, 256), (32, 32), 32, 64, 64, "f16", 2),
    "2d_bf16": SpectralConvCase("2d_bf16", (256, 256), (32, 32), 32, 64, 64, "bf16", 2),
    "3d_f32": SpectralConvCase("3d_f32", (64, 64, 64), (16, 16, 16), 4, 32, 32, "f32", 3),
}
FNO_CASE = FnoCase("fno2d_f32")


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def to_storage(a, dtype: str) -> np.ndarray:
    """Round values once to the storage dtype (a cast, no arithmetic).  The
    host array is float32 for f32 and bf16 (bfloat16 values are exact in
    float32) and float16 for f16."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(torch.bfloat16)
        return t.to(torch.float32).numpy()
    return np.asarray(a).astype(np.float16 if dtype == "f16" else np.float32)


def to_torch_storage(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Host storage array -> CPU tensor of the storage dtype."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(TORCH_DTYPES[dtype])


def make_x(case: SpectralConvCase, seed: int | None = None) -> np.ndarray:
    """N(0,1) input in the storage dtype, shape (B, Cin, N...)."""
    g = _gen(1000 + case.index if seed is None else seed)
    x = torch.randn(case.x_shape, generator=g, dtype=torch.float64)
    return to_storage(x.numpy(), case.dtype)


def make_w(case: SpectralConvCase, seed: int | None = None) -> np.ndarray:
    """Complex weights as interleaved (re, im) in the storage dtype,
    shape (nblk, Cin, Cout, m..., 2); re and im ~ U[0,1) / (Cin*Cout)."""
    g = _gen(2000 + case.index if seed is None else seed)
    w = torch.rand(case.weight_shape + (2,), generator=g, dtype=torch.float64)
    w = w / float(case.cin * case.cout)
    return to_storage(w.numpy(), case.dtype)


def as_complex(w: np.ndarray) -> np.ndarray:
    """Interleaved (..., 2) storage -> complex128 (upcast, no arithmetic)."""
    w = np.asarray(w, dtype=np.float64)
    return w[..., 0] + 1j * w[..., 1]


def make_fno_inputs(case: FnoCase = FNO_CASE, batch: int | None = None):
    """Input (B, 3, H, W) float32: channel 0 ~ N(0,1); channel 1 = linspace(0,1)
    along H; channel 2 = linspace(0,1) along W."""
    b = case.batch if batch is None else batch
    g = _gen(1000 + case.index)
    field = torch.randn((b, 1, case.h, case.w), generator=g, dtype=torch.float64)
    gx = torch.linspace(0.0, 1.0, case.h, dtype=torch.float64).view(1, 1, case.h, 1)
    gy = torch.linspace(0.0, 1.0, case.w, dtype=torch.float64).view(1, 1, 1, case.w)
    x = torch.cat([field, gx.expand(b, 1, case.h, case.w),
                   gy.expand(b, 1, case.h, case.w)], dim=1)
    assert case.cin_lift == 3
    return x.numpy().astype(np.float32)


def make_fno_params(case: FnoCase = FNO_CASE) -> Dict[str, np.ndarray]:
    """FNO parameters in float32 storage.  spec_w is interleaved complex,
    shape (L, 2, W, W, m0, m1, 2); linear weights are (out, in)."""
    gs = _gen(2000 + case.index)
    gl = _gen(3000 + case.index)

    def kaiming(shape, fan_in):
        bound = math.sqrt(6.0 / fan_in)
        return (torch.rand(shape, generator=gl, dtype=torch.float64) * 2 - 1) * bound

    def bias(shape, fan_in):
        bound = 1.0 / math.sqrt(fan_in)
        return (torch.rand(shape, generator=gl, dtype=torch.float64) * 2 - 1) * bound

    W, L = case.width, case.nlayers
    p = {
        "lift_w": kaiming((W, case.cin_lift), case.cin_lift),
        "lift_b": bias((W,), case.cin_lift),
    }
    spec, pw, pb = [], [], []
    for _ in range(L):
        spec.append(torch.rand((2, W, W) + tuple(case.modes) + (2,), generator=gs,
                               dtype=torch.float64) / float(W * W))
        pw.append(kaiming((W, W), W))
        pb.append(bias((W,), W))
    p["spec_w"] = torch.stack(spec)
    p["pw_w"] = torch.stack(pw)
    p["pw_b"] = torch.stack(pb)
    p["proj1_w"] = kaiming((case.hidden, W), W)
    p["proj1_b"] = bias((case.hidden,), W)
    p["proj2_w"] = kaiming((case.cout, case.hidden), case.hidden)
    p["proj2_b"] = bias((case.cout,), case.hidden)
    return {k: v.numpy().astype(np.float32) for k, v in p.items()}


def fno_params_for_oracle(p: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    """Upcast the stored parameters; spec_w becomes complex128."""
    q = {k: np.asarray(v, dtype=np.float64) for k, v in p.items()}
    q["spec_w"] = as_complex(p["spec_w"])
    return q


def small_case(n, modes, batch, cin, cout, dtype="f32", index=0, name="small"):
    return SpectralConvCase(name, tuple(n), tuple(modes), batch, cin, cout, dtype, index)
