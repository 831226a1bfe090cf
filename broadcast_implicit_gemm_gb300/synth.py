"""Seeded synthetic inputs for the conv and broadcast workloads.

This module only draws random numbers and names shapes; it holds none of the
method's arithmetic, so the CUDA path and the CPU oracle can both take their
inputs from it.  Every tensor is made on the host from a fixed seed with a
``torch.Generator`` and is then rounded once to the dtype the kernel reads.

Workloads (layer shapes only; no model weights or datasets are involved):
  * ``resnet_last``  -- N=1, CI=CO=512, 7x7, 3x3, stride 1, pad 1, fp32; the
    layer tuned in "Tuning High Performance Convolution on NVIDIA GPUs".
    data and kernel uniform[-1,1].
  * ``sweep_fp32``   -- five batch-1 fp32 layers; data uniform[-1,1], kernel
    N(0, 2/(CI*K*K)).
  * ``resnet50_fp16`` -- five ResNet-50 bottleneck layers at N=256, fp16 in and
    out; activations |N(0,1)|, kernels N(0, 2/fan_in).
  * ``bcast``        -- [128,256,32,32] fp32, var uniform[-2,2]; the fused conv
    (CI=CO=256, 32x32, 3x3 pad 1, N=32, fp16 in, fp32 out) with data
    uniform[-1,1], kernel N(0, 2/(CI*9)) and bias uniform[-1,1].
  * ``depthwise_fp16`` -- four depthwise layers at N=64, fp16; data
    uniform[-1,1], kernel N(0, 2/(K*K)).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class ConvSpec:
    name: str
    N: int
    CI: int
    CO: int
    H: int
    W: int
    K: int
    stride: int
    pad: int
    groups: int = 1
    in_dtype: str = "f32"          # "f32" | "f16" | "bf16"
    out_dtype: str = "f32"
    data_dist: str = "uniform"     # "uniform" [-1,1] | "absnormal" |N(0,1)|
    kernel_dist: str = "he"        # "uniform" [-1,1] | "he" N(0, 2/fan_in) | "dw" N(0, 2/(K*K))
    epi: str = "none"              # "none" | "bias" | "bias_exp" | "bias_rsqrt" | "bias_recip" | "bias_relu"

    def with_batch(self, N: int) -> "ConvSpec":
        return replace(self, N=N, name=f"{self.name}@N{N}")


def _s(name, CI, CO, HW, K, stride, pad, **kw):
    N = kw.pop("N", 1)
    return ConvSpec(name, N, CI, CO, HW, HW, K, stride, pad, **kw)


RESNET_LAST = [_s("resnet_last_512x512_7x7_k3", 512, 512, 7, 3, 1, 1,
                  data_dist="uniform", kernel_dist="uniform")]

SWEEP_FP32 = [
    _s("sweep_64x64_56_k3", 64, 64, 56, 3, 1, 1),
    _s("sweep_128x128_28_k3", 128, 128, 28, 3, 1, 1),
    _s("sweep_256x256_14_k3", 256, 256, 14, 3, 1, 1),
    _s("sweep_256x512_14_k3s2", 256, 512, 14, 3, 2, 1),
    _s("sweep_1024x256_14_k1", 1024, 256, 14, 1, 1, 0),
]

_R50 = dict(N=256, in_dtype="f16", out_dtype="f16", data_dist="absnormal", kernel_dist="he")
RESNET50_FP16 = [
    _s("r50_64x64_56_k1", 64, 64, 56, 1, 1, 0, **_R50),
    _s("r50_64x64_56_k3", 64, 64, 56, 3, 1, 1, **_R50),
    _s("r50_64x256_56_k1", 64, 256, 56, 1, 1, 0, **_R50),
    _s("r50_512x512_7_k3", 512, 512, 7, 3, 1, 1, **_R50),
    _s("r50_256x512_28_k1s2", 256, 512, 28, 1, 2, 0, **_R50),
]

FUSED_CONV = [_s("fused_256x256_32_k3_exp", 256, 256, 32, 3, 1, 1, N=32, in_dtype="f16",
                 out_dtype="f32", data_dist="uniform", kernel_dist="he", epi="bias_exp")]

_DW = dict(N=64, in_dtype="f16", out_dtype="f16", data_dist="uniform", kernel_dist="dw")
DEPTHWISE_FP16 = [
    _s("dw_32_112_k3", 32, 32, 112, 3, 1, 1, groups=32, **_DW),
    _s("dw_96_112_k3s2", 96, 96, 112, 3, 2, 1, groups=96, **_DW),
    _s("dw_144_56_k3", 144, 144, 56, 3, 1, 1, groups=144, **_DW),
    _s("dw_576_14_k5", 576, 576, 14, 5, 1, 2, groups=576, **_DW),
]

BCAST_SHAPE = (128, 256, 32, 32)   # N, C, H, W
# general [1,P,1] => [B0,P,B1] broadcasts, fp32 outputs larger than L2: short
# rows (7x7 and 4x4 planes), single-element rows ([N, C] from [C]), and a tiny
# preserved axis with long rows
BCAST_GENERAL = [(1024, 1024, 49), (512, 4096, 16), (32768, 1024, 1), (64, 16, 65536)]
BCAST_EPS = 1e-5

ALL_CONVS = RESNET_LAST + SWEEP_FP32 + RESNET50_FP16 + FUSED_CONV + DEPTHWISE_FP16

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _draw(shape, dist: str, g: torch.Generator, fan: int = 1, K: int = 1) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "absnormal":
        return torch.randn(shape, generator=g, dtype=torch.float32).abs()
    if dist == "he":
        return torch.randn(shape, generator=g, dtype=torch.float32) * (2.0 / fan) ** 0.5
    if dist == "dw":
        return torch.randn(shape, generator=g, dtype=torch.float32) * (2.0 / (K * K)) ** 0.5
    raise ValueError(dist)


def conv_inputs(spec: ConvSpec, seed: int = 0, dtype: str | None = None):
    """(data [N,CI,H,W], kernel [CO,CI/groups,K,K], bias [CO] fp32 or None), CPU tensors.
    data and kernel are rounded once to ``dtype`` (default: the spec's input dtype)."""
    dt = TORCH_DTYPES[dtype or spec.in_dtype]
    g = _gen(seed)
    data = _draw((spec.N, spec.CI, spec.H, spec.W), spec.data_dist, g)
    cig = spec.CI // spec.groups
    kern = _draw((spec.CO, cig, spec.K, spec.K), spec.kernel_dist, g,
                 fan=cig * spec.K * spec.K, K=spec.K)
    bias = None
    if spec.epi != "none":
        bias = torch.rand((spec.CO,), generator=g, dtype=torch.float32) * 2.0 - 1.0
    return data.to(dt).contiguous(), kern.to(dt).contiguous(), bias


def bcast_var(C: int, seed: int = 0) -> torch.Tensor:
    """var[C] uniform[-2,2], fp32."""
    g = _gen(seed)
    return (torch.rand((C,), generator=g, dtype=torch.float32) * 4.0 - 2.0).contiguous()


def random_flat_indices(total: int, count: int, seed: int = 0) -> torch.Tensor:
    """Distinct sample positions (int64) in [0, total)."""
    g = _gen(seed)
    count = min(count, total)
    if count == total:
        return torch.arange(total, dtype=torch.int64)
    idx = torch.randint(0, total, (count * 2,), generator=g, dtype=torch.int64)
    idx = torch.unique(idx)[:count]
    return idx
