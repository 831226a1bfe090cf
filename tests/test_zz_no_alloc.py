"""The allocation-free convolution entry point, checked against the planned one.

conv2d_nchw_run_noalloc is for callers that cannot allocate device memory
(they cannot create a plan, which owns cudaMalloc'd scratch); it keeps its
scratch in a fixed array inside the library.  These tests call it through the
C ABI twice in a row -- different shapes and inputs, so stale scratch from the
first call would show in the second -- and compare each output with
conv2d_nchw_run on the same inputs.  Each of the two results is within
tau * S of the exact convolution (S = sum |a*w|, from the CPU oracle), so they
may differ by up to 2 * tau * S.  The file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import broadcast_implicit_gemm_gb300 as bg
import oracle
from broadcast_implicit_gemm_gb300 import synth
from tests.tolerance import TAU, assert_within, conv_bound, epi_bound

pytestmark = pytest.mark.gpu

DT = {"f32": bg.F32, "f16": bg.F16, "bf16": bg.BF16}

CASES = [
    # fp32 (tf32 MMAs), N=1: few tiles, so the K dimension is split (partial sums in scratch)
    synth.RESNET_LAST[0],
    # fp16 3x3 with the fused exp epilogue, several tiles, no split
    synth.ConvSpec("noalloc_f16_exp", 2, 64, 96, 15, 13, 3, 1, 1, 1, "f16", "f32", "uniform", "he",
                   "bias_exp"),
    # bf16, stride 2, ragged channels
    synth.ConvSpec("noalloc_bf16_s2", 3, 40, 72, 17, 17, 3, 2, 1, 1, "bf16", "bf16"),
]


def _outputs(spec, seed):
    x, w, b = synth.conv_inputs(spec, seed)
    xd, wd = x.cuda(), w.cuda()
    bd = b.cuda() if b is not None else None
    Ho = bg.out_size(spec.H, spec.K, spec.stride, spec.pad)
    Wo = bg.out_size(spec.W, spec.K, spec.stride, spec.pad)
    odt = synth.TORCH_DTYPES[spec.out_dtype]
    epi = bg.EPI_NAMES[spec.epi]
    planned = torch.full((spec.N, spec.CO, Ho, Wo), float("nan"), dtype=odt, device="cuda")
    plan = bg.conv2d_nchw_plan(spec.N, spec.H, spec.W, spec.CO, spec.CI, spec.K, spec.K,
                               spec.stride, spec.pad, 1, DT[spec.in_dtype], DT[spec.out_dtype],
                               epi, 0)
    bg.conv2d_nchw_run(plan, xd, wd, bd, 1e-5, planned)
    free = torch.full_like(planned, float("nan"))
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    bg.conv2d_nchw_run_noalloc(spec.N, spec.H, spec.W, spec.CO, spec.CI, spec.K, spec.K,
                               spec.stride, spec.pad, DT[spec.in_dtype], DT[spec.out_dtype], epi,
                               xd, wd, bd, 1e-5, free, flag)
    torch.cuda.synchronize()
    plan.close()
    assert flag.item() == 0, "a device wait timed out"
    return x, w, b, planned.cpu().double().numpy(), free.cpu().double().numpy()


def _bound(spec, x, w, b):
    tau = 2 * (TAU["tf32"] if spec.in_dtype == "f32" else TAU["half"])
    if spec.epi == "none":
        ref, sabs = oracle.conv2d_nchw(x, w, stride=spec.stride, pad=spec.pad, nthreads=8)
        return conv_bound(ref, sabs, tau, spec.out_dtype)
    ref, sabs = oracle.conv2d_nchw(x, w, stride=spec.stride, pad=spec.pad, bias=b,
                                   epi=oracle.EPI_BIAS_EXP, nthreads=8)
    pre, _ = oracle.conv2d_nchw(x, w, stride=spec.stride, pad=spec.pad, nthreads=8)
    arg = pre + b.double().numpy().reshape(1, -1, 1, 1)
    return epi_bound(arg, sabs, tau, spec.epi, spec.out_dtype, ref)


@pytest.mark.parametrize("first,second", [(0, 1), (1, 2), (2, 0)])
def test_noalloc_matches_planned_run_on_two_calls_in_a_row(first, second):
    for i, seed in ((first, 10 + first), (second, 20 + second)):
        spec = CASES[i]
        x, w, b, planned, free = _outputs(spec, seed)
        assert not np.isnan(free).any(), f"{spec.name}: unwritten outputs"
        assert_within(free, planned, _bound(spec, x, w, b), f"noalloc vs planned {spec.name}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # channels-last copy of the data alone is 256*64*56*56*2 bytes, far above 16 MiB
    x = torch.empty(16, dtype=torch.float16, device="cuda")
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_run_noalloc(256, 56, 56, 64, 64, 3, 3, 1, 1, bg.F16, bg.F16, bg.EPI_NONE,
                                   x, x, None, 1e-5, x)
    assert e.value.status == 2
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_run_noalloc(1, 8, 8, 64, 64, 3, 3, 1, 1, bg.F16, bg.F32, bg.EPI_BIAS_EXP,
                                   x, x, None, 1e-5, x)
    assert e.value.status == 1
