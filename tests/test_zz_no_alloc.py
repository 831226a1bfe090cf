"""The allocation-free convolution entry point, checked against the oracle and
against the planned entry point.

conv2d_nchw_run_noalloc serves callers that cannot allocate device memory: code
running where cudaMalloc is forbidden, or inside a memory budget that someone
else fixed.  Such callers cannot create a plan, because a plan owns cudaMalloc'd
scratch, so the call keeps its scratch in a fixed array inside the library.
These tests call it through the C ABI twice in a row -- different shapes and
inputs, so stale scratch from the first call would show in the second -- and
compare each output element with the exact convolution from the CPU oracle
within tau * S (S = sum |a*w|), and with conv2d_nchw_run on the same inputs
within 2 * tau * S (each of the two is within tau * S of the exact result).
The file is collected last on purpose: a run that stops at the first failure
has then run every other test.
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
ORACLE_EPI = {"bias": oracle.EPI_BIAS, "bias_exp": oracle.EPI_BIAS_EXP,
              "bias_rsqrt": oracle.EPI_BIAS_RSQRT, "bias_recip": oracle.EPI_BIAS_RECIP,
              "bias_relu": oracle.EPI_BIAS_RELU}

CASES = [
    # fp32 (tf32 MMAs), N=1: few tiles, so the K dimension is split (partial sums in scratch)
    synth.RESNET_LAST[0],
    # fp16 3x3 with the fused exp epilogue, several tiles, no split
    synth.ConvSpec("noalloc_f16_exp", 2, 64, 96, 15, 13, 3, 1, 1, 1, "f16", "f32", "uniform", "he",
                   "bias_exp"),
    # bf16, stride 2, ragged channels, add + ReLU
    synth.ConvSpec("noalloc_bf16_s2", 3, 40, 72, 17, 17, 3, 2, 1, 1, "bf16", "bf16", "uniform", "he",
                   "bias_relu"),
    # N=1, one tile and 36 K blocks: split K, then 1/(acc + bias) and fp16 rounding in the
    # reduction pass (non-negative operands keep the argument away from zero)
    synth.ConvSpec("noalloc_f16_split_recip", 1, 256, 128, 8, 8, 3, 1, 1, 1, "f16", "f16",
                   "absnormal", "absnormal", "bias_recip"),
    # split K with exp(acc + bias) rounded to bf16 in the reduction pass
    synth.ConvSpec("noalloc_bf16_split_exp", 1, 192, 64, 7, 9, 3, 1, 1, 1, "bf16", "bf16",
                   "uniform", "he", "bias_exp"),
    # fp32 with an 11.8 MB kernel copy: the split the SM count asks for (60 slices of partial
    # sums) does not fit beside it in the 16 MiB array, so the call takes fewer slices
    synth.ConvSpec("noalloc_f32_split_lowered", 1, 640, 512, 7, 7, 3, 1, 1, 1, "f32", "f32",
                   "uniform", "he"),
]


def _inputs(spec, seed):
    x, w, b = synth.conv_inputs(spec, seed)
    return x, w, b, x.cuda(), w.cuda(), (b.cuda() if b is not None else None)


def _out_shape(spec):
    return (spec.N, spec.CO, bg.out_size(spec.H, spec.K, spec.stride, spec.pad),
            bg.out_size(spec.W, spec.K, spec.stride, spec.pad))


def _noalloc(spec, xd, wd, bd, flag):
    out = torch.full(_out_shape(spec), float("nan"), dtype=synth.TORCH_DTYPES[spec.out_dtype],
                     device="cuda")
    bg.conv2d_nchw_run_noalloc(spec.N, spec.H, spec.W, spec.CO, spec.CI, spec.K, spec.K,
                               spec.stride, spec.pad, DT[spec.in_dtype], DT[spec.out_dtype],
                               bg.EPI_NAMES[spec.epi], xd, wd, bd, 1e-5, out, flag)
    return out


def _planned(spec, xd, wd, bd):
    out = torch.full(_out_shape(spec), float("nan"), dtype=synth.TORCH_DTYPES[spec.out_dtype],
                     device="cuda")
    plan = bg.conv2d_nchw_plan(spec.N, spec.H, spec.W, spec.CO, spec.CI, spec.K, spec.K,
                               spec.stride, spec.pad, 1, DT[spec.in_dtype], DT[spec.out_dtype],
                               bg.EPI_NAMES[spec.epi], 0)
    bg.conv2d_nchw_run(plan, xd, wd, bd, 1e-5, out)
    torch.cuda.synchronize()
    plan.close()
    return out


def _oracle(spec, x, w, b, scale):
    """The exact result and the per-element bound at scale * tau."""
    tau = scale * (TAU["tf32"] if spec.in_dtype == "f32" else TAU["half"])
    if spec.epi == "none":
        ref, sabs = oracle.conv2d_nchw(x, w, stride=spec.stride, pad=spec.pad, nthreads=8)
        return ref, conv_bound(ref, sabs, tau, spec.out_dtype)
    ref, sabs = oracle.conv2d_nchw(x, w, stride=spec.stride, pad=spec.pad, bias=b,
                                   epi=ORACLE_EPI[spec.epi], nthreads=8)
    pre, _ = oracle.conv2d_nchw(x, w, stride=spec.stride, pad=spec.pad, nthreads=8)
    arg = pre + b.double().numpy().reshape(1, -1, 1, 1)
    return ref, epi_bound(arg, sabs, tau, spec.epi, spec.out_dtype, ref)


def _check_call(spec, seed):
    x, w, b, xd, wd, bd = _inputs(spec, seed)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    free = _noalloc(spec, xd, wd, bd, flag)
    torch.cuda.synchronize()
    assert flag.item() == 0, "a device wait timed out"
    got = free.cpu().double().numpy()
    assert not np.isnan(got).any(), f"{spec.name}: unwritten outputs"
    ref, bound = _oracle(spec, x, w, b, 1.0)
    assert_within(got, ref, bound, f"noalloc vs oracle {spec.name}")
    planned = _planned(spec, xd, wd, bd).cpu().double().numpy()
    _, bound2 = _oracle(spec, x, w, b, 2.0)
    assert_within(got, planned, bound2, f"noalloc vs planned {spec.name}")


@pytest.mark.parametrize("first,second", [(0, 1), (1, 2), (2, 0), (3, 4), (4, 5), (5, 3)])
def test_noalloc_matches_oracle_and_planned_run_on_two_calls_in_a_row(first, second):
    _check_call(CASES[first], 10 + first)
    _check_call(CASES[second], 20 + second)


def test_noalloc_without_a_flag_reports_through_the_sticky_word():
    """With timeout_flag NULL the kernels raise the library's sticky flag, which
    the call never clears: a timeout recorded before it stays visible after it."""
    spec = CASES[2]
    _, _, _, xd, wd, bd = _inputs(spec, 5)
    bg.bigemm_clear_device_error()
    bg.bigemm_debug_wait_timeout(20_000)          # a bounded wait that runs out: flag set
    torch.cuda.synchronize()
    _noalloc(spec, xd, wd, bd, None)
    assert bg.bigemm_last_device_error() == 4     # still reported after the no-alloc call
    bg.bigemm_clear_device_error()
    out = _noalloc(spec, xd, wd, bd, None)
    assert bg.bigemm_last_device_error() == 0
    assert not torch.isnan(out.float()).any()


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
