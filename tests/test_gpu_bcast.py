"""GPU parity of the per-channel broadcast against the oracle (2 ulp of the
fp32-rounded fp64 value; NaN and inf where the oracle has them)."""
import numpy as np
import pytest
import torch

import broadcast_implicit_gemm_gb300 as bg
import oracle
from broadcast_implicit_gemm_gb300 import synth
from tests.tolerance import assert_within, ulp

pytestmark = pytest.mark.gpu

OPS = {"copy": bg.BC_COPY, "exp": bg.BC_EXP, "rsqrt": bg.BC_RSQRT, "recip": bg.BC_RECIP}
TD = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def ref_values(var, op, eps=1e-5):
    return np.array([oracle.bcast_value(OPS[op], float(v), eps) for v in var.numpy()])


def check_planes(out, var, op, dt, eps=1e-5):
    """Every plane (n, c) must hold one value, equal to op(var[c]) within bounds."""
    N, C, H, W = out.shape
    ref64 = ref_values(var, op, eps)
    if dt == "f32":
        refq = ref64.astype(np.float32).astype(np.float64)
        bound = 2 * ulp(refq, "f32")
    else:
        # the kernel rounds its fp32 value once more to the output type
        refq = ref64
        bound = 2 * ulp(ref64.astype(np.float32), "f32") + ulp(ref64, dt)
    o = out.float().cpu().reshape(N, C, H * W).double().numpy()
    first = o[:, :, :1]
    assert np.array_equal(np.isnan(o), np.isnan(np.broadcast_to(first, o.shape)))
    same = (o == first) | (np.isnan(o) & np.isnan(first))
    assert same.all(), "a plane holds more than one value"
    for n in range(N):
        assert_within(o[n, :, 0], refq, bound, f"bcast {op} {dt} n={n}")


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("op", list(OPS))
@pytest.mark.parametrize("shape", [(2, 5, 4, 8), (3, 7, 5, 3), (1, 33, 1, 1), (4, 16, 9, 9)])
def test_bcast_small(shape, op, dt):
    N, C, H, W = shape
    var = synth.bcast_var(C, seed=C)
    if op == "rsqrt":
        var[0] = 0.0
        var[-1] = -float(np.float32(1e-5))   # the float sum is exactly zero: +inf
    out = torch.full((N, C, H, W), 7.0, dtype=TD[dt], device="cuda")
    bg.bcast_nchw_run(N, C, H, W, OPS[op], var.cuda(), 1e-5, out, bg.DTYPE_CODES[dt])
    torch.cuda.synchronize()
    check_planes(out, var, op, dt)
    out2 = torch.full_like(out, 7.0)
    bg.bcast_nchw_run_flat(N, C, H, W, OPS[op], var.cuda(), 1e-5, out2, bg.DTYPE_CODES[dt])
    torch.cuda.synchronize()
    assert torch.equal(torch.nan_to_num(out, 1.0), torch.nan_to_num(out2, 1.0))


@pytest.mark.parametrize("op", ["exp", "rsqrt"])
def test_bcast_full_size(op):
    N, C, H, W = synth.BCAST_SHAPE
    var = synth.bcast_var(C, seed=0)
    out = torch.empty((N, C, H, W), dtype=torch.float32, device="cuda")
    bg.bcast_nchw_run(N, C, H, W, OPS[op], var.cuda(), synth.BCAST_EPS, out, bg.F32)
    torch.cuda.synchronize()
    check_planes(out, var, op, "f32")
    if op == "rsqrt":   # var ~ U[-2,2]: about half the channels are NaN
        assert 0.3 < torch.isnan(out[0, :, 0, 0]).float().mean().item() < 0.7


def test_bcast_unaligned_output_pointer():
    N, C, H, W = 2, 6, 4, 4
    var = synth.bcast_var(C, seed=9)
    buf = torch.zeros(N * C * H * W + 1, dtype=torch.float32, device="cuda")
    out = buf[1:].view(N, C, H, W)
    bg.bcast_nchw_run(N, C, H, W, bg.BC_EXP, var.cuda(), 1e-5, out, bg.F32)
    torch.cuda.synchronize()
    assert buf[0].item() == 0.0
    check_planes(out, var, "exp", "f32")
