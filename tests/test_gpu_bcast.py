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
    check_planes(out2, var, op, dt)       # the flat schedule against the oracle itself
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


@pytest.mark.parametrize("op", list(OPS))
def test_bcast_flat_full_size(op):
    # the fused-flat-index schedule (one flat loop, op(var[c]) recomputed per
    # element) at the benchmark's size, against the oracle
    N, C, H, W = synth.BCAST_SHAPE
    var = synth.bcast_var(C, seed=3)
    out = torch.full((N, C, H, W), 7.0, dtype=torch.float32, device="cuda")
    bg.bcast_nchw_run_flat(N, C, H, W, OPS[op], var.cuda(), synth.BCAST_EPS, out, bg.F32)
    torch.cuda.synchronize()
    check_planes(out, var, op, "f32")


def test_bcast_unaligned_output_pointer():
    N, C, H, W = 2, 6, 4, 4
    var = synth.bcast_var(C, seed=9)
    buf = torch.zeros(N * C * H * W + 1, dtype=torch.float32, device="cuda")
    out = buf[1:].view(N, C, H, W)
    bg.bcast_nchw_run(N, C, H, W, bg.BC_EXP, var.cuda(), 1e-5, out, bg.F32)
    torch.cuda.synchronize()
    assert buf[0].item() == 0.0
    check_planes(out, var, "exp", "f32")


# ---------------------------------------------------------- [1,P,1] => [B0,P,B1]
# The general form is the NCHW one with N = B0, C = P, H*W = B1, so the same
# oracle values and plane check apply (viewed as [B0, P, 1, B1]).  Short rows
# (B1 * element size < 1 KB) take the short-row kernel, long rows the
# per-channel one; both vector and element stores.
GENERAL = [
    (3, 5, 1), (2, 7, 3), (4, 64, 4), (1, 1000, 2), (5, 9, 17), (2, 33, 64), (7, 3, 255),
    (2, 6, 256), (3, 4, 1031), (128, 2, 8), (1, 1, 1),
]


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("op", ["copy", "exp", "rsqrt", "recip"])
@pytest.mark.parametrize("shape", GENERAL, ids=lambda s: "x".join(map(str, s)))
def test_bcast_general(shape, op, dt):
    B0, P, B1 = shape
    var = synth.bcast_var(P, seed=P + B1)
    if op == "rsqrt" and P > 1:
        var[0] = 0.0
    guard = 64
    buf = torch.full((B0 * P * B1 + 2 * guard,), 7.0, dtype=TD[dt], device="cuda")
    out = buf[guard:guard + B0 * P * B1].view(B0, P, 1, B1)
    bg.bcast_run(B0, P, B1, OPS[op], var.cuda(), 1e-5, out, bg.DTYPE_CODES[dt])
    torch.cuda.synchronize()
    assert bool(torch.all(buf[:guard] == 7.0)) and bool(torch.all(buf[-guard:] == 7.0))
    check_planes(out, var, op, dt)


@pytest.mark.parametrize("shape", [(16, 1024, 49), (8, 3, 100000), (64, 4096, 1)])
def test_bcast_general_unaligned_and_large(shape):
    # output 4 bytes past a 16-byte boundary: element stores in either kernel
    B0, P, B1 = shape
    var = synth.bcast_var(P, seed=3)
    buf = torch.zeros(B0 * P * B1 + 1, dtype=torch.float32, device="cuda")
    out = buf[1:].view(B0, P, 1, B1)
    bg.bcast_run(B0, P, B1, bg.BC_EXP, var.cuda(), 1e-5, out, bg.F32)
    torch.cuda.synchronize()
    assert buf[0].item() == 0.0
    check_planes(out, var, "exp", "f32")


def test_bcast_general_matches_nchw():
    N, C, H, W = 4, 12, 5, 7
    var = synth.bcast_var(C, seed=4).cuda()
    a = torch.empty((N, C, H, W), dtype=torch.float16, device="cuda")
    b = torch.empty_like(a)
    bg.bcast_nchw_run(N, C, H, W, bg.BC_RSQRT, var, 1e-5, a, bg.F16)
    bg.bcast_run(N, C, H * W, bg.BC_RSQRT, var, 1e-5, b, bg.F16)
    torch.cuda.synchronize()
    assert torch.equal(torch.nan_to_num(a, 1.0), torch.nan_to_num(b, 1.0))


@pytest.mark.parametrize("args,status", [((0, 4, 4), 1), ((2, 0, 4), 1), ((2, 4, 0), 1),
                                         ((1, 65536, 65536), 2)])
def test_bcast_general_rejects(args, status):
    var = torch.zeros(4, dtype=torch.float32, device="cuda")
    out = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(bg.BigemmError) as e:
        bg.bcast_run(*args, bg.BC_EXP, var, 1e-5, out, bg.F32)
    assert e.value.status == status
