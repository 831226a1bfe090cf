"""Pins for the CPU oracle, each against something other than the oracle itself.

* hand-worked integer cases (tests/golden/conv_hand_cases.txt);
* closed forms: 1x1 identity, centre-tap identity, all-ones counts, a single
  spike kernel that shifts the image, a negated batch image;
* the output-size rule floor((H + 2p - K)/s) + 1 on the workload shapes;
* the FLOP count against the tuning log printed with the TVM tutorial;
* a float64 library convolution (torch CPU) on small random shapes;
* the broadcast's special values (0, +inf, NaN) and its plane structure.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.golden_io import hand_cases, tuning_log


def _conv(orc, shape, data, kernel, **kw):
    N, CI, H, W, CO, KH, KW, s, p, g = shape
    x = np.asarray(data, np.float64).reshape(N, CI, H, W)
    w = np.asarray(kernel, np.float64).reshape(CO, CI // g, KH, KW)
    return oracle.conv2d_nchw(x, w, stride=s, pad=p, groups=g, lib=orc, **kw)


@pytest.mark.parametrize("case", hand_cases(), ids=lambda c: c["name"])
def test_hand_cases(orc, case):
    out, sabs = _conv(orc, case["shape"], case["data"], case["kernel"])
    np.testing.assert_array_equal(out.ravel(), case["out"])
    np.testing.assert_array_equal(sabs.ravel(), case["absum"])


@pytest.mark.parametrize("case", hand_cases(), ids=lambda c: c["name"])
def test_hand_cases_points(orc, case):
    """The sampled-output entry point agrees with the worked values at every index."""
    N, CI, H, W, CO, KH, KW, s, p, g = case["shape"]
    x = case["data"].reshape(N, CI, H, W)
    w = case["kernel"].reshape(CO, CI // g, KH, KW)
    idx = np.arange(case["out"].size)[::-1].copy()
    out, sabs = oracle.conv2d_nchw_points(x, w, idx, stride=s, pad=p, groups=g, lib=orc)
    np.testing.assert_array_equal(out, case["out"][idx])
    np.testing.assert_array_equal(sabs, case["absum"][idx])


def test_epilogue_bias_exp_per_channel(orc):
    case = [c for c in hand_cases() if c["name"] == "two_channels_two_filters_1x1"][0]
    bias = np.array([0.25, -0.5])
    hand = case["out"].reshape(1, 2, 2, 2)
    out, _ = _conv(orc, case["shape"], case["data"], case["kernel"] / 64.0,
                   bias=bias, epi=oracle.EPI_BIAS_EXP)
    want = np.exp(hand / 64.0 + bias.reshape(1, 2, 1, 1))
    np.testing.assert_allclose(out, want, rtol=1e-15)
    out, _ = _conv(orc, case["shape"], case["data"], case["kernel"],
                   bias=bias, epi=oracle.EPI_BIAS)
    np.testing.assert_array_equal(out, hand + bias.reshape(1, 2, 1, 1))
    out, _ = _conv(orc, case["shape"], case["data"], case["kernel"],
                   bias=bias, epi=oracle.EPI_BIAS_RSQRT, eps=0.25)
    np.testing.assert_allclose(out, 1.0 / np.sqrt(hand + bias.reshape(1, 2, 1, 1) + 0.25),
                               rtol=1e-15)
    # div: the reciprocal of the biased sum, per channel
    out, _ = _conv(orc, case["shape"], case["data"], case["kernel"],
                   bias=bias, epi=oracle.EPI_BIAS_RECIP)
    np.testing.assert_allclose(out, 1.0 / (hand + bias.reshape(1, 2, 1, 1)), rtol=1e-15)


def test_epilogue_recip_closed_form(orc):
    """All-ones data and kernel: an interior output sums CI*K*K ones, a corner of
    a pad-1 3x3 conv only the 4 taps inside the image, so with bias b the
    reciprocal is 1/(count + b) exactly, sign included."""
    CI, CO, H, W = 3, 2, 5, 6
    x = np.ones((1, CI, H, W))
    w = np.ones((CO, CI, 3, 3))
    bias = np.array([-30.0, 0.5])
    out, _ = oracle.conv2d_nchw(x, w, stride=1, pad=1, bias=bias, epi=oracle.EPI_BIAS_RECIP, lib=orc)
    assert out[0, 0, 2, 2] == 1.0 / (27 - 30.0) and out[0, 1, 2, 2] == 1.0 / 27.5
    assert out[0, 0, 0, 0] == 1.0 / (12 - 30.0) and out[0, 1, 0, 0] == 1.0 / 12.5


def test_epilogue_relu_hand_case(orc):
    """add + ReLU on the hand-worked 1x1 case: max(conv + bias[f], 0) per
    channel, with channel 0's bias set so that its outputs fall on both sides
    of zero (and one exactly on it)."""
    case = [c for c in hand_cases() if c["name"] == "two_channels_two_filters_1x1"][0]
    hand = case["out"].reshape(1, 2, 2, 2)
    bias = np.array([-hand[0, 0, 0, 1], 0.5])
    out, _ = _conv(orc, case["shape"], case["data"], case["kernel"], bias=bias,
                   epi=oracle.EPI_BIAS_RELU)
    np.testing.assert_array_equal(out, np.maximum(hand + bias.reshape(1, 2, 1, 1), 0.0))
    assert out[0, 0, 0, 1] == 0.0
    assert (out[0, 0] == 0.0).any() and (out[0, 0] > 0.0).any()


def test_epilogue_relu_closed_form(orc):
    """All-ones data and kernel, 3x3 pad 1, CI = 3: an output sums 27 ones inside,
    18 on an edge, 12 in a corner.  With bias -20 channel 0 keeps only the
    interior (7), with -12.5 channel 1 keeps interior and edges (14.5, 5.5) and
    zeroes the corners."""
    out, _ = oracle.conv2d_nchw(np.ones((1, 3, 5, 6)), np.ones((2, 3, 3, 3)), stride=1, pad=1,
                                bias=np.array([-20.0, -12.5]), epi=oracle.EPI_BIAS_RELU, lib=orc)
    assert out[0, 0, 2, 2] == 7.0 and out[0, 0, 0, 2] == 0.0 and out[0, 0, 0, 0] == 0.0
    assert out[0, 1, 2, 2] == 14.5 and out[0, 1, 0, 2] == 5.5 and out[0, 1, 0, 0] == 0.0


def _rand(shape, seed):
    return np.random.default_rng(seed).uniform(-1, 1, shape)


@pytest.mark.parametrize("K,p", [(1, 0), (3, 1), (5, 2)])
def test_identity_kernels(orc, K, p):
    """A kernel that is the identity on channels at the centre tap returns the input."""
    CI, H, W = 5, 6, 7
    x = _rand((2, CI, H, W), 1)
    w = np.zeros((CI, CI, K, K))
    for c in range(CI):
        w[c, c, K // 2, K // 2] = 1.0
    out, sabs = oracle.conv2d_nchw(x, w, stride=1, pad=p, lib=orc)
    np.testing.assert_array_equal(out, x)
    np.testing.assert_array_equal(sabs, np.abs(x))


@pytest.mark.parametrize("H,W,K,s,p", [(5, 7, 3, 1, 1), (6, 5, 3, 2, 1), (7, 7, 5, 1, 2),
                                       (8, 9, 3, 2, 0), (4, 4, 1, 1, 0), (9, 6, 5, 3, 2)])
def test_all_ones_counts_valid_taps(orc, H, W, K, s, p):
    """data = 1, kernel = 1: out = CI * (#taps inside the image), a per-axis count."""
    CI, CO = 3, 2
    out, sabs = oracle.conv2d_nchw(np.ones((1, CI, H, W)), np.ones((CO, CI, K, K)),
                                   stride=s, pad=p, lib=orc)
    Ho, Wo = (H + 2 * p - K) // s + 1, (W + 2 * p - K) // s + 1
    cy = [sum(1 for r in range(K) if 0 <= y * s + r - p < H) for y in range(Ho)]
    cx = [sum(1 for r in range(K) if 0 <= x * s + r - p < W) for x in range(Wo)]
    want = CI * np.outer(cy, cx)
    assert out.shape == (1, CO, Ho, Wo)
    for f in range(CO):
        np.testing.assert_array_equal(out[0, f], want)
    np.testing.assert_array_equal(sabs, out)


@pytest.mark.parametrize("ry,rx", [(0, 0), (0, 2), (2, 1), (1, 0)])
def test_spike_kernel_shifts(orc, ry, rx):
    """A single non-zero tap at (ry, rx) reads the input shifted by (ry-p, rx-p)."""
    H, W, K, p = 5, 6, 3, 1
    x = _rand((1, 2, H, W), 2)
    w = np.zeros((1, 2, K, K))
    w[0, 1, ry, rx] = 1.0
    out, _ = oracle.conv2d_nchw(x, w, stride=1, pad=p, lib=orc)
    for y in range(H):
        for xx in range(W):
            iy, ix = y + ry - p, xx + rx - p
            want = x[0, 1, iy, ix] if (0 <= iy < H and 0 <= ix < W) else 0.0
            assert out[0, 0, y, xx] == want


@pytest.mark.parametrize("H,K,s,p,want", [
    (7, 3, 1, 1, 7), (56, 3, 1, 1, 56), (56, 1, 1, 0, 56), (14, 3, 2, 1, 7),
    (28, 1, 2, 0, 14), (112, 3, 2, 1, 56), (14, 5, 1, 2, 14), (32, 3, 1, 1, 32),
    (2, 3, 1, 0, 0), (5, 5, 1, 0, 1)])
def test_output_size_rule(orc, H, K, s, p, want):
    assert oracle.out_size(H, K, s, p, lib=orc) == want


def test_flop_count_matches_tuning_log(orc):
    """2*N*CO*Ho*Wo*CI*KH*KW for the tuned layer reproduces every GFLOPS figure in the
    log within 0.3% (plus the half-unit of its printed two decimals); adding the padding stage's element-wise work (7 compare/and ops
    per padded element, the reading that explains the residual) reproduces each
    printed figure to its two decimals."""
    flops = oracle.conv_flops(1, 512, 7, 7, 512, 3, 3, 1, 1, lib=orc)
    assert flops == 231_211_008
    pad_ops = 7 * 1 * 512 * (7 + 2) * (7 + 2)
    log = tuning_log()
    assert len(log["trials"]) == 5
    for _, gflops, cost in log["trials"]:
        assert abs(flops / cost / 1e9 - gflops) <= 3e-3 * gflops + 0.005
        assert round((flops + pad_ops) / cost / 1e9, 2) == gflops
    # the best trial and the 400-run re-timing agree to 2%
    best = min(c for _, _, c in log["trials"])
    assert abs(best - log["retimed"]) / best < 0.02


@pytest.mark.parametrize("N,CI,CO,H,W,KH,KW,s,p,g", [
    (2, 3, 4, 9, 7, 3, 3, 1, 1, 1),
    (1, 6, 5, 8, 8, 3, 3, 2, 1, 1),
    (1, 4, 4, 10, 11, 5, 5, 1, 2, 4),
    (2, 6, 6, 9, 9, 3, 3, 2, 1, 6),
    (1, 4, 6, 7, 9, 1, 3, 1, 1, 2),
    (1, 8, 3, 5, 5, 2, 4, 3, 2, 1),
    (3, 2, 2, 4, 4, 4, 4, 1, 0, 1),
])
def test_against_float64_library_conv(orc, N, CI, CO, H, W, KH, KW, s, p, g):
    rng = np.random.default_rng(N * 1000 + CI * 100 + CO)
    x = rng.uniform(-1, 1, (N, CI, H, W))
    w = rng.uniform(-1, 1, (CO, CI // g, KH, KW))
    b = rng.uniform(-1, 1, (CO,))
    out, sabs = oracle.conv2d_nchw(x, w, stride=s, pad=p, groups=g, lib=orc)
    ref = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(w),
                                     stride=s, padding=p, groups=g).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    sref = torch.nn.functional.conv2d(torch.from_numpy(np.abs(x)), torch.from_numpy(np.abs(w)),
                                      stride=s, padding=p, groups=g).numpy()
    np.testing.assert_allclose(sabs, sref, rtol=0, atol=1e-12)
    outb, _ = oracle.conv2d_nchw(x, w, stride=s, pad=p, groups=g, bias=b,
                                 epi=oracle.EPI_BIAS_EXP, lib=orc)
    np.testing.assert_allclose(outb, np.exp(ref + b.reshape(1, -1, 1, 1)), rtol=1e-12)


def test_points_match_full(orc):
    rng = np.random.default_rng(7)
    x = rng.uniform(-1, 1, (2, 6, 9, 10))
    w = rng.uniform(-1, 1, (4, 3, 3, 3))
    out, sabs = oracle.conv2d_nchw(x, w, stride=2, pad=1, groups=2, lib=orc)
    idx = rng.choice(out.size, 50, replace=False)
    po, ps = oracle.conv2d_nchw_points(x, w, idx, stride=2, pad=1, groups=2, lib=orc)
    np.testing.assert_array_equal(po, out.ravel()[idx])
    np.testing.assert_array_equal(ps, sabs.ravel()[idx])


def test_invalid_shapes_rejected(orc):
    with pytest.raises(ValueError):
        oracle.conv2d_nchw(np.ones((1, 3, 2, 2)), np.ones((1, 3, 3, 3)), pad=0, lib=orc)
    with pytest.raises(ValueError):
        oracle.conv2d_nchw_points(np.ones((1, 1, 3, 3)), np.ones((1, 1, 3, 3)), [9], pad=1,
                                  lib=orc)


def test_abs_sum_bounds_output(orc):
    rng = np.random.default_rng(3)
    x = rng.uniform(-1, 1, (2, 5, 8, 8))
    w = rng.uniform(-1, 1, (3, 5, 3, 3))
    out, sabs = oracle.conv2d_nchw(x, w, stride=1, pad=1, lib=orc)
    assert np.all(np.abs(out) <= sabs + 1e-15)


# ------------------------------------------------------------------ broadcast

def test_bcast_special_values(orc):
    f32 = np.float32
    assert oracle.bcast_value(oracle.BC_EXP, 0.0, lib=orc) == 1.0
    assert oracle.bcast_value(oracle.BC_COPY, 0.75, lib=orc) == 0.75
    assert abs(oracle.bcast_value(oracle.BC_EXP, 1.0, lib=orc) - math.e) <= 4.5e-16
    # rsqrt(0 + 1e-5f): the argument is the float nearest 1e-5
    assert oracle.bcast_value(oracle.BC_RSQRT, 0.0, 1e-5, lib=orc) == \
        1.0 / math.sqrt(float(f32(1e-5)))
    # var = -1e-5f: the float sum is exactly zero -> +inf
    assert oracle.bcast_value(oracle.BC_RSQRT, float(-f32(1e-5)), 1e-5, lib=orc) == math.inf
    assert math.isnan(oracle.bcast_value(oracle.BC_RSQRT, -1.0, 1e-5, lib=orc))
    assert oracle.bcast_value(oracle.BC_RSQRT, 3.0, 1.0, lib=orc) == 0.5
    assert oracle.bcast_value(oracle.BC_RECIP, 4.0, lib=orc) == 0.25


def test_bcast_plane_structure(orc):
    """Every (n, h, w) of channel c holds op(var[c]); channels differ."""
    N, C, H, W = 3, 5, 4, 6
    var = np.array([0.0, 1.0, -1.0, 2.0, 0.5], np.float32)
    out = oracle.bcast_nchw(N, C, H, W, oracle.BC_EXP, var, lib=orc)
    assert out.shape == (N, C, H, W)
    for c in range(C):
        assert np.all(out[:, c] == out[0, c, 0, 0])
    np.testing.assert_allclose(out[0, :, 0, 0], np.exp(var.astype(np.float64)), rtol=1e-15)
    assert out[0, 0, 0, 0] == 1.0 and out[1, 1, 2, 3] == math.exp(1.0)


def test_bcast_rsqrt_eps_is_a_float_add(orc):
    """The +eps of rsqrt(var + eps) is one fp32 addition (the device's order of
    operations); 1 + 1e-5 is not representable in fp32, so this pins the step."""
    f32 = np.float32
    got = oracle.bcast_value(oracle.BC_RSQRT, 1.0, 1e-5, lib=orc)
    assert got == 1.0 / math.sqrt(float(f32(1.0) + f32(1e-5)))
    assert got != 1.0 / math.sqrt(1.0 + float(f32(1e-5)))
