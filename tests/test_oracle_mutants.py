"""The oracle's pins catch plausible mistakes.

Each case copies oracle/oracle.c, plants one mistake in the copy (a dropped
term, a wrong sign or index, a transposed operand, a wrong rounding step),
compiles it on the CPU, and checks that the pin battery below rejects it --
while the unmodified oracle passes the same battery.
"""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tests.golden_io import hand_cases, tuning_log

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "kernel_taps_transposed": ("* s->KH + ry) * s->KW + rx]", "* s->KH + rx) * s->KW + ry]"),
    "pad_sign_flipped_rows": ("y * s->stride + ry - s->pad", "y * s->stride + ry + s->pad"),
    "group_offset_dropped": ("const int ci = g * cig + rc;", "const int ci = rc;"),
    "last_column_tap_dropped": ("rx < s->KW; ++rx", "rx < s->KW - 1; ++rx"),
    "out_size_ceil": ("return span / stride + 1;", "return (span + stride - 1) / stride + 1;"),
    "absum_signed": ("sabs += fabs(a * w);", "sabs += a * w;"),
    "bias_channel_zero": ("return exp(acc + bias[f]);", "return exp(acc + bias[0]);"),
    "recip_bias_dropped": ("return 1.0 / (acc + bias[f]);", "return 1.0 / acc;"),
    "rsqrt_eps_dropped": ("return 1.0 / sqrt(acc + bias[f] + eps);", "return 1.0 / sqrt(acc + bias[f]);"),
    "relu_before_bias": ("return acc + bias[f] > 0.0 ? acc + bias[f] : 0.0;",
                         "return (acc > 0.0 ? acc : 0.0) + bias[f];"),
    "relu_dropped": ("return acc + bias[f] > 0.0 ? acc + bias[f] : 0.0;", "return acc + bias[f];"),
    "eps_added_in_double": ("volatile float t = v + eps;", "volatile double t = (double)v + eps;"),
    "image_index_dropped": ("data[(((size_t)n * s->CI + ci)", "data[(((size_t)0 * s->CI + ci)"),
    "flops_missing_factor2": ("return 2.0 * N * CO", "return 1.0 * N * CO"),
}


def _build_variant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    return oracle.load(oracle.build(force=True, src=str(path), out=str(tmp_path / f"{name}.so")))


def _battery(lib):
    """Returns the list of failed pins (empty = all pass)."""
    failed = []
    for c in hand_cases():
        N, CI, H, W, CO, KH, KW, s, p, g = c["shape"]
        x = c["data"].reshape(N, CI, H, W)
        w = c["kernel"].reshape(CO, CI // g, KH, KW)
        try:
            out, sabs = oracle.conv2d_nchw(x, w, stride=s, pad=p, groups=g, lib=lib)
            if not (np.array_equal(out.ravel(), c["out"]) and np.array_equal(sabs.ravel(), c["absum"])):
                failed.append("hand:" + c["name"])
        except ValueError:
            failed.append("hand-rejected:" + c["name"])
    rng = np.random.default_rng(11)
    for (N, CI, CO, H, W, KH, KW, s, p, g) in [(2, 3, 4, 9, 7, 3, 3, 1, 1, 1),
                                               (1, 4, 4, 10, 11, 5, 5, 2, 2, 4)]:
        x = rng.uniform(-1, 1, (N, CI, H, W))
        w = rng.uniform(-1, 1, (CO, CI // g, KH, KW))
        b = rng.uniform(-1, 1, (CO,))
        ref = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(w), stride=s,
                                         padding=p, groups=g).numpy()
        try:
            out, _ = oracle.conv2d_nchw(x, w, stride=s, pad=p, groups=g, bias=b,
                                        epi=oracle.EPI_BIAS_EXP, lib=lib)
            if out.shape != ref.shape or not np.allclose(out, np.exp(ref + b.reshape(1, -1, 1, 1)),
                                                         rtol=1e-12, atol=0):
                failed.append("torch")
        except ValueError:
            failed.append("torch-rejected")
    if oracle.out_size(14, 3, 2, 1, lib=lib) != 7:
        failed.append("out_size")
    flops = oracle.conv_flops(1, 512, 7, 7, 512, 3, 3, 1, 1, lib=lib)
    if any(abs(flops / cost / 1e9 - gf) > 3e-3 * gf + 0.005 for _, gf, cost in tuning_log()["trials"]):
        failed.append("flops")
    f32 = np.float32
    if oracle.bcast_value(oracle.BC_RSQRT, 1.0, 1e-5, lib=lib) != \
            1.0 / math.sqrt(float(f32(1.0) + f32(1e-5))):
        failed.append("rsqrt_eps_fp32")
    if oracle.bcast_value(oracle.BC_EXP, 0.0, lib=lib) != 1.0:
        failed.append("exp0")
    # div epilogue on all-ones data and kernel (interior sum 27, corner 12)
    try:
        out, _ = oracle.conv2d_nchw(np.ones((1, 3, 5, 6)), np.ones((2, 3, 3, 3)), stride=1, pad=1,
                                    bias=np.array([-30.0, 0.5]), epi=oracle.EPI_BIAS_RECIP, lib=lib)
        if out[0, 0, 2, 2] != 1.0 / -3.0 or out[0, 1, 0, 0] != 1.0 / 12.5:
            failed.append("recip")
    except ValueError:
        failed.append("recip-rejected")
    # rsqrt epilogue with eps on the same sums: 1/sqrt(27 - 26 + 0.25) inside
    try:
        out, _ = oracle.conv2d_nchw(np.ones((1, 3, 5, 6)), np.ones((2, 3, 3, 3)), stride=1, pad=1,
                                    bias=np.array([-26.0, 0.5]), epi=oracle.EPI_BIAS_RSQRT, eps=0.25,
                                    lib=lib)
        if out[0, 0, 2, 2] != 1.0 / math.sqrt(1.25):
            failed.append("rsqrt")
    except ValueError:
        failed.append("rsqrt-rejected")
    # add + ReLU: interior 27 - 20 = 7, a corner 12 - 12.5 clamps to 0
    try:
        out, _ = oracle.conv2d_nchw(np.ones((1, 3, 5, 6)), np.ones((2, 3, 3, 3)), stride=1, pad=1,
                                    bias=np.array([-20.0, -12.5]), epi=oracle.EPI_BIAS_RELU, lib=lib)
        if out[0, 0, 2, 2] != 7.0 or out[0, 1, 0, 0] != 0.0 or out[0, 1, 0, 2] != 5.5:
            failed.append("relu")
    except ValueError:
        failed.append("relu-rejected")
    return failed


@pytest.fixture(scope="module")
def have_gcc():
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")


def test_unmodified_oracle_passes_battery(orc, have_gcc):
    assert _battery(orc) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, have_gcc, name):
    old, new = MUTANTS[name]
    lib = _build_variant(tmp_path, name, old, new)
    assert _battery(lib), f"planted mistake {name} passed every pin"
