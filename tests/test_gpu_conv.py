"""GPU parity of the convolution kernels against the CPU oracle, through the C ABI.

Every case draws seeded inputs, runs the library (heuristic plan, a forced
kernel, or the timed search), and compares every output element with the
oracle's fp64 result within the bound of tests/tolerance.py.  Outputs start
NaN-filled inside a guard band, so an unwritten element or a write outside
the tensor fails the case.  Full-size cases (the benchmark's batch sizes)
compare sampled output positions.
"""
import os

import numpy as np
import pytest
import torch

import broadcast_implicit_gemm_gb300 as bg
import oracle
from broadcast_implicit_gemm_gb300 import synth
from tests.tolerance import TAU, assert_within, conv_bound, epi_bound

pytestmark = pytest.mark.gpu

DT = {"f32": bg.F32, "f16": bg.F16, "bf16": bg.BF16}
NTH = max(1, os.cpu_count() or 1)
GUARD = 4096
SENTINEL = -7.25   # exact in fp32, fp16 and bf16


def _alloc_out(shape, dtype):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=dtype, device="cuda")
    out = buf[GUARD:GUARD + n].view(shape)
    out.fill_(float("nan"))
    return buf, out


def _guard_intact(buf):
    g = torch.cat([buf[:GUARD], buf[-GUARD:]]).float().cpu()
    return bool(torch.all(g == SENTINEL))


def run(spec, options=None, search=0, seed=0, eps=1e-5):
    x, w, b = synth.conv_inputs(spec, seed)
    epi = bg.EPI_NAMES[spec.epi]
    plan = bg.conv2d_nchw_plan_ex(spec.N, spec.H, spec.W, spec.CO, spec.CI, spec.K, spec.K,
                                  spec.stride, spec.pad, spec.groups, DT[spec.in_dtype],
                                  DT[spec.out_dtype], epi, search, options)
    Ho = bg.out_size(spec.H, spec.K, spec.stride, spec.pad)
    Wo = bg.out_size(spec.W, spec.K, spec.stride, spec.pad)
    buf, out = _alloc_out((spec.N, spec.CO, Ho, Wo), synth.TORCH_DTYPES[spec.out_dtype])
    bg.conv2d_nchw_run(plan, x.cuda(), w.cuda(), b.cuda() if b is not None else None, eps, out)
    torch.cuda.synchronize()
    assert bg.bigemm_last_device_error() == 0, "a device wait timed out"
    assert _guard_intact(buf), "write outside the output tensor"
    info = plan.describe()
    plan.close()
    return info, x, w, b, out


def tau_for(spec, info):
    if spec.in_dtype in ("f16", "bf16"):
        return TAU["half"]
    return TAU["tf32"] if info["kind"] == "umma" else TAU["fp32"]


def check(spec, options=None, search=0, seed=0):
    info, x, w, b, out = run(spec, options, search, seed)
    got = out.cpu().double().numpy()
    tau = tau_for(spec, info)
    if spec.epi == "none":
        ref, sabs = oracle.conv2d_nchw(x, w, stride=spec.stride, pad=spec.pad, groups=spec.groups,
                                       nthreads=NTH)
        bound = conv_bound(ref, sabs, tau, spec.out_dtype)
    else:
        epi = {"bias": oracle.EPI_BIAS, "bias_exp": oracle.EPI_BIAS_EXP,
               "bias_rsqrt": oracle.EPI_BIAS_RSQRT, "bias_recip": oracle.EPI_BIAS_RECIP,
               "bias_relu": oracle.EPI_BIAS_RELU}[spec.epi]
        ref, sabs = oracle.conv2d_nchw(x, w, stride=spec.stride, pad=spec.pad, groups=spec.groups,
                                       bias=b, epi=epi, nthreads=NTH)
        pre, _ = oracle.conv2d_nchw(x, w, stride=spec.stride, pad=spec.pad, groups=spec.groups,
                                    nthreads=NTH)
        arg = pre + b.double().numpy().reshape(1, -1, 1, 1)
        bound = epi_bound(arg, sabs, tau, spec.epi, spec.out_dtype, ref)
    assert_within(got, ref, bound, f"{spec.name} [{info['cand']}]")
    return info


# ------------------------------------------------- workload shapes, heuristic plan
SMALL = ([s for s in synth.RESNET_LAST] + synth.SWEEP_FP32
         + [s.with_batch(2) for s in synth.RESNET50_FP16]
         + [s.with_batch(2) for s in synth.FUSED_CONV]
         + [s.with_batch(2) for s in synth.DEPTHWISE_FP16])


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
def test_workload_shapes_heuristic(spec):
    info = check(spec)
    if spec.groups == 1:
        assert info["kind"] == "umma"


# ------------------------------------------------- every kernel, forced
FORCED_SHAPES = [synth.SWEEP_FP32[0], synth.SWEEP_FP32[3], synth.SWEEP_FP32[4],
                 synth.RESNET50_FP16[1].with_batch(1), synth.RESNET50_FP16[4].with_batch(1)]


@pytest.mark.parametrize("spec", FORCED_SHAPES, ids=lambda s: s.name)
def test_simt_tiled_matches(spec):
    info = check(spec, {"kind": bg.KIND_SIMT})
    assert info["cand"] == "simt:tiled"


@pytest.mark.parametrize("bn", [64, 128, 256])
@pytest.mark.parametrize("spec", [synth.SWEEP_FP32[1], synth.RESNET50_FP16[1].with_batch(1),
                                  synth.RESNET50_FP16[3].with_batch(2)], ids=lambda s: s.name)
def test_umma_tile_n(spec, bn):
    info = check(spec, {"kind": bg.KIND_UMMA, "tile_n": bn})
    assert info["kind"] == "umma" and info["bn"] == bn


@pytest.mark.parametrize("split", [1, 2, 3, 8, 32])
def test_umma_split_k(split):
    spec = synth.RESNET_LAST[0]
    info = check(spec, {"kind": bg.KIND_UMMA, "tile_n": 128, "split_k": split})
    kb = info["k_blocks"]
    assert info["split"] == -(-kb // -(-kb // split))   # slices of ceil(kb/split) blocks


@pytest.mark.parametrize("box", [(8, 16), (16, 8), (32, 4), (64, 2), (8, 8), (8, 4), (56, 1)])
def test_umma_pixel_boxes(box):
    spec = synth.RESNET50_FP16[1].with_batch(1)
    info = check(spec, {"kind": bg.KIND_UMMA, "box_w": box[0], "box_h": box[1]})
    assert info["box"][:2] == list(box) and info["amode"] == "nhwc"


def test_umma_direct_and_nhwc_agree_on_1x1():
    spec = synth.RESNET50_FP16[2].with_batch(2)
    a = check(spec, {"kind": bg.KIND_UMMA, "tile_n": 128})
    b = check(spec, {"kind": bg.KIND_UMMA, "tile_n": 128, "box_w": 8, "box_h": 16})
    assert a["amode"] == "direct" and b["amode"] == "nhwc"


# ------------------------------------------------- halo mode (stride 1, K x K)
def _H(name, N, CI, CO, H, W, K, p, i="f16", o="f16", epi="none"):
    return synth.ConvSpec(name, N, CI, CO, H, W, K, 1, p, 1, i, o, "uniform", "he", epi)


HALO = [
    synth.RESNET50_FP16[1].with_batch(1),
    synth.SWEEP_FP32[0], synth.SWEEP_FP32[1], synth.SWEEP_FP32[2],
    _H("halo_ragged_13x11_ci24_co40", 2, 24, 40, 13, 11, 3, 1),
    _H("halo_k5_bf16", 1, 32, 96, 17, 19, 5, 2, i="bf16", o="bf16"),
    _H("halo_k7_pad3", 1, 16, 64, 20, 18, 7, 3),
    _H("halo_k3_pad0", 2, 64, 128, 18, 18, 3, 0),
    _H("halo_exp_f32out", 2, 64, 256, 32, 32, 3, 1, o="f32", epi="bias_exp"),
    _H("halo_rect_1x3", 1, 64, 64, 9, 30, 3, 1),
]


@pytest.mark.parametrize("spec", HALO, ids=lambda s: s.name)
def test_umma_halo_mode(spec):
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO})
    assert info["amode"] == "halo"


@pytest.mark.parametrize("bn", [64, 128, 256])
def test_umma_halo_tile_n(bn):
    spec = _H("halo_bn", 1, 64, 300, 20, 24, 3, 1)
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO, "tile_n": bn})
    assert info["bn"] == bn and info["amode"] == "halo"


@pytest.mark.parametrize("split", [2, 4, 16])
def test_umma_halo_split_k(split):
    spec = synth.RESNET_LAST[0]
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO, "tile_n": 128, "split_k": split})
    assert info["amode"] == "halo" and info["split"] > 1


# ------------------------------------------------- edge cases
def S(name, N, CI, CO, H, W, K, s, p, g=1, i="f16", o="f16", epi="none", dd="uniform", kd="he"):
    return synth.ConvSpec(name, N, CI, CO, H, W, K, s, p, g, i, o, dd, kd, epi)


# ------------------------------------------------- resident weights, nhwc / direct
# Each block keeps one output-channel tile's weights in shared memory and
# streams only pixels; the grid is a whole number of tile groups.
RES_MAIN = [
    (S("rm_direct_64_64", 2, 64, 64, 56, 56, 1, 1, 0), bg.MODE_DIRECT, 0),
    (S("rm_direct_64_256_bf16", 1, 64, 256, 28, 28, 1, 1, 0, i="bf16", o="bf16"), bg.MODE_DIRECT, 0),
    (S("rm_direct_bias_f32", 2, 128, 200, 16, 16, 1, 1, 0, o="f32", epi="bias"), bg.MODE_DIRECT, 64),
    (S("rm_sub_256_512_s2", 2, 256, 512, 28, 28, 1, 2, 0), bg.MODE_SUB, 128),
    (S("rm_nhwc_k3_ci32", 2, 32, 64, 19, 21, 3, 1, 1), bg.MODE_NHWC, 0),
    (S("rm_nhwc_tf32_1x1", 1, 96, 72, 14, 14, 1, 1, 0, i="f32", o="f32"), bg.MODE_NHWC, 0),
    (S("rm_nhwc_exp_ragged", 1, 40, 136, 13, 11, 3, 1, 1, o="f32", epi="bias_exp"), bg.MODE_NHWC, 64),
]


@pytest.mark.parametrize("case", RES_MAIN, ids=lambda c: c[0].name)
def test_umma_resident_weights_main(case):
    spec, mode, bn = case
    opts = {"kind": bg.KIND_UMMA, "mode": mode, "resident_b": 1}
    if bn:
        opts["tile_n"] = bn
    info = check(spec, opts)
    assert info["resident_b"] and info["split"] == 1 and info["grid"] % info["co_tiles"] == 0


@pytest.mark.parametrize("opts", [{"mode": bg.MODE_NHWC, "split_k": 2, "resident_b": 1},
                                  {"mode": bg.MODE_DIRECT, "tile_n": 256, "resident_b": 1}])
def test_resident_weights_main_rejected(opts):
    base = {"kind": bg.KIND_UMMA}
    base.update(opts)
    with pytest.raises(bg.BigemmError) as e:
        # 2048 input channels: 32 K blocks of 32 KB cannot stay resident
        bg.conv2d_nchw_plan_ex(1, 16, 16, 256, 2048, 1, 1, 1, 0, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                               base)
    assert e.value.status == 2


# ------------------------------------------------- how K slices are summed
# fp32 outputs with no epilogue or a bias take the slices' partial tiles as
# atomic adds into the zeroed output (TMA reduce-add boxes, or per-element adds
# where TMA cannot store); other outputs go through the workspace and the
# reduction pass.
SPLIT_SUM = [
    (S("ss_halo_f32_tma_add", 1, 256, 128, 12, 12, 3, 1, 1, i="f32", o="f32"), bg.MODE_HALO, "add"),
    (S("ss_halo_f32_ragged_atomic", 1, 256, 96, 7, 7, 3, 1, 1, i="f32", o="f32"), bg.MODE_HALO, "add"),
    (S("ss_nhwc_bias_f32", 2, 128, 96, 9, 12, 3, 1, 1, o="f32", epi="bias"), bg.MODE_NHWC, "add"),
    (S("ss_nhwc_s2_f32", 1, 256, 64, 14, 14, 3, 2, 1, i="f32", o="f32"), bg.MODE_NHWC, "add"),
    (S("ss_direct_bias_f32", 2, 256, 64, 16, 16, 1, 1, 0, o="f32", epi="bias"), bg.MODE_DIRECT, "add"),
    (S("ss_exp_f32_reduce", 1, 128, 64, 9, 12, 3, 1, 1, o="f32", epi="bias_exp"), bg.MODE_HALO, "reduce"),
    (S("ss_f16_out_reduce", 1, 128, 64, 9, 12, 3, 1, 1), bg.MODE_HALO, "reduce"),
]


@pytest.mark.parametrize("split", [2, 4])
@pytest.mark.parametrize("case", SPLIT_SUM, ids=lambda c: c[0].name)
def test_split_k_sums(case, split):
    spec, mode, how = case
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": mode, "split_k": split})
    assert info["split"] > 1 and info["split_sum"] == how


# 56-byte fp32 output rows under whole-row 14 x 8 boxes: each group of four lanes
# adds a 4-pixel run with one 16-byte vector atomic
@pytest.mark.parametrize("split", [2, 4])
@pytest.mark.parametrize("spec", [
    S("va_nhwc_14_tf32", 1, 256, 96, 14, 14, 3, 1, 1, i="f32", o="f32"),
    S("va_nhwc_14_f16in_bias", 2, 128, 80, 14, 14, 1, 1, 0, o="f32", epi="bias"),
    S("va_nhwc_28_tf32_ragged_co", 1, 128, 72, 28, 28, 3, 1, 1, i="f32", o="f32"),
], ids=lambda s: s.name)
def test_split_k_vector_atomics(spec, split):
    bw = spec.W
    bh = {14: 8, 28: 4}[bw]                    # 112-pixel tiles: whole, 4-aligned lane groups
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_NHWC, "box_w": bw, "box_h": bh,
                        "split_k": split})
    assert info["split"] > 1 and info["split_sum"] == "add" and info["store"] == "direct"



# ------------------------------------------------- halo units of two stacked tiles
# A unit of 32 output rows x 8 columns: two 128-pixel M tiles share every
# weight tile (BN <= 128), accumulators BN TMEM columns apart.
TWO = [
    _H("two_fused_like_exp", 2, 256, 256, 32, 32, 3, 1, o="f32", epi="bias_exp"),
    _H("two_ragged_ci40_co72", 2, 40, 72, 19, 21, 3, 1),
    _H("two_rows_not_whole", 1, 64, 128, 45, 24, 3, 1),
    _H("two_tf32", 1, 64, 128, 34, 16, 3, 1, i="f32", o="f32"),
    _H("two_bf16_pad0", 1, 64, 96, 40, 24, 3, 0, i="bf16", o="bf16"),
]


@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("spec", TWO, ids=lambda s: s.name)
def test_umma_halo_two_tiles(spec, bn):
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO, "box_w": 8, "box_h": 32,
                        "tile_n": bn, "resident_b": -1})
    assert info["amode"] == "halo" and info["box"][:2] == [8, 32] and info["bn"] == bn


def test_umma_halo_two_tiles_stacked_and_split():
    spec = synth.RESNET50_FP16[3].with_batch(3)                  # 512 -> 512 on 7 x 7
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_STACK, "box_w": 8, "box_h": 32,
                        "tile_n": 128, "split_k": 2})
    assert info["pack"] == "stack" and info["box"][:2] == [8, 32] and info["split"] == 2


def test_umma_halo_two_tiles_need_bn_128():
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(1, 32, 32, 256, 64, 3, 3, 1, 1, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                               {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO, "box_w": 8,
                                "box_h": 32, "tile_n": 256})
    assert e.value.status == 2


# ------------------------------------------------- halo with resident weights
# Resident weights need one 64-channel output tile and one 128-byte channel
# block (9 taps x 8 KB beside three halo stages).
RES = [
    synth.RESNET50_FP16[1].with_batch(1),                        # 64 -> 64, 56 x 56
    _H("res_ragged_ci40_co56", 2, 40, 56, 19, 21, 3, 1),
    _H("res_bf16_co48", 1, 64, 48, 17, 18, 3, 1, i="bf16", o="bf16"),
    _H("res_tf32_ci32", 1, 32, 64, 20, 20, 3, 1, i="f32", o="f32"),
    _H("res_exp_f32out", 2, 64, 64, 16, 24, 3, 1, o="f32", epi="bias_exp"),
]


@pytest.mark.parametrize("spec", RES, ids=lambda s: s.name)
def test_umma_halo_resident_weights(spec):
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO, "resident_b": 1})
    assert info["amode"] == "halo" and info["resident_b"] and info["halo_stages"] >= 2


def test_umma_halo_resident_weights_stacked():
    spec = _H("res_stack", 5, 64, 64, 7, 7, 3, 1, o="f32")
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_STACK, "resident_b": 1})
    assert info["resident_b"] and info["pack"] == "stack"


def test_umma_halo_streamed_weights_forced():
    spec = synth.RESNET50_FP16[1].with_batch(1)
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO, "resident_b": -1})
    assert not info["resident_b"]


@pytest.mark.parametrize("shape", [(256, 64, 128), (64, 256, 64)], ids=["two_co_tiles", "too_large"])
def test_resident_weights_rejected_when_they_cannot_stay(shape):
    co, ci, bn = shape
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(1, 16, 16, co, ci, 3, 3, 1, 1, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                               {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO, "tile_n": bn,
                                "resident_b": 1})
    assert e.value.status == 2


# ------------------------------------------------- halo tiles over stacked images
# The pack writes the images one under another with `pad` zero rows between
# them; a 16-row tile then spans several images and the gap rows are the
# padding of both neighbours.  Output rows that fall on a gap are computed
# and dropped.
STACK = [
    synth.RESNET50_FP16[3].with_batch(3),                        # 512 -> 512 on 7 x 7
    _H("stack_7x7_ragged_ci40_co72", 5, 40, 72, 7, 7, 3, 1),
    _H("stack_11x12_f32out_tma_store", 3, 64, 96, 11, 12, 3, 1, o="f32"),   # 12 rows per image
    _H("stack_k5_pad2_6x6_bf16", 4, 32, 64, 6, 6, 5, 2, i="bf16", o="bf16"),
    _H("stack_k3_pad0_9x9", 3, 64, 64, 9, 9, 3, 0),
    _H("stack_tf32_5x5", 3, 48, 64, 5, 5, 3, 1, i="f32", o="f32"),
    _H("stack_exp_7x7", 4, 64, 128, 7, 7, 3, 1, o="f32", epi="bias_exp"),
    _H("stack_one_image", 1, 64, 64, 7, 7, 3, 1),
]


@pytest.mark.parametrize("spec", STACK, ids=lambda s: s.name)
def test_umma_halo_stacked_images(spec):
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_STACK})
    assert info["amode"] == "halo" and info["pack"] == "stack"


@pytest.mark.parametrize("split", [2, 5])
def test_umma_halo_stacked_split_k(split):
    spec = _H("stack_split", 3, 256, 128, 7, 7, 3, 1, o="f32")
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_STACK, "split_k": split})
    assert info["pack"] == "stack" and info["split"] > 1


def test_stacking_rejects_padding_wider_than_the_kernel():
    # pad 3 with a 3x3 kernel: 11 output rows per image, but only 10 stacked rows
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(2, 7, 7, 64, 64, 3, 3, 1, 3, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                               {"kind": bg.KIND_UMMA, "mode": bg.MODE_STACK})
    assert e.value.status == 2


# ------------------------------------------------- pack launches with grouped work
# The whole-plane pack moves several 128-byte channel tiles of an image per
# block when the grid still gives every SM two blocks.  These shapes reach it
# with ragged last groups (a partial channel tile, a group of fewer tiles),
# beside the large-plane form for comparison.
PACK_GROUPS = [
    (_H("pack_groups_7x7_ci200_co76", 160, 200, 76, 7, 7, 3, 1), bg.MODE_STACK),
    (_H("pack_groups_4x4_ci1024_co32", 80, 1024, 32, 4, 4, 3, 1), bg.MODE_STACK),
    (_H("pack_groups_tf32_7x7_ci100_co40", 160, 100, 40, 7, 7, 3, 1, i="f32", o="f32"), bg.MODE_STACK),
    (_H("pack_groups_bf16_6x6_ci136_co20_exp", 160, 136, 20, 6, 6, 3, 1, i="bf16", o="f32", epi="bias_exp"),
     bg.MODE_NHWC),
    (_H("pack_groups_rows_20x20_ci96_co50", 2, 96, 50, 20, 20, 3, 1), bg.MODE_HALO),
]


@pytest.mark.parametrize("case", PACK_GROUPS, ids=lambda c: c[0].name)
def test_pack_groups(case):
    spec, mode = case
    check(spec, {"kind": bg.KIND_UMMA, "mode": mode})


def test_heuristic_stacks_small_images():
    spec = synth.RESNET50_FP16[3].with_batch(2)
    info = check(spec)
    assert info["amode"] == "halo" and info["pack"] == "stack"


# ------------------------------------------------- subsampling pack (strided 1x1)
SUB = [
    synth.RESNET50_FP16[4].with_batch(2),                        # 256 -> 512, 28 x 28, stride 2
    S("sub_s2_13x13_ragged", 3, 40, 72, 13, 13, 1, 2, 0),
    S("sub_s3_tf32", 2, 64, 64, 16, 17, 1, 3, 0, i="f32", o="f32"),
    S("sub_s2_bf16_bias", 2, 128, 96, 14, 14, 1, 2, 0, i="bf16", o="f32", epi="bias"),
    S("sub_s4_one_column", 1, 32, 64, 9, 1, 1, 4, 0),
    # rows of whole 8-byte words: the subsampling whole-plane pack
    S("sub_s2_tf32_words", 2, 48, 64, 20, 12, 1, 2, 0, i="f32", o="f32"),
    S("sub_s3_f16_words", 2, 64, 64, 24, 24, 1, 3, 0),
    S("sub_s2_bf16_ragged_ci100", 1, 100, 64, 32, 32, 1, 2, 0, i="bf16", o="bf16"),
    S("sub_s2_f16_wide_16x40", 2, 64, 96, 16, 40, 1, 2, 0),
]


@pytest.mark.parametrize("spec", SUB, ids=lambda s: s.name)
def test_umma_subsampled_1x1(spec):
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_SUB})
    assert info["amode"] == "nhwc" and info["pack"] == "sub"


def test_subsampled_and_strided_boxes_agree():
    spec = synth.RESNET50_FP16[4].with_batch(1)
    a = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_SUB, "tile_n": 128})
    b = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_NHWC, "tile_n": 128})
    assert a["pack"] == "sub" and b["pack"] == "plain"


def test_subsampling_needs_a_strided_1x1():
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(1, 8, 8, 64, 64, 3, 3, 2, 1, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                               {"kind": bg.KIND_UMMA, "mode": bg.MODE_SUB})
    assert e.value.status == 2


EDGE = [
    S("ragged_13x11_ci24_co40", 2, 24, 40, 13, 11, 3, 1, 1),
    S("ragged_fp32_ci20_co200", 1, 20, 200, 9, 10, 3, 1, 1, i="f32", o="f32"),
    S("first_layer_ci3_k7_s2", 2, 3, 64, 31, 29, 7, 2, 3),
    S("k5_pad2_bf16", 1, 32, 96, 17, 17, 5, 1, 2, i="bf16", o="bf16"),
    S("k1_pad1_border", 1, 16, 32, 6, 6, 1, 1, 1),
    S("stride3_k3", 1, 16, 48, 20, 20, 3, 3, 0),
    S("out_1x1", 2, 64, 64, 3, 3, 3, 1, 0),
    S("tall_kernel_5x1", 1, 16, 32, 12, 9, 5, 1, 0),
    S("bias_exp_f32out", 2, 64, 128, 10, 10, 3, 1, 1, o="f32", epi="bias_exp"),
    S("bias_rsqrt", 1, 32, 64, 8, 8, 3, 1, 1, o="f32", epi="bias_rsqrt", dd="absnormal"),
    S("bias_only_bf16", 1, 32, 64, 8, 8, 3, 1, 1, i="bf16", o="f32", epi="bias"),
    S("f32_in_f16_out", 1, 32, 64, 8, 8, 3, 1, 1, i="f32", o="f16"),
    S("grouped_g2", 1, 16, 32, 9, 9, 3, 1, 1, g=2),
    S("depthwise_k3_ragged", 3, 24, 24, 15, 13, 3, 2, 1, g=24, kd="dw"),
    S("depthwise_k7", 1, 8, 8, 20, 20, 7, 1, 3, g=8, kd="dw"),
    S("many_images_small", 37, 32, 32, 5, 5, 3, 1, 1),
]


@pytest.mark.parametrize("spec", EDGE, ids=lambda s: s.name)
def test_edge_cases(spec):
    check(spec)


@pytest.mark.parametrize("spec", [e for e in EDGE if e.groups == 1][:8], ids=lambda s: s.name)
def test_edge_cases_simt(spec):
    check(spec, {"kind": bg.KIND_SIMT})


# ------------------------------------------------- the div epilogue, 1/(conv + bias)
# Non-negative data and kernels keep every argument well away from zero.
def _R(name, N, CI, CO, H, W, K, s, p, g=1, i="f16", o="f32"):
    return S(name, N, CI, CO, H, W, K, s, p, g=g, i=i, o=o, epi="bias_recip", dd="absnormal",
             kd="absnormal")


RECIP = [
    (_R("recip_halo_f32", 2, 64, 96, 12, 12, 3, 1, 1), {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO}),
    (_R("recip_nhwc_f16", 1, 32, 64, 9, 11, 3, 1, 1, o="f16"), {"kind": bg.KIND_UMMA, "mode": bg.MODE_NHWC}),
    (_R("recip_direct_bf16", 2, 64, 128, 16, 16, 1, 1, 0, i="bf16", o="bf16"),
     {"kind": bg.KIND_UMMA, "mode": bg.MODE_DIRECT}),
    (_R("recip_tf32_split_reduce", 1, 256, 64, 9, 12, 3, 1, 1, i="f32"),
     {"kind": bg.KIND_UMMA, "mode": bg.MODE_NHWC, "split_k": 4}),
    (_R("recip_simt_tiled", 1, 16, 40, 10, 9, 3, 1, 1, i="f32"), {"kind": bg.KIND_SIMT}),
    (_R("recip_depthwise_stream", 2, 16, 16, 14, 16, 3, 1, 1, g=16), None),
    (_R("recip_depthwise_plane_k5", 2, 24, 24, 14, 14, 5, 1, 2, g=24), {"kind": bg.KIND_SIMT, "mode": 4}),
]


@pytest.mark.parametrize("case", RECIP, ids=lambda c: c[0].name)
def test_div_epilogue(case):
    spec, opts = case
    info = check(spec, opts)
    if opts and opts.get("split_k"):
        assert info["split_sum"] == "reduce"


# ------------------------------------------------- im2col tiles: 128 flattened output pixels
# A tile runs across output rows and images (7 x 7 planes: one tile holds parts
# of three images), and each tap's operand is one TMA im2col load whose
# out-of-image reads are zeros.  Cases: tiles spanning images with a partial
# last tile, stride 2 (odd and even input sizes), 5 x 5 and 7 x 7 kernels,
# unpadded and non-square kernels, ragged channels (zero-padded K blocks,
# partial output-channel tiles), bf16, tf32, BN 64 / 128 / 256, resident
# weights, 16 epilogue warps, split K adding into fp32 and through the
# reduction pass, fused epilogues.
IM2COL = [
    (S("i2c_r50_7x7_like", 5, 128, 256, 7, 7, 3, 1, 1), {"tile_n": 256}),
    (S("i2c_14x14_bn64", 2, 64, 64, 14, 14, 3, 1, 1), {"tile_n": 64}),
    (S("i2c_s2_odd", 3, 64, 128, 15, 15, 3, 2, 1, o="f32", epi="bias"), {"tile_n": 128}),
    (S("i2c_s2_even_bf16", 2, 64, 64, 16, 12, 3, 2, 1, i="bf16", o="bf16"), {"tile_n": 64}),
    (S("i2c_k5_ragged_ci", 2, 40, 96, 9, 9, 5, 1, 2, o="f32", epi="bias_exp"), {"tile_n": 128}),
    (S("i2c_k7_s2", 1, 32, 64, 16, 16, 7, 2, 3), {"tile_n": 64}),
    (S("i2c_valid_p0", 2, 64, 64, 10, 10, 3, 1, 0, epi="bias_relu"), {"tile_n": 64}),
    (S("i2c_tf32_split_add", 1, 256, 64, 7, 7, 3, 1, 1, i="f32", o="f32"),
     {"tile_n": 64, "split_k": 8}),
    (S("i2c_split_reduce_f16", 1, 256, 128, 7, 7, 3, 1, 1, epi="bias_rsqrt", dd="absnormal"),
     {"tile_n": 128, "split_k": 4}),
    (S("i2c_resident_e16", 4, 64, 128, 8, 8, 3, 1, 1), {"tile_n": 128, "resident_b": 1, "epi_warps": 16}),
    (S("i2c_recip_bf16", 3, 64, 64, 6, 9, 3, 1, 1, i="bf16", o="f32", epi="bias_recip", dd="absnormal",
       kd="absnormal"), {"tile_n": 64}),
]


@pytest.mark.parametrize("case", IM2COL, ids=lambda c: c[0].name)
def test_im2col_tiles(case):
    spec, opts = case
    info = check(spec, dict({"kind": bg.KIND_UMMA, "mode": bg.MODE_IM2COL}, **opts))
    assert info["cand"].startswith("umma:nhwc:") and ":im2col" in info["cand"]
    assert info["pack"] == "im2col"


def test_im2col_non_square_kernel():
    # 3 x 5 kernel, pad 1: the corners differ per spatial dimension
    spec = S("i2c_3x5", 2, 32, 64, 9, 11, 3, 1, 1)
    x, _, _ = synth.conv_inputs(spec, 3)
    # the spec helper draws square kernels: the 3 x 5 kernel is drawn here
    g = torch.Generator().manual_seed(7)
    w35 = (torch.randn(64, 32, 3, 5, generator=g) * 0.1).to(torch.float16)
    xd, wd = x.cuda(), w35.cuda()
    Ho, Wo = 9, 11 + 2 - 5 + 1
    out = torch.empty(2, 64, Ho, Wo, dtype=torch.float16, device="cuda")
    plan = bg.conv2d_nchw_plan_ex(2, 9, 11, 64, 32, 3, 5, 1, 1, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                                  {"kind": bg.KIND_UMMA, "mode": bg.MODE_IM2COL, "tile_n": 64})
    bg.conv2d_nchw_run(plan, xd, wd, None, 1e-5, out)
    torch.cuda.synchronize()
    assert plan.describe()["pack"] == "im2col"
    plan.close()
    ref, sabs = oracle.conv2d_nchw(x, w35, stride=1, pad=1, nthreads=NTH)
    assert_within(out.cpu().double().numpy(), ref, conv_bound(ref, sabs, TAU["half"], "f16"), "im2col 3x5")


def test_im2col_rejects_1x1_and_stride_3():
    x = torch.empty(16, dtype=torch.float16, device="cuda")
    for K, st in ((1, 1), (3, 3)):
        with pytest.raises(bg.BigemmError) as e:
            bg.conv2d_nchw_plan_ex(1, 12, 12, 64, 64, K, K, st, K // 2, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                                   {"kind": bg.KIND_UMMA, "mode": bg.MODE_IM2COL})
        assert e.value.status == 2


# ------------------------------------------------- add + ReLU, max(conv + bias, 0)
# Data and kernels of both signs, so about half of the outputs clamp to zero.
def _U(name, N, CI, CO, H, W, K, s, p, g=1, i="f16", o="f32", kd="he"):
    return S(name, N, CI, CO, H, W, K, s, p, g=g, i=i, o=o, epi="bias_relu", kd=kd)


RELU = [
    (_U("relu_halo_f32", 2, 64, 96, 12, 12, 3, 1, 1), {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO}),
    (_U("relu_nhwc_f16", 1, 32, 64, 9, 11, 3, 1, 1, o="f16"), {"kind": bg.KIND_UMMA, "mode": bg.MODE_NHWC}),
    (_U("relu_direct_bf16", 2, 64, 128, 16, 16, 1, 1, 0, i="bf16", o="bf16"),
     {"kind": bg.KIND_UMMA, "mode": bg.MODE_DIRECT}),
    (_U("relu_strided_f16", 2, 64, 128, 12, 16, 1, 2, 0, o="f16"),
     {"kind": bg.KIND_UMMA, "mode": bg.MODE_STRIDED}),
    (_U("relu_tf32_split_reduce", 1, 256, 64, 9, 12, 3, 1, 1, i="f32"),
     {"kind": bg.KIND_UMMA, "mode": bg.MODE_NHWC, "split_k": 4}),
    (_U("relu_simt_tiled", 1, 16, 40, 10, 9, 3, 1, 1, i="f32"), {"kind": bg.KIND_SIMT}),
    (_U("relu_depthwise_stream", 2, 16, 16, 14, 16, 3, 1, 1, g=16, kd="dw"), None),
    (_U("relu_depthwise_plane_k5", 2, 24, 24, 14, 14, 5, 1, 2, g=24, kd="dw"), {"kind": bg.KIND_SIMT, "mode": 4}),
    (_U("relu_depthwise_band", 2, 16, 16, 13, 15, 3, 2, 1, g=16, kd="dw"), {"kind": bg.KIND_SIMT, "mode": 2, "box_h": 4}),
]


@pytest.mark.parametrize("case", RELU, ids=lambda c: c[0].name)
def test_relu_epilogue(case):
    spec, opts = case
    info = check(spec, opts)
    if opts and opts.get("split_k"):
        assert info["split_sum"] == "reduce"


# ------------------------------------------------- depthwise kernels
DW = [
    S("dws_k3s1_f16_w16", 2, 24, 24, 21, 16, 3, 1, 1, g=24, kd="dw"),
    S("dws_k3s1_f16_ragged_w", 2, 16, 16, 19, 13, 3, 1, 1, g=16, kd="dw"),
    S("dws_k3s2_bf16", 3, 40, 40, 23, 24, 3, 2, 1, g=40, i="bf16", o="bf16", kd="dw"),
    S("dws_k5s1_f16_14", 2, 48, 48, 14, 14, 5, 1, 2, g=48, kd="dw"),
    S("dws_k5s2_f32", 2, 8, 8, 17, 20, 5, 2, 2, g=8, i="f32", o="f32", kd="dw"),
    S("dws_k7s1_f16", 1, 8, 8, 30, 32, 7, 1, 3, g=8, kd="dw"),
    S("dws_k7s2_f32out", 1, 8, 8, 29, 29, 7, 2, 3, g=8, o="f32", kd="dw"),
    S("dws_k3s1_f32_bias_exp", 2, 16, 16, 12, 12, 3, 1, 1, g=16, i="f32", o="f32", epi="bias_exp", kd="dw"),
    S("dws_k3s1_rsqrt", 1, 16, 16, 16, 16, 3, 1, 1, g=16, o="f32", epi="bias_rsqrt", dd="absnormal", kd="dw"),
    S("dws_one_row", 2, 8, 8, 1, 40, 3, 1, 1, g=8, kd="dw"),
    S("dws_k3s1_f32_w10_words", 2, 8, 8, 9, 10, 3, 1, 1, g=8, i="f32", o="f32", kd="dw"),
    S("dws_k3s2_f16_w18_words", 2, 8, 8, 11, 18, 3, 2, 1, g=8, kd="dw"),
]


@pytest.mark.parametrize("spec", DW, ids=lambda s: s.name)
def test_depthwise_heuristic(spec):
    info = check(spec)
    # stride 1 with outputs at most 16 wide and 32 tall: the small-plane kernel
    if spec.stride == 1 and spec.W <= 16 and spec.H <= 32:
        assert info["cand"] == f"simt:depthwise:small{4 if spec.H > 8 else 2}"
    else:
        assert info["cand"].startswith("simt:depthwise:stream")


@pytest.mark.parametrize("rows", [2, 4, 8])
@pytest.mark.parametrize("spec", [DW[0], DW[2], DW[4], DW[10]], ids=lambda s: s.name)
def test_depthwise_streaming_rows(spec, rows):
    info = check(spec, {"kind": bg.KIND_SIMT, "mode": 3, "box_h": rows})
    assert info["cand"].startswith("simt:depthwise:stream")


@pytest.mark.parametrize("spec", DW[:5], ids=lambda s: s.name)
def test_depthwise_staged_band(spec):
    info = check(spec, {"kind": bg.KIND_SIMT, "mode": 2, "box_h": 4})
    assert info["cand"] == "simt:depthwise:rows4"


# Whole planes per warp (H, W <= 32): two planes per warp for outputs up to
# 16 wide, one above; an odd plane count leaves the last warp one plane.
DW_PLANE = [x for x in DW if x.H <= 32 and x.W <= 32] + [
    S("dwp_odd_planes_k3", 1, 7, 7, 14, 14, 3, 1, 1, g=7, kd="dw"),
    S("dwp_k5_576_like", 2, 24, 24, 14, 14, 5, 1, 2, g=24, kd="dw"),
    S("dwp_k3s2_32wide", 1, 12, 12, 32, 32, 3, 2, 1, g=12, o="f32", epi="bias", kd="dw"),
]


@pytest.mark.parametrize("spec", DW_PLANE, ids=lambda s: s.name)
def test_depthwise_whole_planes(spec):
    info = check(spec, {"kind": bg.KIND_SIMT, "mode": 4})
    assert info["cand"] == "simt:depthwise:plane"


# Small planes (stride 1, outputs at most 16 wide and 32 tall), 2 x 8 or 4 x 8
# outputs per thread: several planes per warp (up to sixteen for 7 x 7), one
# plane per warp at 16 x 32, ragged column and row blocks, plane counts that
# leave the last warp short, element counts that rule out the 16-byte staging
# and output copies, each dtype and epilogue, an fp32 output from 16-bit
# inputs, K = 3, 5, 7 (a 7x7 over a 1-row image reads only border rows).
DW_SMALL = [
    S("dwr_k5_576_like", 2, 24, 24, 14, 14, 5, 1, 2, g=24, kd="dw"),
    S("dwr_k3_7x7_odd_planes", 1, 7, 7, 7, 7, 3, 1, 1, g=7, kd="dw"),
    S("dwr_k3_bf16_ragged", 3, 40, 40, 11, 13, 3, 1, 1, g=40, i="bf16", o="bf16", kd="dw"),
    S("dwr_k7_f32_16x32", 2, 6, 6, 32, 16, 7, 1, 3, g=6, i="f32", o="f32", kd="dw"),
    S("dwr_k5_f16_bias_exp", 2, 16, 16, 9, 12, 5, 1, 2, g=16, o="f32", epi="bias_exp", kd="dw"),
    S("dwr_k3_rsqrt", 1, 16, 16, 16, 16, 3, 1, 1, g=16, o="f32", epi="bias_rsqrt", dd="absnormal",
      kd="dw"),
    S("dwr_k3_recip", 2, 12, 12, 5, 6, 3, 1, 1, g=12, epi="bias_recip", dd="absnormal",
      kd="absnormal"),
    S("dwr_k7_relu_bf16", 1, 10, 10, 12, 15, 7, 1, 3, g=10, i="bf16", o="bf16", epi="bias_relu",
      kd="dw"),
    S("dwr_k7_one_row", 2, 8, 8, 1, 9, 7, 1, 3, g=8, kd="dw"),
    S("dwr_k5_f32_bias_3x3", 3, 9, 9, 3, 3, 5, 1, 2, g=9, i="f32", o="f32", epi="bias", kd="dw"),
]


@pytest.mark.parametrize("ty", [2, 4])
@pytest.mark.parametrize("spec", DW_SMALL, ids=lambda s: s.name)
def test_depthwise_small_planes(spec, ty):
    info = check(spec, {"kind": bg.KIND_SIMT, "mode": 5, "box_h": ty})
    assert info["cand"] == f"simt:depthwise:small{ty}"


@pytest.mark.parametrize("shape", [(14, 17, 3, 1), (33, 8, 3, 1), (14, 14, 3, 2), (14, 14, 4, 1)])
def test_depthwise_small_planes_rejects_other_shapes(shape):
    H, W, K, stride = shape
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(1, H, W, 8, 8, K, K, stride, K // 2, 8, bg.F16, bg.F16,
                               bg.EPI_NONE, 0, {"kind": bg.KIND_SIMT, "mode": 5})
    assert e.value.status == 2


# Bands of rows (input rows of 16-byte chunks up to 512 bytes), 4 x 8 outputs
# per thread, stride 1 and 2: the workload's 112- and 56-wide layers at N = 2,
# several bands per plane with a ragged last band, rows whose width is not a
# multiple of 8 outputs (scalar stores), one row block per warp (32 column
# blocks), fp32 and bf16, fp32 output from 16-bit input, each epilogue, K = 5
# and 7, a stride-2 layer with an odd input height.
DW_BAND = [
    S("dwb_32_112_k3", 2, 32, 32, 112, 112, 3, 1, 1, g=32, kd="dw"),
    S("dwb_96_112_k3s2", 2, 96, 96, 112, 112, 3, 2, 1, g=96, kd="dw"),
    S("dwb_144_56_k3", 2, 16, 16, 56, 56, 3, 1, 1, g=16, kd="dw"),
    S("dwb_ragged_rows_k5", 3, 8, 8, 37, 24, 5, 1, 2, g=8, kd="dw", epi="bias"),
    S("dwb_wide_256_k3_bf16", 1, 4, 4, 9, 256, 3, 1, 1, g=4, i="bf16", o="bf16", kd="dw"),
    S("dwb_f32_k7_s2", 2, 6, 6, 29, 64, 7, 2, 3, g=6, i="f32", o="f32", kd="dw"),
    S("dwb_f32_k3_exp", 2, 8, 8, 20, 20, 3, 1, 1, g=8, i="f32", o="f32", epi="bias_exp", kd="dw"),
    S("dwb_rsqrt_f32out", 1, 16, 16, 16, 40, 3, 1, 1, g=16, o="f32", epi="bias_rsqrt",
      dd="absnormal", kd="dw"),
    S("dwb_recip_s2_odd_h", 2, 8, 8, 31, 48, 3, 2, 1, g=8, epi="bias_recip", dd="absnormal",
      kd="absnormal"),
    S("dwb_relu_k7", 1, 12, 12, 21, 72, 7, 1, 3, g=12, i="bf16", o="bf16", epi="bias_relu",
      kd="dw"),
    S("dwb_k5_s2_w24", 2, 10, 10, 24, 24, 5, 2, 2, g=10, kd="dw"),
]


@pytest.mark.parametrize("spec", DW_BAND, ids=lambda s: s.name)
def test_depthwise_bands(spec):
    info = check(spec, {"kind": bg.KIND_SIMT, "mode": 6})
    assert info["cand"] == "simt:depthwise:band"


@pytest.mark.parametrize("shape", [(16, 20, 3, 1, "f16"), (8, 264, 3, 1, "f16"), (8, 16, 3, 3, "f16"),
                                   (8, 130, 3, 1, "f32")])
def test_depthwise_bands_reject_other_shapes(shape):
    H, W, K, stride, dt = shape
    d = {"f16": bg.F16, "f32": bg.F32}[dt]
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(1, H, W, 8, 8, K, K, stride, K // 2, 8, d, d, bg.EPI_NONE, 0,
                               {"kind": bg.KIND_SIMT, "mode": 6})
    assert e.value.status == 2


def test_depthwise_small_planes_rejects_other_block_heights():
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(1, 14, 14, 8, 8, 3, 3, 1, 1, 8, bg.F16, bg.F16, bg.EPI_NONE, 0,
                               {"kind": bg.KIND_SIMT, "mode": 5, "box_h": 3})
    assert e.value.status == 1


def test_depthwise_whole_planes_rejects_wide_rows():
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(1, 8, 40, 8, 8, 3, 3, 1, 1, 8, bg.F16, bg.F16, bg.EPI_NONE, 0,
                               {"kind": bg.KIND_SIMT, "mode": 4})
    assert e.value.status == 2


# ------------------------------------------------- strided mode: stride-2 1x1 read in place
# The data is read as rows of 2W elements (an even input row and the odd one
# below it); warps of the kernel keep the even pixels.  Cases: the ResNet-50
# downsampling layer at N = 2, several column boxes per row (Wo > 16), rows
# TMA can store (Wo = 16), bf16, ragged channels, BN 64 / 128 / 256, split K
# (adding into fp32, and through the reduction pass), fused epilogues, an
# image narrower than 16 columns.
STRIDED = [
    (S("str_r50_like", 2, 256, 512, 28, 28, 1, 2, 0), {}),
    (S("str_w32_ragged_h", 1, 64, 128, 22, 32, 1, 2, 0), {"tile_n": 128}),
    (S("str_wide_rows_56", 1, 64, 128, 56, 56, 1, 2, 0), {}),
    (S("str_tma_rows_32", 2, 64, 64, 32, 32, 1, 2, 0), {}),
    (S("str_bf16_ragged", 3, 40, 72, 12, 20, 1, 2, 0, i="bf16", o="bf16"), {}),
    (S("str_tiny", 2, 16, 16, 2, 4, 1, 2, 0), {}),
    (S("str_bn64_exp", 2, 128, 96, 14, 28, 1, 2, 0, o="f32", epi="bias_exp"), {"tile_n": 64}),
    (S("str_bn256_bias_f16", 1, 64, 256, 18, 12, 1, 2, 0, epi="bias"), {"tile_n": 256}),
    (S("str_split_add_f32", 1, 512, 128, 14, 16, 1, 2, 0, o="f32", epi="bias"), {"split_k": 4}),
    (S("str_split_reduce_recip", 1, 256, 64, 10, 16, 1, 2, 0, o="f16", epi="bias_recip",
       dd="absnormal", kd="absnormal"), {"split_k": 2}),
]


@pytest.mark.parametrize("case", STRIDED, ids=lambda c: c[0].name)
def test_umma_strided_mode(case):
    spec, extra = case
    info = check(spec, dict({"kind": bg.KIND_UMMA, "mode": bg.MODE_STRIDED}, **extra))
    # one launch and no scratch, unless K slices go through the reduction pass
    assert info["amode"] == "strided"
    if info["split_sum"] != "reduce":
        assert info["launches"] == 1 and info["scratch_bytes"] == 0


def test_strided_and_subsampled_agree():
    spec = S("str_vs_sub", 2, 128, 256, 28, 28, 1, 2, 0)
    a = run(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_STRIDED})[-1]
    b = run(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_SUB})[-1]
    # both fp32-accumulated sums of the same fp16 products, rounded to fp16
    assert torch.allclose(a.float(), b.float(), rtol=2e-3, atol=2e-3)


@pytest.mark.parametrize("shape,dt", [((1, 8, 16, 64, 64), bg.F32),    # tf32: K-major only
                                      ((1, 9, 16, 64, 64), bg.F16),    # odd H
                                      ((1, 8, 6, 64, 64), bg.F16),     # 2W*2 = 24 bytes
                                      ((1, 8, 16, 64, 60), bg.F16)])   # CI*2 = 120 bytes
def test_strided_mode_rejected(shape, dt):
    N, H, W, CO, CI = shape
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(N, H, W, CO, CI, 1, 1, 2, 0, 1, dt, dt, bg.EPI_NONE, 0,
                               {"kind": bg.KIND_UMMA, "mode": bg.MODE_STRIDED})
    assert e.value.status == 2


# ------------------------------------------------- CTA pairs: two blocks share each MMA
# tcgen05 cta_group::2 (M = 256): each block of a cluster pair loads its own
# 16 x 8 halo tile and half of the resident weights; the even block issues the
# pair's MMAs.  Cases: the ResNet-50 64 -> 64 3x3 layer at N = 2, an odd tile
# count (the odd block's last tile is past the output), stacked images, bf16,
# tf32, a 5x5 kernel, ragged CO, BN = 128, fused exp into fp32.
PAIR = [
    S("pair_r50_like", 2, 64, 64, 56, 56, 3, 1, 1),
    S("pair_odd_tiles", 1, 64, 64, 40, 8, 3, 1, 1),
    S("pair_bf16_ragged_co", 2, 40, 48, 20, 24, 3, 1, 1, i="bf16", o="bf16"),
    S("pair_tf32", 1, 32, 64, 18, 16, 3, 1, 1, i="f32", o="f32"),
    S("pair_k5", 1, 64, 64, 24, 16, 5, 1, 2),
    S("pair_bn128_exp", 2, 64, 128, 16, 24, 3, 1, 1, o="f32", epi="bias_exp"),
]


@pytest.mark.parametrize("stack", [False, True])
@pytest.mark.parametrize("spec", PAIR, ids=lambda s: s.name)
def test_umma_halo_cta_pair(spec, stack):
    opts = {"kind": bg.KIND_UMMA, "mode": bg.MODE_STACK if stack else bg.MODE_HALO,
            "resident_b": 1, "cta_pair": 1, "tile_n": 64 if spec.CO <= 64 else 128}
    info = check(spec, opts)
    assert info["cta_pair"] and info["grid"] % 2 == 0


def test_cta_pair_and_single_block_agree():
    spec = S("pair_vs_single", 2, 64, 64, 28, 28, 3, 1, 1)
    base = {"kind": bg.KIND_UMMA, "mode": bg.MODE_HALO, "resident_b": 1, "tile_n": 64}
    a = run(spec, dict(base, cta_pair=1))[-1]
    b = run(spec, dict(base, cta_pair=-1))[-1]
    # the same fp32 sums of the same fp16 products, in the same order
    assert torch.equal(a, b)


@pytest.mark.parametrize("opts", [{"mode": bg.MODE_HALO, "resident_b": -1, "cta_pair": 1},    # streamed weights
                                  {"mode": bg.MODE_NHWC, "cta_pair": 1},                       # not the halo mode
                                  {"mode": bg.MODE_HALO, "resident_b": 1, "cta_pair": 1, "split_k": 2}])
def test_cta_pair_rejected(opts):
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(1, 16, 16, 64, 64, 3, 3, 1, 1, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                               dict({"kind": bg.KIND_UMMA, "tile_n": 64}, **opts))
    assert e.value.status == 2


# ------------------------------------------------- full size, sampled outputs
FULL = synth.RESNET50_FP16 + synth.FUSED_CONV + synth.DEPTHWISE_FP16


@pytest.mark.parametrize("spec", FULL, ids=lambda s: s.name)
def test_full_size_sampled(spec):
    info, x, w, b, out = run(spec)
    total = out.numel()
    idx = synth.random_flat_indices(total, 3000, seed=5)
    # plus every border pixel of two planes
    Ho, Wo = out.shape[2], out.shape[3]
    planes = [0, total // (Ho * Wo) - 1]
    border = [pl * Ho * Wo + y * Wo + xx for pl in planes for y in range(Ho) for xx in range(Wo)
              if y in (0, Ho - 1) or xx in (0, Wo - 1)]
    idx = torch.unique(torch.cat([idx, torch.tensor(border, dtype=torch.int64)])).numpy()
    got = out.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().double().numpy()
    tau = tau_for(spec, info)
    if spec.epi == "none":
        ref, sabs = oracle.conv2d_nchw_points(x, w, idx, stride=spec.stride, pad=spec.pad,
                                              groups=spec.groups)
        bound = conv_bound(ref, sabs, tau, spec.out_dtype)
    else:
        ref, sabs = oracle.conv2d_nchw_points(x, w, idx, stride=spec.stride, pad=spec.pad,
                                              groups=spec.groups, bias=b, epi=oracle.EPI_BIAS_EXP)
        pre, _ = oracle.conv2d_nchw_points(x, w, idx, stride=spec.stride, pad=spec.pad,
                                           groups=spec.groups)
        f = (idx // (Ho * Wo)) % spec.CO
        arg = pre + b.double().numpy()[f]
        bound = epi_bound(arg, sabs, tau, spec.epi, spec.out_dtype, ref)
    assert_within(got, ref, bound, f"{spec.name} [{info['cand']}]")
    assert not torch.isnan(out).any()


# ------------------------------------------------- plan search and cache
def test_search_picks_a_timed_candidate_and_caches_it():
    spec = S("search_small", 2, 64, 64, 14, 14, 3, 1, 1)
    info = check(spec, search=1)
    assert info["chosen_by"] in ("search", "cache")
    if info["chosen_by"] == "search":
        recs = info["search"]
        assert len(recs) >= 3
        ok = [r for r in recs if r["status"] == 0]
        chosen = [r["ms"] for r in ok if r["cand"] == info["cand"]]
        assert chosen and min(chosen) == min(r["ms"] for r in ok)
    again = bg.conv2d_nchw_plan(spec.N, spec.H, spec.W, spec.CO, spec.CI, 3, 3, 1, 1, 1,
                                bg.F16, bg.F16, bg.EPI_NONE, 1)
    d = again.describe()
    assert d["chosen_by"] == "cache" and d["cand"] == info["cand"]
    again.close()


_PLAN_LOG_CHILD = """
import sys
sys.path.insert(0, {root!r})
import broadcast_implicit_gemm_gb300 as bg
p = bg.conv2d_nchw_plan(2, 13, 15, 72, 48, 3, 3, 1, 1, 1, bg.F16, bg.F32, bg.EPI_BIAS, 1)
d = p.describe()
print("PLAN", d["chosen_by"], d["cand"])
"""


def _plan_in_fresh_process(log_path):
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, BIGEMM_PLAN_CACHE=str(log_path))
    r = subprocess.run([sys.executable, "-c", _PLAN_LOG_CHILD.format(root=root)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("PLAN ")][-1]
    return line.split()[1:]


def test_plan_log_round_trip(tmp_path):
    # The tuning-log flow: a search writes its best record to the JSONL log
    # (BIGEMM_PLAN_CACHE); a later process with the same log takes the plan
    # from it without searching.
    log = tmp_path / "plans.jsonl"
    chosen_by, cand = _plan_in_fresh_process(log)
    assert chosen_by == "search"
    lines = log.read_text().splitlines()
    assert len(lines) == 1 and f'"cand": "{cand}"' in lines[0] and "|N2|H13|W15|CO72|CI48|" in lines[0]
    assert _plan_in_fresh_process(log) == ["cache", cand]
    assert len(log.read_text().splitlines()) == 1      # a cache hit appends nothing


def test_forced_invalid_tiling_is_rejected_before_launch():
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(1, 8, 8, 64, 64, 3, 3, 1, 1, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                               {"kind": bg.KIND_UMMA, "tile_n": 96})
    assert e.value.status == 2


def test_misaligned_pointer_rejected():
    plan = bg.conv2d_nchw_plan(1, 8, 8, 64, 64, 3, 3, 1, 1, 1, bg.F16, bg.F16, bg.EPI_NONE, 0)
    x = torch.zeros(1 * 64 * 8 * 8 + 1, dtype=torch.float16, device="cuda")
    w = torch.zeros(64 * 64 * 9, dtype=torch.float16, device="cuda")
    o = torch.zeros(64 * 64, dtype=torch.float16, device="cuda")
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_run(plan, x.data_ptr() + 2, w, None, 0.0, o)
    assert e.value.status == 1
    plan.close()


# ------------------------------------------------- 16 epilogue warps
# 128-channel tiles drained by four warps per TMEM lane quadrant (one 32-channel
# chunk each, 2 KB of staging each) instead of two.
EPI16 = [
    (S("e16_direct_64_256", 2, 64, 256, 28, 28, 1, 1, 0), bg.MODE_DIRECT, 0, 1),
    (S("e16_direct_ragged_co200_bias_f32", 1, 128, 200, 16, 16, 1, 1, 0, o="f32", epi="bias"),
     bg.MODE_DIRECT, 0, 1),
    (S("e16_nhwc_k3_exp_f32", 1, 64, 136, 13, 11, 3, 1, 1, o="f32", epi="bias_exp"), bg.MODE_NHWC, 0, 1),
    # non-negative data and kernel keep every rsqrt argument well above zero
    (S("e16_nhwc_tf32_rsqrt", 1, 96, 128, 9, 12, 3, 1, 1, i="f32", o="f32", epi="bias_rsqrt",
       dd="absnormal", kd="absnormal"), bg.MODE_NHWC, -1, 1),
    (S("e16_sub_s2_bf16", 2, 256, 256, 28, 28, 1, 2, 0, i="bf16", o="bf16"), bg.MODE_SUB, 1, 1),
    (S("e16_nhwc_split_add_f32", 1, 256, 128, 14, 14, 3, 1, 1, i="f32", o="f32"), bg.MODE_NHWC, -1, 4),
    (S("e16_nhwc_split_reduce_f16", 1, 256, 128, 12, 12, 3, 1, 1), bg.MODE_NHWC, -1, 2),
]


# each case with streamed weights, and with resident weights where they can stay
# (split 1 and a tile's weights within shared memory)
EPI16_RUNS = [(c, r) for c in EPI16 for r in ((0, 1) if c[2] != -1 else (0,))]


@pytest.mark.parametrize("case,resident", EPI16_RUNS,
                         ids=lambda v: v[0].name if isinstance(v, tuple) else f"res{v}")
def test_sixteen_epilogue_warps(case, resident):
    spec, mode, res, split = case
    opts = {"kind": bg.KIND_UMMA, "mode": mode, "tile_n": 128, "split_k": split, "epi_warps": 16,
            "resident_b": 1 if resident else -1}
    info = check(spec, opts)
    assert info["epi_warps"] == 16 and info["bn"] == 128 and info["resident_b"] == bool(resident)


def test_eight_epilogue_warps_on_request():
    spec = S("e8_direct_64_256", 1, 64, 256, 28, 28, 1, 1, 0)
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": bg.MODE_DIRECT, "tile_n": 128, "epi_warps": 8})
    assert info["epi_warps"] == 8


# 64-channel tiles with 16 epilogue warps: two groups of eight take alternate
# units (and accumulators); an odd unit count per block leaves group 1 a unit
# short.  Direct and per-tap modes, resident and streamed weights, split K
# adding into fp32, 16-bit register stores, fused epilogues.
EPI16_64 = [
    (S("e16g_direct_64_64_56", 2, 64, 64, 56, 56, 1, 1, 0), bg.MODE_DIRECT, 1, 1),
    (S("e16g_direct_ragged_co40_exp", 1, 64, 40, 20, 28, 1, 1, 0, o="f32", epi="bias_exp"),
     bg.MODE_DIRECT, -1, 1),
    (S("e16g_nhwc_k3_relu_bf16", 2, 48, 64, 13, 11, 3, 1, 1, i="bf16", o="bf16", epi="bias_relu"),
     bg.MODE_NHWC, -1, 1),
    (S("e16g_nhwc_tf32_split_add", 1, 256, 64, 14, 14, 3, 1, 1, i="f32", o="f32"), bg.MODE_NHWC, -1, 8),
    (S("e16g_nhwc_regstores_14", 2, 64, 64, 14, 14, 1, 1, 0), bg.MODE_NHWC, 1, 1),
    (S("e16g_sub_s2", 2, 128, 64, 28, 28, 1, 2, 0), bg.MODE_SUB, 1, 1),
]


@pytest.mark.parametrize("case", EPI16_64, ids=lambda c: c[0].name)
def test_sixteen_epilogue_warps_64_channel_tiles(case):
    spec, mode, res, split = case
    opts = {"kind": bg.KIND_UMMA, "mode": mode, "tile_n": 64, "split_k": split, "epi_warps": 16,
            "resident_b": res}
    info = check(spec, opts)
    assert info["epi_warps"] == 16 and info["bn"] == 64


@pytest.mark.parametrize("opts,status", [
    ({"kind": 1, "mode": bg.MODE_DIRECT, "tile_n": 256, "epi_warps": 16}, 2),
    ({"kind": 1, "mode": bg.MODE_HALO, "tile_n": 128, "epi_warps": 16}, 2),
    ({"kind": 1, "mode": bg.MODE_DIRECT, "tile_n": 128, "epi_warps": 12}, 1),
])
def test_sixteen_epilogue_warps_rejected(opts, status):
    k = 3 if opts["mode"] == bg.MODE_HALO else 1
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_plan_ex(1, 16, 16, 256, 64, k, k, 1, k // 2, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                               opts)
    assert e.value.status == status


# ------------------------------------------------- stores from registers
# Outputs whose rows no TMA box can address (Wo x element size not a multiple
# of 16 bytes) leave the epilogue from registers: as 4-pixel runs where each
# group of four lanes holds four consecutive pixels of a plane at a 4-element
# boundary (or none at all), as single elements otherwise.
REG_STORE = [
    (S("rs_sub_14_f16_bn128", 2, 256, 256, 28, 28, 1, 2, 0), bg.MODE_SUB, 128),
    (S("rs_nhwc_14_f16_ragged_co", 2, 96, 136, 14, 14, 1, 1, 0), bg.MODE_NHWC, 64),
    (S("rs_nhwc_14_bf16_bn256", 1, 64, 256, 14, 14, 1, 1, 0, i="bf16", o="bf16"), bg.MODE_NHWC, 256),
    (S("rs_halo_28_bf16", 1, 64, 72, 28, 28, 3, 1, 1, i="bf16", o="bf16"), bg.MODE_HALO, 64),
    (S("rs_nhwc_14_f32_bias", 1, 64, 80, 14, 14, 3, 1, 1, i="f32", o="f32", epi="bias"), bg.MODE_NHWC, 64),
    (S("rs_halo_10x6_f32_exp", 2, 32, 48, 10, 6, 3, 1, 1, o="f32", epi="bias_exp"), bg.MODE_HALO, 64),
    (S("rs_halo_7_f16_elements", 2, 64, 64, 7, 7, 3, 1, 1), bg.MODE_HALO, 64),
    (S("rs_nhwc_9x5_f16_elements", 1, 32, 40, 9, 5, 3, 1, 1), bg.MODE_NHWC, 64),
]


@pytest.mark.parametrize("case", REG_STORE, ids=lambda c: c[0].name)
def test_register_stores(case):
    spec, mode, bn = case
    info = check(spec, {"kind": bg.KIND_UMMA, "mode": mode, "tile_n": bn, "split_k": 1})
    assert info["store"] == "direct" and info["split"] == 1


@pytest.mark.parametrize("spec", [S("rs_forced_direct_56", 1, 64, 64, 56, 56, 1, 1, 0),
                                  S("rs_forced_halo_16", 2, 64, 96, 16, 16, 3, 1, 1, o="f32")],
                         ids=lambda s: s.name)
def test_register_stores_forced(spec, monkeypatch):
    # rows TMA could store, written from registers instead
    monkeypatch.setenv("BIGEMM_NO_TMA_STORE", "1")
    info = check(spec, {"kind": bg.KIND_UMMA, "split_k": 1})
    assert info["store"] == "direct"


def test_misaligned_output_rejected():
    # outputs must start on a 16-byte boundary: one 2 bytes past it is refused
    # before any launch, and nothing is written
    plan = bg.conv2d_nchw_plan_ex(1, 14, 14, 72, 64, 1, 1, 1, 0, 1, bg.F16, bg.F16, bg.EPI_NONE, 0,
                                  {"kind": bg.KIND_UMMA, "mode": bg.MODE_NHWC, "split_k": 1})
    x = torch.zeros((1, 64, 14, 14), dtype=torch.float16, device="cuda")
    w = torch.zeros((72, 64, 1, 1), dtype=torch.float16, device="cuda")
    n = 72 * 14 * 14
    buf = torch.full((n + 1,), SENTINEL, dtype=torch.float16, device="cuda")
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_run(plan, x, w, None, 0.0, buf[1:].view(1, 72, 14, 14))
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert bool(torch.all(buf.float().cpu() == SENTINEL))
    plan.close()


def test_missing_bias_rejected():
    plan = bg.conv2d_nchw_plan(1, 8, 8, 64, 64, 3, 3, 1, 1, 1, bg.F16, bg.F32, bg.EPI_BIAS_EXP, 0)
    x = torch.zeros((1, 64, 8, 8), dtype=torch.float16, device="cuda")
    w = torch.zeros((64, 64, 3, 3), dtype=torch.float16, device="cuda")
    o = torch.zeros((1, 64, 8, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(bg.BigemmError) as e:
        bg.conv2d_nchw_run(plan, x, w, None, 0.0, o)
    assert e.value.status == 1
    plan.close()


def test_bounded_wait_reports_timeout_without_fault():
    bg.bigemm_clear_device_error()
    bg.bigemm_debug_wait_timeout(2_000_000)      # 2 ms on a barrier nothing completes
    assert bg.bigemm_last_device_error() == 4
    bg.bigemm_clear_device_error()
    assert bg.bigemm_last_device_error() == 0
    # the context is still usable
    check(S("after_timeout", 1, 16, 32, 8, 8, 3, 1, 1))


def test_profile_records_kernel_launches():
    spec = synth.RESNET50_FP16[1].with_batch(1)
    bg.bigemm_profile_enable(True)
    run(spec)
    rec = bg.bigemm_profile_read()
    bg.bigemm_profile_enable(False)
    assert any(k.startswith("umma_conv") for k in rec)
    assert all(v[0] >= 1 and v[1] > 0 for v in rec.values())
