"""Parity of the plans the benchmark runs, at the benchmark's sizes and inputs.

For every layer of every benchmark workload this runs the timed plan search on
the same shape, batch and seeded inputs as bench.py, so the plan it picks is
the one the benchmark would pick.  The search can rank near-equal candidates
differently from run to run, so the test then forces every candidate the search
timed successfully (by its description: operand mode, tile, pixel boxes,
split-K, resident weights, epilogue warps) and checks that each, too, matches
the oracle.  Layers at N <= 2 are compared element by element; the larger
batches at 3000 sampled output positions plus every border pixel of the first
and the last output plane.
"""
import re

import numpy as np
import pytest
import torch

import broadcast_implicit_gemm_gb300 as bg
import oracle
from broadcast_implicit_gemm_gb300 import synth
from tests.test_gpu_conv import DT, NTH, _alloc_out, _guard_intact
from tests.tolerance import TAU, assert_within, conv_bound, epi_bound

pytestmark = pytest.mark.gpu

WORKLOADS = {"resnet50_fp16": synth.RESNET50_FP16, "fused": synth.FUSED_CONV,
             "depthwise_fp16": synth.DEPTHWISE_FP16, "sweep_fp32": synth.SWEEP_FP32,
             "resnet_last": synth.RESNET_LAST}
# (workload, layer index, spec): bench.py draws layer i's inputs with seed i
LAYERS = [(w, i, s) for w, specs in WORKLOADS.items() for i, s in enumerate(specs)]
ORACLE_EPI = {"none": oracle.EPI_NONE, "bias": oracle.EPI_BIAS, "bias_exp": oracle.EPI_BIAS_EXP,
              "bias_rsqrt": oracle.EPI_BIAS_RSQRT, "bias_recip": oracle.EPI_BIAS_RECIP}
_UMMA = re.compile(r"umma:(nhwc|halo|direct|strided):bn(\d+):box(\d+)x(\d+)x(\d+):split(\d+)((?::\w+)*)$")


def cand_options(cand):
    """Plan options that force the candidate a search record names."""
    m = _UMMA.match(cand)
    if m:
        amode, bn, bw, bh, _bpt, split, flags = m.groups()
        flags = set(flags.split(":")[1:])
        mode = {"nhwc": bg.MODE_SUB if "sub" in flags else bg.MODE_IM2COL if "im2col" in flags
                else bg.MODE_NHWC,
                "halo": bg.MODE_STACK if "stack" in flags else bg.MODE_HALO,
                "direct": bg.MODE_DIRECT, "strided": bg.MODE_STRIDED}[amode]
        return {"kind": bg.KIND_UMMA, "mode": mode, "tile_n": int(bn), "box_w": int(bw),
                "box_h": int(bh), "split_k": int(split),
                "resident_b": 1 if "bres" in flags else -1,
                "epi_warps": 16 if "e16" in flags else 8,
                "cta_pair": 1 if "pair" in flags else -1}
    if cand == "simt:depthwise:plane":
        return {"kind": bg.KIND_SIMT, "mode": 4}
    if cand == "simt:depthwise:band":
        return {"kind": bg.KIND_SIMT, "mode": 6}
    m = re.match(r"simt:depthwise:small(\d)$", cand)
    if m:
        return {"kind": bg.KIND_SIMT, "mode": 5, "box_h": int(m.group(1))}
    m = re.match(r"simt:depthwise:(stream|rows)(\d+)$", cand)
    if m:
        return {"kind": bg.KIND_SIMT, "mode": 3 if m.group(1) == "stream" else 2,
                "box_h": int(m.group(2))}
    if cand in ("simt:tiled", "simt:naive"):
        return {"kind": bg.KIND_SIMT, "mode": 1}
    raise AssertionError(f"unknown candidate {cand}")


def _sample(shape):
    N, CO, Ho, Wo = shape
    total = N * CO * Ho * Wo
    idx = synth.random_flat_indices(total, 3000, seed=7)
    planes = [0, N * CO - 1]
    border = [pl * Ho * Wo + y * Wo + x for pl in planes for y in range(Ho) for x in range(Wo)
              if y in (0, Ho - 1) or x in (0, Wo - 1)]
    return torch.unique(torch.cat([idx, torch.tensor(border, dtype=torch.int64)])).numpy()


def _reference(spec, x, w, b, idx, shape):
    """Exact values (at idx, or everywhere when idx is None) and the bound for tau = 1."""
    kw = dict(stride=spec.stride, pad=spec.pad, groups=spec.groups)
    if idx is None:
        pre, sabs = oracle.conv2d_nchw(x, w, nthreads=NTH, **kw)
        f = np.arange(shape[1]).reshape(1, -1, 1, 1)
    else:
        pre, sabs = oracle.conv2d_nchw_points(x, w, idx, **kw)
        f = (idx // (shape[2] * shape[3])) % shape[1]
    if spec.epi == "none":
        return pre, lambda tau: conv_bound(pre, sabs, tau, spec.out_dtype)
    if idx is None:
        ref, _ = oracle.conv2d_nchw(x, w, bias=b, epi=ORACLE_EPI[spec.epi], nthreads=NTH, **kw)
    else:
        ref, _ = oracle.conv2d_nchw_points(x, w, idx, bias=b, epi=ORACLE_EPI[spec.epi], **kw)
    arg = pre + b.double().numpy()[f]
    return ref, lambda tau: epi_bound(arg, sabs, tau, spec.epi, spec.out_dtype, ref)


def _tau(spec, cand):
    if spec.in_dtype in ("f16", "bf16"):
        return TAU["half"]
    return TAU["tf32"] if cand.startswith("umma") else TAU["fp32"]


@pytest.mark.parametrize("layer", LAYERS, ids=lambda l: f"{l[0]}-{l[2].name}")
def test_benched_plans_match_the_oracle(layer):
    workload, seed, spec = layer
    x, w, b = synth.conv_inputs(spec, seed)
    xd, wd = x.cuda(), w.cuda()
    bd = b.cuda() if b is not None else None
    shape = (spec.N, spec.CO, bg.out_size(spec.H, spec.K, spec.stride, spec.pad),
             bg.out_size(spec.W, spec.K, spec.stride, spec.pad))
    args = (spec.N, spec.H, spec.W, spec.CO, spec.CI, spec.K, spec.K, spec.stride, spec.pad,
            spec.groups, DT[spec.in_dtype], DT[spec.out_dtype], bg.EPI_NAMES[spec.epi])
    searched = bg.conv2d_nchw_plan(*args, 1)
    info = searched.describe()
    timed = [r["cand"] for r in info.get("search", []) if r["status"] == 0]
    cands = [info["cand"]] + [c for c in timed if c != info["cand"]]
    idx = None if spec.N <= 2 else _sample(shape)
    ref, bound_at = _reference(spec, x, w, b, idx, shape)
    for cand in cands:
        plan = searched if cand == info["cand"] else bg.conv2d_nchw_plan_ex(
            *args, 0, cand_options(cand))
        assert plan.describe()["cand"] == cand, f"forcing {cand} gave {plan.describe()['cand']}"
        buf, out = _alloc_out(shape, synth.TORCH_DTYPES[spec.out_dtype])
        bg.conv2d_nchw_run(plan, xd, wd, bd, 1e-5, out)
        torch.cuda.synchronize()
        assert bg.bigemm_last_device_error() == 0, f"{cand}: a device wait timed out"
        assert _guard_intact(buf), f"{cand}: write outside the output tensor"
        if idx is None:
            got = out.cpu().double().numpy()
        else:
            assert not torch.isnan(out).any(), f"{cand}: unwritten outputs"
            got = out.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().double().numpy()
        assert_within(got, ref, bound_at(_tau(spec, cand)), f"{spec.name} [{cand}]")
        plan.close()
