"""Seeded random shapes through every tensor-core operand mode, output form and
epilogue: each case is checked element by element against the oracle, like the
hand-picked cases of test_gpu_conv.py.  A forced choice that the library
refuses for a shape (UNSUPPORTED, before any launch) is redrawn from the case's
own generator, up to eight times, and then left to the library (tensor cores,
automatic operand mode and tiling), so that every case runs."""
import numpy as np
import pytest

import broadcast_implicit_gemm_gb300 as bg
from tests.test_gpu_conv import DT, S, check

pytestmark = pytest.mark.gpu

MODES = {"auto": None, "nhwc": bg.MODE_NHWC, "halo": bg.MODE_HALO, "direct": bg.MODE_DIRECT,
         "sub": bg.MODE_SUB, "stack": bg.MODE_STACK, "strided": bg.MODE_STRIDED,
         "im2col": bg.MODE_IM2COL}


def _draw_opts(rng):
    mode = str(rng.choice(list(MODES)))
    opts = {"kind": bg.KIND_UMMA}
    if MODES[mode] is not None:
        opts["mode"] = MODES[mode]
    r = rng.random()
    if r < 0.3:
        opts["tile_n"] = 128
        opts["epi_warps"] = 16
    elif r < 0.5:
        opts["split_k"] = int(rng.choice([2, 3, 4]))
    elif r < 0.65:
        opts["resident_b"] = 1
    return mode, opts


def _cases(n=48, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        K = int(rng.choice([1, 1, 3, 3, 3, 5]))
        stride = int(rng.choice([1, 1, 1, 2]))
        pad = int(rng.integers(0, K // 2 + 1))
        H, W = int(rng.integers(K, 31)), int(rng.integers(K, 31))
        CI = int(rng.choice([8, 16, 24, 40, 64, 96, 128]))
        CO = int(rng.choice([16, 40, 64, 72, 128, 136, 200, 256]))
        N = int(rng.integers(1, 4))
        i_dt = str(rng.choice(["f16", "bf16", "f32"]))
        o_dt = str(rng.choice(["f16", "f32"])) if i_dt == "f16" else (i_dt if rng.random() < 0.5 else "f32")
        epi = str(rng.choice(["none", "none", "bias", "bias_exp", "bias_recip", "bias_relu"]))
        dd, kd = ("absnormal", "absnormal") if epi == "bias_recip" else ("uniform", "he")
        if epi == "bias_exp":
            o_dt = "f32"          # exp of a large sum would overflow a 16-bit output
        mode, opts = _draw_opts(rng)
        spec = S(f"rand{i}_{mode}_k{K}s{stride}p{pad}_{H}x{W}_ci{CI}_co{CO}_{i_dt}{o_dt}_{epi}",
                 N, CI, CO, H, W, K, stride, pad, i=i_dt, o=o_dt, epi=epi, dd=dd, kd=kd)
        out.append((spec, opts, seed * 1000 + i))
    return out


def _accepted(spec, opts):
    """Whether the library takes the forced choice for this shape (no launch)."""
    try:
        plan = bg.conv2d_nchw_plan_ex(spec.N, spec.H, spec.W, spec.CO, spec.CI, spec.K, spec.K,
                                      spec.stride, spec.pad, spec.groups, DT[spec.in_dtype],
                                      DT[spec.out_dtype], bg.EPI_NAMES[spec.epi], 0, opts)
    except bg.BigemmError as e:
        if e.status == 2:
            return False
        raise
    plan.close()
    return True


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0].name)
def test_random_shape(case):
    spec, opts, seed = case
    rng = np.random.default_rng(seed)
    for _ in range(8):
        if _accepted(spec, opts):
            break
        opts = _draw_opts(rng)[1]
    else:
        opts = {"kind": bg.KIND_UMMA}
    info = check(spec, opts)
    assert info["kind"] == "umma"


# ------------------------------------------------------------- depthwise
# Seeded random depthwise shapes through every SIMT depthwise kernel: the
# staged band (2), streaming (3), whole-plane (4), small-plane (5) and band of
# rows (6) kernels, or the library's own choice.  Widths are drawn so that both
# the 16-byte-row and the odd-width paths come up.
DW_MODES = [None, (2, 4), (3, 2), (3, 4), (4, 0), (5, 2), (5, 4), (6, 0)]


def _dw_opts(rng):
    m = DW_MODES[int(rng.integers(0, len(DW_MODES)))]
    if m is None:
        return {"kind": bg.KIND_SIMT}
    opts = {"kind": bg.KIND_SIMT, "mode": m[0]}
    if m[1]:
        opts["box_h"] = m[1]
    return opts


def _dw_cases(n=40, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        K = int(rng.choice([3, 3, 5, 7]))
        stride = int(rng.choice([1, 1, 2]))
        H = int(rng.integers(1, 41))
        W = int(rng.choice([int(rng.integers(1, 41)), 8 * int(rng.integers(1, 9))]))
        C = int(rng.choice([2, 3, 8, 16, 24, 40]))
        N = int(rng.integers(1, 4))
        i_dt = str(rng.choice(["f16", "bf16", "f32"]))
        o_dt = i_dt if rng.random() < 0.6 else "f32"
        epi = str(rng.choice(["none", "bias", "bias_exp", "bias_relu", "bias_recip"]))
        dd, kd = ("absnormal", "absnormal") if epi == "bias_recip" else ("uniform", "dw")
        if epi == "bias_exp":
            o_dt = "f32"
        spec = S(f"rdw{i}_k{K}s{stride}_{H}x{W}_c{C}_n{N}_{i_dt}{o_dt}_{epi}", N, C, C, H, W, K,
                 stride, K // 2, g=C, i=i_dt, o=o_dt, epi=epi, dd=dd, kd=kd)
        out.append((spec, _dw_opts(rng), seed * 1000 + i))
    return out


@pytest.mark.parametrize("case", _dw_cases(), ids=lambda c: c[0].name)
def test_random_depthwise(case):
    spec, opts, seed = case
    rng = np.random.default_rng(seed)
    for _ in range(8):
        if _accepted(spec, opts):
            break
        opts = _dw_opts(rng)
    else:
        opts = {"kind": bg.KIND_SIMT}
    info = check(spec, opts)
    assert info["kind"] == "simt"


# ------------------------------------------------------------- searched plans
# Seeded random shapes planned by the timed search over every candidate the
# library generates (all operand modes, tiles, splits, resident weights,
# epilogue-warp counts, pairs), as the benchmark plans its layers: whichever
# candidate wins must compute the conv, and it must be the fastest valid one
# of the search's own records.
def _search_cases(n=12, seed=4242):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        K = int(rng.choice([1, 3, 3, 5]))
        stride = int(rng.choice([1, 1, 2]))
        pad = int(rng.integers(0, K // 2 + 1))
        H, W = int(rng.integers(K + 2, 40)), int(rng.integers(K + 2, 40))
        CI = int(rng.choice([16, 32, 64, 96, 128]))
        CO = int(rng.choice([32, 64, 96, 128, 256]))
        N = int(rng.integers(1, 5))
        i_dt = str(rng.choice(["f16", "bf16", "f32"]))
        o_dt = "f32" if i_dt == "f32" or rng.random() < 0.3 else i_dt
        epi = str(rng.choice(["none", "bias", "bias_relu"]))
        spec = S(f"srch{i}_k{K}s{stride}p{pad}_{H}x{W}_ci{CI}_co{CO}_n{N}_{i_dt}{o_dt}_{epi}",
                 N, CI, CO, H, W, K, stride, pad, i=i_dt, o=o_dt, epi=epi)
        out.append((spec, seed * 1000 + i))
    return out


@pytest.mark.parametrize("case", _search_cases(), ids=lambda c: c[0].name)
def test_random_shape_searched_plan(case):
    spec, seed = case
    info = check(spec, search=1, seed=seed)
    assert info["chosen_by"] in ("search", "cache")
    if info["chosen_by"] == "search":
        ok = [r for r in info["search"] if r["status"] == 0]
        chosen = [r["ms"] for r in ok if r["cand"] == info["cand"]]
        assert chosen and min(chosen) == min(r["ms"] for r in ok)   # the fastest record


def _dw_search_cases(n=8, seed=99):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        K = int(rng.choice([3, 5, 7]))
        stride = int(rng.choice([1, 2]))
        H = int(rng.integers(5, 60))
        W = int(rng.choice([int(rng.integers(5, 60)), 8 * int(rng.integers(1, 9))]))
        C = int(rng.choice([8, 24, 32, 96]))
        N = int(rng.integers(1, 5))
        i_dt = str(rng.choice(["f16", "bf16", "f32"]))
        o_dt = i_dt if rng.random() < 0.6 else "f32"
        epi = str(rng.choice(["none", "bias", "bias_relu"]))
        spec = S(f"sdw{i}_k{K}s{stride}_{H}x{W}_c{C}_n{N}_{i_dt}{o_dt}_{epi}", N, C, C, H, W, K,
                 stride, K // 2, g=C, i=i_dt, o=o_dt, epi=epi, kd="dw")
        out.append((spec, seed * 1000 + i))
    return out


@pytest.mark.parametrize("case", _dw_search_cases(), ids=lambda c: c[0].name)
def test_random_depthwise_searched_plan(case):
    # the timed search over the depthwise kernels that take the shape
    spec, seed = case
    info = check(spec, search=1, seed=seed)
    assert info["kind"] == "simt" and info["chosen_by"] in ("search", "cache")
    if info["chosen_by"] == "search":
        ok = [r for r in info["search"] if r["status"] == 0]
        chosen = [r["ms"] for r in ok if r["cand"] == info["cand"]]
        assert chosen and min(chosen) == min(r["ms"] for r in ok)
