"""Error bounds used by the parity tests (the oracle's fp64 result is `ref`).

conv:  |gpu - ref| <= tau * S + u_out * |ref|, S = sum |a*w| (from the oracle),
       tau = 2e-3 (TF32 operands), 4e-3 (fp16/bf16 operands, fp32 accumulate),
       1e-5 (fp32 operands on the FP32 pipes).  u_out is 2^-8 for bf16 outputs
       (the rounding of the stored result, which alone would fill the 4e-3
       budget) and 0 for fp32 and fp16 outputs, whose rounding (at most
       2^-24 |ref| and 2^-11 |ref|, with |ref| <= S) the tau * S term holds.
epilogue f(acc + bias):  the conv bound propagated through f, i.e. the largest
       |f(t) - f(arg)| for |t - arg| <= tau*S + |arg|*2^-23, plus 4 ulp of the output
       type (f's own rounding, <= 2 ulp, and the final store).
bcast: |gpu - fl32(ref)| <= 2 ulp of fl32(ref); NaN where ref is NaN, inf where inf.
"""
import numpy as np

TAU = {"tf32": 2e-3, "half": 4e-3, "fp32": 1e-5}
UNIT = {"f32": 2.0 ** -24, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def ulp(x, out_dtype):
    x = np.abs(np.asarray(x, np.float64))
    if out_dtype == "f32":
        return np.spacing(x.astype(np.float32)).astype(np.float64)
    if out_dtype == "f16":
        return np.spacing(np.minimum(x, 65504).astype(np.float16)).astype(np.float64)
    # bf16: 8 significant bits
    e = np.floor(np.log2(np.maximum(x, 1e-38)))
    return 2.0 ** (e - 7)


# output rounding allowed on top of tau * S: bf16 only
U_OUT = {"f32": 0.0, "f16": 0.0, "bf16": 2.0 ** -8}


def conv_bound(ref, sabs, tau, out_dtype):
    return tau * sabs + U_OUT[out_dtype] * np.abs(ref) + 1e-30


def epi_bound(arg, sabs, tau, epi, out_dtype, ref, eps=1e-5):
    d = tau * sabs + np.abs(arg) * 2.0 ** -23
    if epi in ("bias", "bias_relu"):   # max(., 0) moves a value no more than its argument
        prop = d
    elif epi == "bias_exp":
        prop = np.exp(arg + d) - np.exp(arg)
    elif epi == "bias_rsqrt":
        lo = arg + eps - d
        with np.errstate(divide="ignore", invalid="ignore"):
            prop = np.where(lo > 0, 1.0 / np.sqrt(lo) - 1.0 / np.sqrt(arg + eps), np.inf)
    elif epi == "bias_recip":
        # 1/x moves by at most 1/(|x| - d) - 1/|x| while x keeps its sign
        lo = np.abs(arg) - d
        with np.errstate(divide="ignore", invalid="ignore"):
            prop = np.where(lo > 0, 1.0 / lo - 1.0 / np.abs(arg), np.inf)
    else:
        raise ValueError(epi)
    return prop + 4 * ulp(ref, out_dtype) + 1e-30


def assert_within(got, ref, bound, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref), f"{what}: NaN positions differ"
    inf_ref = np.isinf(ref)
    assert np.array_equal(got[inf_ref], ref[inf_ref]), f"{what}: inf positions differ"
    m = ~(nan_ref | inf_ref)
    bound = np.broadcast_to(bound, ref.shape)
    err = np.abs(got[m] - ref[m])
    ok = err <= bound[m]
    if not np.all(ok):
        i = np.argmax(err - bound[m])
        raise AssertionError(f"{what}: {np.count_nonzero(~ok)} of {ok.size} outside bound; "
                             f"worst err {err[i]:.4e} bound {bound[m][i]:.4e} "
                             f"(got {got[m][i]!r}, ref {ref[m][i]!r})")
    return float(np.max(err / bound[m])) if err.size else 0.0
