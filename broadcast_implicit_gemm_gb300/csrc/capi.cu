// capi.cu -- broadcast entry points ([1,C,1,1] => [N,C,H,W] and the general
// [1,P,1] => [B0,P,B1]), status strings and the version string.
#include "internal.h"

using namespace bigemm;

namespace {

bigemm_status bcast_impl(int N, int C, int H, int W, int op, const float *var, float eps, void *out,
                         bigemm_dtype out_dtype, void *stream, int flat)
{
    if (N < 1 || C < 1 || H < 1 || W < 1) return BIGEMM_ERR_INVALID_ARG;
    if (op < BIGEMM_BC_COPY || op > BIGEMM_BC_RECIP) return BIGEMM_ERR_INVALID_ARG;
    if (out_dtype < BIGEMM_F32 || out_dtype > BIGEMM_BF16) return BIGEMM_ERR_INVALID_ARG;
    if (!var || !out) return BIGEMM_ERR_INVALID_ARG;
    if ((long long)H * W > (1ll << 30)) return BIGEMM_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(out) % dtype_size(out_dtype)) != 0) return BIGEMM_ERR_INVALID_ARG;
    if (!device_state()) return BIGEMM_ERR_CUDA;
    cudaError_t e = launch_bcast(N, C, H * W, op, var, eps, out, out_dtype, flat, (cudaStream_t)stream);
    return e == cudaSuccess ? BIGEMM_OK : BIGEMM_ERR_CUDA;
}

}  // namespace

extern "C" {

bigemm_status bcast_nchw_run(int N, int C, int H, int W, int op, const float *var, float eps,
                             void *out, bigemm_dtype out_dtype, void *stream)
{
    return bcast_impl(N, C, H, W, op, var, eps, out, out_dtype, stream, 0);
}

bigemm_status bcast_nchw_run_flat(int N, int C, int H, int W, int op, const float *var,
                                  float eps, void *out, bigemm_dtype out_dtype, void *stream)
{
    return bcast_impl(N, C, H, W, op, var, eps, out, out_dtype, stream, 1);
}

bigemm_status bcast_run(int B0, int P, int B1, int op, const float *var, float eps, void *out,
                        bigemm_dtype out_dtype, void *stream)
{
    if (B0 < 1 || P < 1 || B1 < 1) return BIGEMM_ERR_INVALID_ARG;
    if (op < BIGEMM_BC_COPY || op > BIGEMM_BC_RECIP) return BIGEMM_ERR_INVALID_ARG;
    if (out_dtype < BIGEMM_F32 || out_dtype > BIGEMM_BF16) return BIGEMM_ERR_INVALID_ARG;
    if (!var || !out) return BIGEMM_ERR_INVALID_ARG;
    if ((long long)P * B1 > 0x7fffffffll) return BIGEMM_ERR_UNSUPPORTED;
    if (bcast_long_rows(B1, out_dtype) && B1 > (1 << 30)) return BIGEMM_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(out) % dtype_size(out_dtype)) != 0) return BIGEMM_ERR_INVALID_ARG;
    if (!device_state()) return BIGEMM_ERR_CUDA;
    const cudaError_t e = launch_bcast_general(B0, P, B1, op, var, eps, out, out_dtype,
                                               (cudaStream_t)stream);
    return e == cudaSuccess ? BIGEMM_OK : BIGEMM_ERR_CUDA;
}

const char *bigemm_status_string(bigemm_status s)
{
    switch (s) {
    case BIGEMM_OK: return "ok";
    case BIGEMM_ERR_INVALID_ARG: return "invalid argument";
    case BIGEMM_ERR_UNSUPPORTED: return "unsupported";
    case BIGEMM_ERR_CUDA: return "CUDA error";
    case BIGEMM_ERR_TIMEOUT: return "device wait timed out";
    case BIGEMM_ERR_NO_CANDIDATE: return "no runnable candidate";
    default: return "unknown status";
    }
}

const char *bigemm_version(void) { return "bigemm 0.1.0 (sm_103a)"; }

}  // extern "C"
