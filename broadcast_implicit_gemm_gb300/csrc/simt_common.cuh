// simt_common.cuh -- pieces shared by the SIMT conv kernels (simt_conv.cu,
// dw_conv.cu): element load / store by dtype, the fused epilogue op, and the
// argument block.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace bigemm {
namespace {


__device__ __forceinline__ float ld_in(const void *p, size_t i, int dt)
{
    if (dt == BIGEMM_F32) return __ldg(static_cast<const float *>(p) + i);
    if (dt == BIGEMM_F16) return __half2float(__ldg(static_cast<const __half *>(p) + i));
    return __bfloat162float(__ldg(static_cast<const __nv_bfloat16 *>(p) + i));
}

__device__ __forceinline__ void st_out(void *p, size_t i, float v, int dt)
{
    if (dt == BIGEMM_F32)
        static_cast<float *>(p)[i] = v;
    else if (dt == BIGEMM_F16)
        static_cast<__half *>(p)[i] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float epi_apply(int epi, float acc, const float *bias, int f, float eps)
{
    switch (epi) {
    case BIGEMM_EPI_NONE: return acc;
    case BIGEMM_EPI_BIAS: return acc + bias[f];
    case BIGEMM_EPI_BIAS_EXP: return expf(acc + bias[f]);
    case BIGEMM_EPI_BIAS_RSQRT: return rsqrtf(acc + bias[f] + eps);
    case BIGEMM_EPI_BIAS_RELU: return fmaxf(acc + bias[f], 0.f);
    default: return 1.0f / (acc + bias[f]);
    }
}

struct SimtArgs {
    int N, CI, H, W, CO, KH, KW, stride, pad, groups, Ho, Wo;
    int in_dt, out_dt, epi;
    float eps;
};


inline SimtArgs make_args(const ConvShape &s, float eps)
{
    SimtArgs a;
    a.N = s.N; a.CI = s.CI; a.H = s.H; a.W = s.W; a.CO = s.CO; a.KH = s.KH; a.KW = s.KW;
    a.stride = s.stride; a.pad = s.pad; a.groups = s.groups; a.Ho = s.Ho; a.Wo = s.Wo;
    a.in_dt = s.in_dt; a.out_dt = s.out_dt; a.epi = s.epi; a.eps = eps;
    return a;
}

}  // namespace
}  // namespace bigemm
