// bcast.cu -- the per-channel NCHW broadcast [1,C,1,1] => [N,C,H,W].
//
// "[CINN] Add the TileBroadcastTactic for NCHW broadcast" (PaddlePaddle PR
// 70092), Performance Impact and Example: give the preserved axis C its own
// block index so that op(var[c]) is loaded and computed once per thread, and
// let the threads of the block sweep the broadcast axes.  Here blockIdx.x = c,
// blockIdx.y strides over n, and each thread writes 16-byte vectors of the
// repeated value across the H*W plane -- a pure store stream at HBM rate.
//
// bcast_flat is the generic schedule the PR compares against: all axes fused
// into one flat index, each output recomputing op(var[(i / HW) % C]).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace bigemm {

namespace {

__device__ __forceinline__ float bc_op(int op, float v, float eps)
{
    switch (op) {
    case BIGEMM_BC_COPY: return v;
    case BIGEMM_BC_EXP: return expf(v);
    case BIGEMM_BC_RSQRT: return rsqrtf(v + eps);
    default: return 1.0f / v;
    }
}

template <typename T>
__device__ __forceinline__ T cvt(float v);
template <>
__device__ __forceinline__ float cvt<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half cvt<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt<__nv_bfloat16>(float v)
{
    return __float2bfloat16_rn(v);
}

// 16 bytes holding the value repeated.
template <typename T>
__device__ __forceinline__ uint4 splat16(T v)
{
    constexpr int per = 16 / sizeof(T);
    union {
        T e[per];
        uint4 u;
    } s;
#pragma unroll
    for (int i = 0; i < per; ++i) s.e[i] = v;
    return s.u;
}

// VEC: the plane (H*W elements) is a whole number of 16-byte vectors and the
// output base is 16-byte aligned.
template <typename T, bool VEC>
__global__ void __launch_bounds__(128) bcast_kernel(int N, int C, long long HW, int op,
                                                    const float *__restrict__ var, float eps,
                                                    T *__restrict__ out)
{
    griddep_enter();
    const int c = blockIdx.x;
    const T tv = cvt<T>(bc_op(op, __ldg(var + c), eps));   // once per thread
    if (VEC) {
        constexpr int per = 16 / sizeof(T);
        const uint4 u = splat16<T>(tv);
        const long long nvec = HW / per;
        for (int n = blockIdx.y; n < N; n += gridDim.y) {
            uint4 *plane = reinterpret_cast<uint4 *>(out + ((long long)n * C + c) * HW);
            for (long long i = threadIdx.x; i < nvec; i += blockDim.x) plane[i] = u;
        }
    } else {
        for (int n = blockIdx.y; n < N; n += gridDim.y) {
            T *plane = out + ((long long)n * C + c) * HW;
            for (long long i = threadIdx.x; i < HW; i += blockDim.x) plane[i] = tv;
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(256) bcast_flat_kernel(long long total, int C, long long HW,
                                                         int op, const float *__restrict__ var,
                                                         float eps, T *__restrict__ out)
{
    griddep_enter();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int c = (int)((i / HW) % C);
        out[i] = cvt<T>(bc_op(op, __ldg(var + c), eps));
    }
}

template <typename T>
cudaError_t launch_typed(int N, int C, long long HW, int op, const float *var, float eps,
                         void *out, int flat, cudaStream_t stream)
{
    DeviceState *ds = device_state();
    const int sms = ds ? ds->sm_count : 148;
    T *o = static_cast<T *>(out);
    if (flat) {
        ProfScope prof("bcast_flat", stream);
        const long long total = (long long)N * C * HW;
        long long g = (total + 255) / 256;
        if (g > (long long)sms * 32) g = (long long)sms * 32;
        return launch_pdl(bcast_flat_kernel<T>, dim3((unsigned)g), dim3(256), 0, stream, total, C, HW,
                          op, var, eps, o);
    }
    ProfScope prof("bcast_nchw", stream);
    // ~64 blocks of 128 threads per SM over the launch, each covering whole
    // planes of one channel (measured on [128,256,32,32] fp32: 16 blocks of
    // 256 threads per SM reached 0.81 of the copy bandwidth, 64 of 128 0.88)
    long long gy = ((long long)sms * 64 + C - 1) / C;
    if (gy > N) gy = N;
    if (gy > 65535) gy = 65535;
    if (gy < 1) gy = 1;
    dim3 grid(C, (unsigned)gy);
    const bool vec = ((HW * (long long)sizeof(T)) % 16 == 0) &&
                     ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    if (vec) return launch_pdl(bcast_kernel<T, true>, grid, dim3(128), 0, stream, N, C, HW, op, var, eps, o);
    return launch_pdl(bcast_kernel<T, false>, grid, dim3(128), 0, stream, N, C, HW, op, var, eps, o);
}

}  // namespace

cudaError_t launch_bcast(int N, int C, int HW, int op, const float *var, float eps, void *out,
                         int out_dt, int flat, cudaStream_t stream)
{
    switch (out_dt) {
    case BIGEMM_F32: return launch_typed<float>(N, C, HW, op, var, eps, out, flat, stream);
    case BIGEMM_F16: return launch_typed<__half>(N, C, HW, op, var, eps, out, flat, stream);
    default: return launch_typed<__nv_bfloat16>(N, C, HW, op, var, eps, out, flat, stream);
    }
}

}  // namespace bigemm
