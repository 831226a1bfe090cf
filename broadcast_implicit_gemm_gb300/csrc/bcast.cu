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
//
// The general form of the same page (Introduction): any [1, P, 1] => [B0, P, B1]
// after axis fusion, the last axis broadcast.  The page says the tactic binds
// the axes three ways by dim size but gives no detail; the bindings here are
// two, chosen by row length: long rows (B1 of 64 vectors or more) take the per-channel
// kernel above with N = B0, C = P, H*W = B1; short rows take bcast_rows, where
// each thread owns a fixed 16-byte piece of a b0 slice's P*B1 run, computes
// op(var[p]) for its elements once and stores the piece into every b0 slice of
// its blockIdx.y stride, so that P and B1 together fill the block's threads
// however small each is.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fastdiv.h"
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

// Short rows: R = P * B1 elements per b0 slice.  VEC: R is a whole number of
// 16-byte vectors and the output base is 16-byte aligned; otherwise one
// element per thread position.
template <typename T, bool VEC>
__global__ void __launch_bounds__(128) bcast_rows_kernel(int B0, long long R, FastDiv fd_b1, int op,
                                                         const float *__restrict__ var, float eps,
                                                         T *__restrict__ out)
{
    griddep_enter();
    constexpr int per = VEC ? 16 / (int)sizeof(T) : 1;
    const long long npos = R / per;
    for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < npos;
         v += (long long)gridDim.x * blockDim.x) {
        union {
            T e[per];
            uint4 u;
        } s;
        const long long e0 = v * per;
#pragma unroll
        for (int k = 0; k < per; ++k)   // once per thread position, for every b0 below
            s.e[k] = cvt<T>(bc_op(op, __ldg(var + fd_div((uint32_t)(e0 + k), fd_b1)), eps));
        for (int b0 = blockIdx.y; b0 < B0; b0 += gridDim.y) {
            if constexpr (VEC)
                reinterpret_cast<uint4 *>(out + (long long)b0 * R)[v] = s.u;
            else
                out[(long long)b0 * R + e0] = s.e[0];
        }
    }
}

template <typename T>
cudaError_t launch_rows(int B0, int P, int B1, int op, const float *var, float eps, void *out,
                        cudaStream_t stream)
{
    DeviceState *ds = device_state();
    const int sms = ds ? ds->sm_count : 148;
    T *o = static_cast<T *>(out);
    ProfScope prof("bcast_rows", stream);
    const long long R = (long long)P * B1;
    const bool vec = ((R * (long long)sizeof(T)) % 16 == 0) &&
                     ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    const long long npos = vec ? R / (16 / (long long)sizeof(T)) : R;
    // thread positions across x (capped at ~64 blocks of 128 per SM), b0 slices across y
    long long gx = (npos + 127) / 128;
    if (gx > (long long)sms * 64) gx = (long long)sms * 64;
    long long gy = ((long long)sms * 64 + gx - 1) / gx;
    if (gy > B0) gy = B0;
    if (gy > 65535) gy = 65535;
    if (gy < 1) gy = 1;
    const FastDiv fd = make_fastdiv((uint32_t)B1);
    dim3 grid((unsigned)gx, (unsigned)gy);
    if (vec)
        return launch_pdl(bcast_rows_kernel<T, true>, grid, dim3(128), 0, stream, B0, R, fd, op, var, eps, o);
    return launch_pdl(bcast_rows_kernel<T, false>, grid, dim3(128), 0, stream, B0, R, fd, op, var, eps, o);
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

// Long rows (64 or more 16-byte vectors per b0 slice of one p) take the
// per-channel kernel, shorter ones bcast_rows.
bool bcast_long_rows(long long B1, int out_dt) { return B1 * dtype_size(out_dt) >= 64 * 16; }

cudaError_t launch_bcast_general(int B0, int P, int B1, int op, const float *var, float eps,
                                 void *out, int out_dt, cudaStream_t stream)
{
    if (bcast_long_rows(B1, out_dt)) return launch_bcast(B0, P, B1, op, var, eps, out, out_dt, 0, stream);
    switch (out_dt) {
    case BIGEMM_F32: return launch_rows<float>(B0, P, B1, op, var, eps, out, stream);
    case BIGEMM_F16: return launch_rows<__half>(B0, P, B1, op, var, eps, out, stream);
    default: return launch_rows<__nv_bfloat16>(B0, P, B1, op, var, eps, out, stream);
    }
}

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
