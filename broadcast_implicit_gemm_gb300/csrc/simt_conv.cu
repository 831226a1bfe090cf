// simt_conv.cu -- direct NCHW convolution on the FP32 pipes (no tensor cores).
//
// The kernels here all compute the tutorial's conv2d_nchw definition with fp32
// accumulation ("Tuning High Performance Convolution on NVIDIA GPUs", Step 1):
//  * conv_tiled  (groups = 1): a 64-channel x 64-pixel output tile per block,
//    256 threads with a 4x4 register block each; each K chunk of 16 reduction
//    terms (ci, ry, rx) stages the kernel slice and the gathered, zero-padded
//    input window in shared memory -- the tutorial's shared-memory cache stages
//    and register accumulator, with padding folded into the gather.
//  * conv_depthwise (groups = C = CO): one block per (image, channel, band of
//    output rows); the band's input rows are staged once in shared memory with
//    explicit zero borders, the channel's KHxKW taps sit in registers, and each
//    thread slides along x producing neighbouring outputs.
//  * conv_naive (any groups): one thread per output; the fallback for grouped
//    shapes neither kernel above covers.
#include <algorithm>

#include "simt_common.cuh"

// (The streaming and whole-plane depthwise kernels are in dw_conv.cu.)
namespace bigemm {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

// grid: (pixel tiles of one image, co tiles, N)
__global__ void __launch_bounds__(256) conv_tiled_kernel(SimtArgs a, const void *__restrict__ x,
                                                         const void *__restrict__ w,
                                                         const float *__restrict__ bias,
                                                         void *__restrict__ out)
{
    griddep_enter();
    __shared__ __align__(16) float ws[TK][TM];
    __shared__ __align__(16) float xs[TK][TN];
    const int n = blockIdx.z;
    const int co0 = blockIdx.y * TM;
    const int p0 = blockIdx.x * TN;
    const int HoWo = a.Ho * a.Wo;
    const int KK = a.KH * a.KW;
    const int K = a.CI * KK;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const size_t xoff = (size_t)n * a.CI * a.H * a.W;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += TK) {
        // kernel slice: ws[kk][m] = w[co0+m][k0+kk]
        for (int e = threadIdx.x; e < TK * TM; e += 256) {
            const int m = e / TK, kk = e - m * TK;
            const int co = co0 + m, k = k0 + kk;
            ws[kk][m] = (co < a.CO && k < K) ? ld_in(w, (size_t)co * K + k, a.in_dt) : 0.f;
        }
        // gathered input: xs[kk][j] = pad(data)[n, ci, y*s+ry-p, x*s+rx-p]
        for (int e = threadIdx.x; e < TK * TN; e += 256) {
            const int kk = e / TN, j = e - kk * TN;
            const int k = k0 + kk, pix = p0 + j;
            float v = 0.f;
            if (k < K && pix < HoWo) {
                const int ci = k / KK, t = k - ci * KK;
                const int ry = t / a.KW, rx = t - ry * a.KW;
                const int y = pix / a.Wo, xo = pix - y * a.Wo;
                const int iy = y * a.stride + ry - a.pad, ix = xo * a.stride + rx - a.pad;
                if (iy >= 0 && iy < a.H && ix >= 0 && ix < a.W)
                    v = ld_in(x, xoff + ((size_t)ci * a.H + iy) * a.W + ix, a.in_dt);
            }
            xs[kk][j] = v;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
            const float4 wv = *reinterpret_cast<const float4 *>(&ws[kk][ty * 4]);
            const float4 xv = *reinterpret_cast<const float4 *>(&xs[kk][tx * 4]);
            const float wr[4] = {wv.x, wv.y, wv.z, wv.w};
            const float xr[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(wr[i], xr[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int co = co0 + ty * 4 + i;
        if (co >= a.CO) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int pix = p0 + tx * 4 + j;
            if (pix < HoWo)
                st_out(out, ((size_t)n * a.CO + co) * HoWo + pix,
                       epi_apply(a.epi, acc[i][j], bias, co, a.eps), a.out_dt);
        }
    }
}

__global__ void conv_naive_kernel(SimtArgs a, const void *__restrict__ x,
                                  const void *__restrict__ w, const float *__restrict__ bias,
                                  void *__restrict__ out)
{
    griddep_enter();
    const long long total = (long long)a.N * a.CO * a.Ho * a.Wo;
    const int cig = a.CI / a.groups, cog = a.CO / a.groups;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        long long t = i;
        const int xo = (int)(t % a.Wo); t /= a.Wo;
        const int y = (int)(t % a.Ho); t /= a.Ho;
        const int f = (int)(t % a.CO);
        const int n = (int)(t / a.CO);
        const int g = f / cog;
        float acc = 0.f;
        for (int rc = 0; rc < cig; ++rc) {
            const int ci = g * cig + rc;
            for (int ry = 0; ry < a.KH; ++ry) {
                const int iy = y * a.stride + ry - a.pad;
                if (iy < 0 || iy >= a.H) continue;
                for (int rx = 0; rx < a.KW; ++rx) {
                    const int ix = xo * a.stride + rx - a.pad;
                    if (ix < 0 || ix >= a.W) continue;
                    acc = fmaf(ld_in(x, (((size_t)n * a.CI + ci) * a.H + iy) * a.W + ix, a.in_dt),
                               ld_in(w, (((size_t)f * cig + rc) * a.KH + ry) * a.KW + rx, a.in_dt),
                               acc);
                }
            }
        }
        st_out(out, (size_t)i, epi_apply(a.epi, acc, bias, f, a.eps), a.out_dt);
    }
}

constexpr int kDwMaxTaps = 49;   // up to 7x7 kernels
constexpr int kDwPX = 8;         // neighbouring outputs per thread along x

// Row pitch of a staged plane band: the left padding, the row, and room for
// every window of the last x group (zeros beyond the row).
__host__ __device__ inline int dw_pitch(int W, int pad, int Wo, int KW, int S)
{
    const int gx = (Wo + kDwPX - 1) / kDwPX;
    const int need = (gx * kDwPX - 1) * S + KW;
    const int wp = W + 2 * pad;
    return need > wp ? need : wp;
}

__device__ __forceinline__ void dw_store8(void *out, size_t o, const float (&v)[kDwPX], int n, int dt,
                                          bool vec)
{
    if (vec && dt != BIGEMM_F32) {
        union {
            uint4 u;
            __half h[8];
            __nv_bfloat16 b[8];
        } pk;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (dt == BIGEMM_F16)
                pk.h[i] = __float2half_rn(v[i]);
            else
                pk.b[i] = __float2bfloat16_rn(v[i]);
        }
        *reinterpret_cast<uint4 *>(static_cast<char *>(out) + o * 2) = pk.u;
        return;
    }
#pragma unroll
    for (int i = 0; i < kDwPX; ++i)
        if (i < n) st_out(out, o + i, v[i], dt);
}

// grid: (plane groups, row bands).  A block owns `ppb` consecutive (image,
// channel) planes and output rows [y0, y0 + rows).  K and S are compile-time
// (0: read from the arguments).
template <int K, int S>
__global__ void __launch_bounds__(256) conv_depthwise_kernel(SimtArgs a, int rows, int ppb,
                                                             const void *__restrict__ x,
                                                             const void *__restrict__ w,
                                                             const float *__restrict__ bias,
                                                             void *__restrict__ out)
{
    griddep_enter();
    extern __shared__ float sm[];
    const int KH = K ? K : a.KH, KW = K ? K : a.KW, st = S ? S : a.stride;
    const int nplanes = a.N * a.CI;
    const int pl0 = blockIdx.x * ppb;
    const int np = min(ppb, nplanes - pl0);
    const int y0 = blockIdx.y * rows;
    const int y1 = min(a.Ho, y0 + rows);
    const int iy0 = y0 * st - a.pad;
    const int rows_in = (y1 - 1 - y0) * st + KH;
    const int pitch = dw_pitch(a.W, a.pad, a.Wo, KW, st);
    const int band = rows_in * pitch;
    float *taps = sm + ppb * band;
    // stage: zero everything, then the in-image part of each row
    for (int e = threadIdx.x; e < np * band; e += blockDim.x) sm[e] = 0.f;
    for (int e = threadIdx.x; e < np * KH * KW; e += blockDim.x) {
        const int j = e / (KH * KW), t = e - j * KH * KW;
        const int c = (pl0 + j) % a.CI;
        taps[e] = ld_in(w, (size_t)c * KH * KW + t, a.in_dt);
    }
    __syncthreads();
    const bool vec_in = a.in_dt != BIGEMM_F32 && (a.W & 7) == 0 &&
                        ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
    if (vec_in) {
        const int vpr = a.W >> 3;                   // 16-byte vectors per row
        const int total = np * rows_in * vpr;
        for (int e = threadIdx.x; e < total; e += blockDim.x) {
            const int j = e / (rows_in * vpr);
            const int rem = e - j * rows_in * vpr;
            const int r = rem / vpr, v = rem - r * vpr;
            const int iy = iy0 + r;
            if (iy < 0 || iy >= a.H) continue;
            const size_t src = ((size_t)(pl0 + j) * a.H + iy) * a.W + (size_t)v * 8;
            union {
                uint4 u;
                __half h[8];
                __nv_bfloat16 b[8];
            } pk;
            pk.u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const char *>(x) + src * 2));
            float *dst = sm + j * band + r * pitch + a.pad + v * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                dst[i] = a.in_dt == BIGEMM_F16 ? __half2float(pk.h[i]) : __bfloat162float(pk.b[i]);
        }
    } else {
        const int total = np * rows_in * a.W;
        for (int e = threadIdx.x; e < total; e += blockDim.x) {
            const int j = e / (rows_in * a.W);
            const int rem = e - j * rows_in * a.W;
            const int r = rem / a.W, ix = rem - r * a.W;
            const int iy = iy0 + r;
            if (iy < 0 || iy >= a.H) continue;
            sm[j * band + r * pitch + a.pad + ix] =
                ld_in(x, ((size_t)(pl0 + j) * a.H + iy) * a.W + ix, a.in_dt);
        }
    }
    __syncthreads();
    const int gx = (a.Wo + kDwPX - 1) / kDwPX;
    const int per_plane = (y1 - y0) * gx;
    const bool vec_out = a.out_dt != BIGEMM_F32 && (a.Wo & 7) == 0 &&
                         ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    for (int e = threadIdx.x; e < np * per_plane; e += blockDim.x) {
        const int j = e / per_plane;
        const int rem = e - j * per_plane;
        const int yy = rem / gx, xg = rem - yy * gx;
        const int xo0 = xg * kDwPX;
        const float *tp = taps + j * KH * KW;
        const float *bandp = sm + j * band;
        float acc[kDwPX];
#pragma unroll
        for (int i = 0; i < kDwPX; ++i) acc[i] = 0.f;
        if (K) {
            constexpr int KK = K ? K : 1, SS = S ? S : 1;
            constexpr int WIN = (kDwPX - 1) * SS + KK;
#pragma unroll
            for (int ry = 0; ry < KK; ++ry) {
                const float *rp = bandp + (yy * SS + ry) * pitch + xo0 * SS;
                float win[WIN];
#pragma unroll
                for (int i = 0; i < WIN; ++i) win[i] = rp[i];
#pragma unroll
                for (int rx = 0; rx < KK; ++rx) {
                    const float t = tp[ry * KK + rx];
#pragma unroll
                    for (int i = 0; i < kDwPX; ++i) acc[i] = fmaf(win[i * SS + rx], t, acc[i]);
                }
            }
        } else {
            for (int ry = 0; ry < KH; ++ry) {
                const float *rp = bandp + (yy * st + ry) * pitch + xo0 * st;
                for (int rx = 0; rx < KW; ++rx) {
                    const float t = tp[ry * KW + rx];
#pragma unroll
                    for (int i = 0; i < kDwPX; ++i) acc[i] = fmaf(rp[i * st + rx], t, acc[i]);
                }
            }
        }
        const int c = (pl0 + j) % a.CI;
        if (a.epi != BIGEMM_EPI_NONE) {
            const float bv = bias[c];
#pragma unroll
            for (int i = 0; i < kDwPX; ++i) {
                if (a.epi == BIGEMM_EPI_BIAS) acc[i] += bv;
                else if (a.epi == BIGEMM_EPI_BIAS_EXP) acc[i] = expf(acc[i] + bv);
                else if (a.epi == BIGEMM_EPI_BIAS_RSQRT) acc[i] = rsqrtf(acc[i] + bv + a.eps);
                else if (a.epi == BIGEMM_EPI_BIAS_RELU) acc[i] = fmaxf(acc[i] + bv, 0.f);
                else acc[i] = 1.0f / (acc[i] + bv);
            }
        }
        const size_t o = ((size_t)(pl0 + j) * a.Ho + (y0 + yy)) * a.Wo + xo0;
        dw_store8(out, o, acc, min(kDwPX, a.Wo - xo0), a.out_dt, vec_out);
    }
}

}  // namespace


// variant 0: naive (any groups); variant 1: tiled (groups = 1)
cudaError_t launch_simt_conv(const ConvShape &s, const void *x, const void *w,
                             const float *bias, float eps, void *out, int variant,
                             cudaStream_t stream)
{
    const SimtArgs a = make_args(s, eps);
    if (variant == 1 && s.groups == 1) {
        ProfScope prof("simt_conv_tiled", stream);
        dim3 grid((s.Ho * s.Wo + TN - 1) / TN, (s.CO + TM - 1) / TM, s.N);
        return launch_pdl(conv_tiled_kernel, grid, dim3(256), 0, stream, a, x, w, bias, out);
    }
    ProfScope prof("simt_conv_naive", stream);
    const long long total = (long long)s.N * s.CO * s.Ho * s.Wo;
    long long g = (total + 255) / 256;
    DeviceState *ds = device_state();
    const long long cap = (long long)(ds ? ds->sm_count : 148) * 32;
    if (g > cap) g = cap;
    return launch_pdl(conv_naive_kernel, dim3((unsigned)g), dim3(256), 0, stream, a, x, w, bias, out);
}

// Planes per block: enough (image, channel) planes that each block has work
// for about 256 threads when a plane is small.
int dw_planes_per_block(const ConvShape &s, int rows)
{
    const int gx = (s.Wo + kDwPX - 1) / kDwPX;
    const int items = std::min(rows, s.Ho) * gx;
    if (items >= 128) return 1;
    return std::max(1, std::min(16, 256 / std::max(1, items)));
}

size_t dw_smem_bytes(const ConvShape &s, int rows)
{
    const int r = std::min(rows, s.Ho);
    const int ppb = dw_planes_per_block(s, rows);
    const size_t band = (size_t)((r - 1) * s.stride + s.KH) * dw_pitch(s.W, s.pad, s.Wo, s.KW, s.stride);
    return (ppb * band + (size_t)ppb * s.KH * s.KW) * sizeof(float);
}

cudaError_t launch_dw_conv(const ConvShape &s, const void *x, const void *w, const float *bias,
                           float eps, void *out, int rows_per_block, cudaStream_t stream)
{
    ProfScope prof("simt_conv_depthwise", stream);
    if (s.KH * s.KW > kDwMaxTaps) return cudaErrorInvalidValue;
    const SimtArgs a = make_args(s, eps);
    const int rows = std::min(rows_per_block, s.Ho);
    const int ppb = dw_planes_per_block(s, rows);
    const size_t smem = dw_smem_bytes(s, rows);
    const long long planes = (long long)s.N * s.CI;
    dim3 grid((unsigned)((planes + ppb - 1) / ppb), (unsigned)((s.Ho + rows - 1) / rows));
    auto go = [&](auto kern) {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
        }
        return launch_pdl(kern, grid, dim3(256), smem, stream, a, rows, ppb, x, w, bias, out);
    };
    const bool sq = s.KH == s.KW;
    if (sq && s.KH == 3 && s.stride == 1) return go(conv_depthwise_kernel<3, 1>);
    if (sq && s.KH == 3 && s.stride == 2) return go(conv_depthwise_kernel<3, 2>);
    if (sq && s.KH == 5 && s.stride == 1) return go(conv_depthwise_kernel<5, 1>);
    if (sq && s.KH == 5 && s.stride == 2) return go(conv_depthwise_kernel<5, 2>);
    if (sq && s.KH == 7 && s.stride == 1) return go(conv_depthwise_kernel<7, 1>);
    return go(conv_depthwise_kernel<0, 0>);
}

// Streaming depthwise: square K in {3, 5, 7} with pad K/2, stride 1 or 2.
}  // namespace bigemm
