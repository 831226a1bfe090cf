// dw_conv.cu -- depthwise convolution (groups = C = CO) on the FP32 pipes for
// square 3x3 / 5x5 / 7x7 kernels with pad K/2 and stride 1 or 2, computing the
// conv2d_nchw definition of "Tuning High Performance Convolution on NVIDIA
// GPUs" (Step 1) per channel with fp32 accumulation.
//  * dw_stream: one thread per 8 neighbouring outputs x R output rows of a
//    plane, reading each input row of its window once with 16-byte loads
//    straight from global memory (neighbours' overlapping vectors hit L1),
//    converting it to fp32 once and adding it into every output row it feeds.
//    No shared memory and no block barrier, so it streams at HBM rate.
//  * dw_plane (H, W <= 32): one or two whole planes per warp, staged in shared
//    memory.
//  * dw_small (stride 1, outputs at most 16 wide and 32 tall): whole planes
//    staged per warp, each thread computing a 2-row x 8-column block.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "simt_common.cuh"
namespace bigemm {

namespace {

// ---------------------------------------------------------- streaming depthwise
constexpr int kDwsXO = 8;   // neighbouring outputs per thread

// Epilogue and stores of a thread's R x 8 outputs (rows y0.., columns x0..).
template <int R>
__device__ __forceinline__ void dw_store_rows(const SimtArgs &a, const float (&acc)[R][kDwsXO],
                                              const float *__restrict__ bias,
                                              void *__restrict__ out, int c, long long plane,
                                              int x0, int y0, int vec_out)
{
    constexpr int XO = kDwsXO;
    const float bv = a.epi != BIGEMM_EPI_NONE ? bias[c] : 0.f;
    const int xn = min(XO, a.Wo - x0);
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int y = y0 + i;
        if (y >= a.Ho) break;
        float o8[XO];
#pragma unroll
        for (int o = 0; o < XO; ++o) {
            float vv = acc[i][o];
            if (a.epi == BIGEMM_EPI_BIAS) vv += bv;
            else if (a.epi == BIGEMM_EPI_BIAS_EXP) vv = expf(vv + bv);
            else if (a.epi == BIGEMM_EPI_BIAS_RSQRT) vv = rsqrtf(vv + bv + a.eps);
            else if (a.epi == BIGEMM_EPI_BIAS_RECIP) vv = 1.0f / (vv + bv);
            else if (a.epi == BIGEMM_EPI_BIAS_RELU) vv = fmaxf(vv + bv, 0.f);
            o8[o] = vv;
        }
        const size_t o = ((size_t)plane * a.Ho + y) * a.Wo + x0;
        if (vec_out && xn == XO) {
            if (a.out_dt == BIGEMM_F32) {
                float4 *q = reinterpret_cast<float4 *>(static_cast<float *>(out) + o);
                q[0] = make_float4(o8[0], o8[1], o8[2], o8[3]);
                q[1] = make_float4(o8[4], o8[5], o8[6], o8[7]);
            } else {
                uint32_t pk[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (a.out_dt == BIGEMM_F16) {
                        const __half2 h = __floats2half2_rn(o8[2 * k], o8[2 * k + 1]);
                        pk[k] = *reinterpret_cast<const uint32_t *>(&h);
                    } else {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(o8[2 * k], o8[2 * k + 1]);
                        pk[k] = *reinterpret_cast<const uint32_t *>(&h);
                    }
                }
                *reinterpret_cast<uint4 *>(static_cast<char *>(out) + o * 2) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        } else {
#pragma unroll
            for (int k = 0; k < XO; ++k)
                if (k < xn) st_out(out, o + k, o8[k], a.out_dt);
        }
    }
}

// DT: input type (BIGEMM_F32 / F16 / BF16); K: kernel size (pad K/2); S: stride;
// R: output rows per thread.  A "row unit" is R output rows of one plane, split
// into gx groups of 8 columns.  rpw > 0: each warp holds rpw whole row units
// (lane = unit * gx + g, gx <= 32), so a group's neighbours are the lanes
// beside it; rpw = 0: thread t -> (g, unit) = (t % gx, t / gx).
template <int DT>
struct DwIn;
template <>
struct DwIn<BIGEMM_F32> {
    static constexpr int VE = 4;
    __device__ static void cvt(const uint4 &u, float *f)
    {
        f[0] = __uint_as_float(u.x), f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z), f[3] = __uint_as_float(u.w);
    }
};
template <>
struct DwIn<BIGEMM_F16> {
    static constexpr int VE = 8;
    __device__ static void cvt(const uint4 &u, float *f)
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 p = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            f[2 * i] = p.x, f[2 * i + 1] = p.y;
        }
    }
};
template <>
struct DwIn<BIGEMM_BF16> {
    static constexpr int VE = 8;
    __device__ static void cvt(const uint4 &u, float *f)
    {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
            f[2 * i] = p.x, f[2 * i + 1] = p.y;
        }
    }
};


template <int DT, int K, int S, int R>
__global__ void __launch_bounds__(128) dw_stream_kernel(SimtArgs a, int gx, int nrr, int rpw,
                                                        FastDiv fd_gx, FastDiv fd_nrr,
                                                        FastDiv fd_ci,
                                                        const void *__restrict__ x,
                                                        const void *__restrict__ w,
                                                        const float *__restrict__ bias,
                                                        void *__restrict__ out, int vec_in,
                                                        int vec_out)
{
    griddep_enter();
    constexpr int XO = kDwsXO;
    constexpr int P = K / 2;
    constexpr int VE = DwIn<DT>::VE;
    constexpr int WIN = (XO - 1) * S + K;            // input columns of one row
    constexpr int NR = (R - 1) * S + K;              // input rows of the window
    constexpr int OWN = XO * S;                      // columns x0*S .. x0*S + OWN - 1
    constexpr int NVO = OWN / VE;                    // their vectors (x0*S is a multiple of VE)
    constexpr int RH = P + 1 - S > 0 ? P + 1 - S : 0;   // columns right of OWN in the window
    static_assert(P + OWN + RH == WIN, "window = left halo + own columns + right halo");
    static_assert(P <= OWN && RH <= OWN, "halos come from the neighbouring lanes");
    // indices stay below 2^31 (checked at launch); divisions by the launch's
    // fixed gx, nrr and CI are multiply-high sequences
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t units = (uint32_t)(a.N * a.CI) * (uint32_t)nrr;
    int g;
    uint32_t unit;
    if (rpw > 0) {
        const int lane = threadIdx.x & 31, ui = lane / gx;
        g = lane - ui * gx;
        unit = (t >> 5) * (uint32_t)rpw + (uint32_t)ui;
        if (ui >= rpw) unit = units;                 // spare lanes of the warp
    } else {
        uint32_t gg;
        unit = fd_divmod(t, fd_gx, &gg);
        g = (int)gg;
    }
    const bool active = unit < units;
    uint32_t rr32, c32;
    const uint32_t plane = fd_divmod(active ? unit : units - 1, fd_nrr, &rr32);
    fd_divmod(plane, fd_ci, &c32);
    const int rr = (int)rr32, c = (int)c32;
    const int x0 = g * XO, y0 = rr * R;
    const int xs = x0 * S - P, iy0 = y0 * S - P;
    const size_t esz = DT == BIGEMM_F32 ? 4 : 2;
    const char *xp = static_cast<const char *>(x) + (size_t)plane * a.H * a.W * esz;

    float wt[K * K];
#pragma unroll
    for (int i = 0; i < K * K; ++i) wt[i] = ld_in(w, (size_t)c * K * K + i, DT);
    float acc[R][XO];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int o = 0; o < XO; ++o) acc[i][o] = 0.f;

    if (vec_in != 0) {
        // Each lane loads only its own columns, every row of the window at
        // once; the halos come from the lanes of the neighbouring x groups
        // (with rpw > 0, groups g - 1 and g + 1 of a unit are lanes - 1 and
        // + 1; at the row ends the halo lies in the zero padding).  The whole
        // warp takes part in the shuffles.
        uint4 raw[NR][NVO];
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const int iy = iy0 + j;
            const bool row_in = active && iy >= 0 && iy < a.H;
            const char *row = xp + (size_t)(row_in ? iy : 0) * a.W * esz;
#pragma unroll
            for (int k = 0; k < NVO; ++k) {
                const int vx = x0 * S + k * VE;
                if (vec_in == 1) {          // 16-byte vectors (W % VE == 0)
                    raw[j][k] = (row_in && vx < a.W)
                                    ? __ldg(reinterpret_cast<const uint4 *>(row + (size_t)vx * esz))
                                    : make_uint4(0u, 0u, 0u, 0u);
                } else {                    // 4-byte words (W * esz % 4 == 0)
                    constexpr int EW = (int)(4 / (DT == BIGEMM_F32 ? 4 : 2));   // elements per word
                    uint32_t wd[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int ex = vx + q * EW;
                        wd[q] = (row_in && ex + EW <= a.W)
                                    ? __ldg(reinterpret_cast<const uint32_t *>(row + (size_t)ex * esz))
                                    : 0u;
                    }
                    raw[j][k] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                }
            }
        }
        const bool left_ok = g > 0, right_ok = g + 1 < gx;
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            float v[WIN];
#pragma unroll
            for (int k = 0; k < NVO; ++k) DwIn<DT>::cvt(raw[j][k], v + P + k * VE);
#pragma unroll
            for (int h = 0; h < P; ++h) {
                const float lv = __shfl_up_sync(0xffffffffu, v[P + OWN - P + h], 1);
                v[h] = left_ok ? lv : 0.f;
            }
#pragma unroll
            for (int h = 0; h < RH; ++h) {
                const float rv = __shfl_down_sync(0xffffffffu, v[P + h], 1);
                v[P + OWN + h] = right_ok ? rv : 0.f;
            }
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int ry = j - i * S;
                if (ry >= 0 && ry < K) {
#pragma unroll
                    for (int rx = 0; rx < K; ++rx) {
                        const float tap = wt[ry * K + rx];
#pragma unroll
                        for (int o = 0; o < XO; ++o)
                            acc[i][o] = fmaf(v[o * S + rx], tap, acc[i][o]);
                    }
                }
            }
        }
    } else {
        // element loads with bounds checks, one row at a time
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const int iy = iy0 + j;
            float v[WIN];
#pragma unroll
            for (int i = 0; i < WIN; ++i) v[i] = 0.f;
            if (active && iy >= 0 && iy < a.H) {
                const char *row = xp + (size_t)iy * a.W * esz;
#pragma unroll
                for (int i = 0; i < WIN; ++i) {
                    const int ix = xs + i;
                    if (ix >= 0 && ix < a.W) v[i] = ld_in(row, (size_t)ix, DT);
                }
            }
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int ry = j - i * S;
                if (ry >= 0 && ry < K) {
#pragma unroll
                    for (int rx = 0; rx < K; ++rx) {
                        const float tap = wt[ry * K + rx];
#pragma unroll
                        for (int o = 0; o < XO; ++o)
                            acc[i][o] = fmaf(v[o * S + rx], tap, acc[i][o]);
                    }
                }
            }
        }
    }
    if (!active) return;
    dw_store_rows<R>(a, acc, bias, out, c, plane, x0, y0, vec_out);
}

// Small planes (depthwise, H and W up to 32): each warp takes one or two whole
// (image, channel) planes at a time (two when the output is at most 16 wide,
// one per half-warp).  The planes are staged as fp32 in the warp's shared
// memory with their zero border, and lane x computes output column x of its
// plane down all rows, keeping K input rows of K values in registers: each
// output row costs S*K shared loads and K*K FMAs.  The row loop is unrolled
// by K so that the ring slot of input row r, r mod K, is a constant.
constexpr int kDwpMax = 32;   // largest H and W of the plane kernel

template <int DT, int K, int S>
__global__ void __launch_bounds__(256) dw_plane_kernel(SimtArgs a, int lp, int tstride, FastDiv fd_w,
                                                       const void *__restrict__ x,
                                                       const void *__restrict__ w,
                                                       const float *__restrict__ bias,
                                                       void *__restrict__ out)
{
    griddep_enter();
    constexpr int P = K / 2;
    extern __shared__ __align__(16) float dwp_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a fixed row pitch (the widest plane plus its border), so that every
    // shared-memory read of the window is a constant offset from the row base
    constexpr int TW = kDwpMax + 2 * P;
    const int TH = a.H + 2 * P;
    const int ppw = 32 / lp;                           // planes per warp
    float *tw = dwp_smem + (size_t)warp * ppw * tstride;
    const int half = lane / lp, xl = lane - half * lp;
    const long long planes = (long long)a.N * a.CI;
    const int HW = a.H * a.W, HWo = a.Ho * a.Wo;
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long pp = ((long long)blockIdx.x * (blockDim.x >> 5) + warp) * ppw; pp < planes;
         pp += nwarps * ppw) {
        const int np = (int)min((long long)ppw, planes - pp);
        __syncwarp();                                  // the previous planes' reads are done
        // zero border (whole tiles), then the interiors
        for (int i = lane * 4; i < ppw * tstride; i += 128)
            *reinterpret_cast<float4 *>(tw + i) = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncwarp();
        // the weights first, so that their loads overlap the plane's
        const long long plane = pp + half;
        const int c = (int)(plane % a.CI);
        float wr[K][K];
#pragma unroll
        for (int ky = 0; ky < K; ++ky)
#pragma unroll
            for (int kx = 0; kx < K; ++kx) wr[ky][kx] = ld_in(w, (size_t)c * K * K + ky * K + kx, DT);
        // the np planes are one contiguous run: 16-byte loads, four per lane in
        // flight, where it is aligned
        constexpr int VE = DwIn<DT>::VE;
        const int nel = np * HW;
        const char *src = static_cast<const char *>(x) + (size_t)(pp * HW) * (DT == BIGEMM_F32 ? 4 : 2);
        if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && nel % VE == 0) {
            const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
            const int nv = nel / VE;
            for (int v0 = 0; v0 < nv; v0 += 128) {
                uint4 u[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int v = v0 + k * 32 + lane;
                    u[k] = v < nv ? __ldg(s4 + v) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int v = v0 + k * 32 + lane;
                    if (v < nv) {
                        float f[VE];
                        DwIn<DT>::cvt(u[k], f);
#pragma unroll
                        for (int e = 0; e < VE; ++e) {
                            const int g = v * VE + e;
                            uint32_t q = 0, r = (uint32_t)g;
                            if (g >= HW) q = 1, r -= (uint32_t)HW;
                            uint32_t ix;
                            const uint32_t iy = fd_divmod(r, fd_w, &ix);
                            tw[q * tstride + (iy + P) * TW + ix + P] = f[e];
                        }
                    }
                }
            }
        } else {
            for (int i = lane; i < nel; i += 32) {
                uint32_t q = 0, r = (uint32_t)i;
                if (i >= HW) q = 1, r -= (uint32_t)HW;
                uint32_t ix;
                const uint32_t iy = fd_divmod(r, fd_w, &ix);
                tw[q * tstride + (iy + P) * TW + ix + P] = ld_in(x, (size_t)(pp * HW) + i, DT);
            }
        }
        __syncwarp();
        if (half >= np || xl >= a.Wo) continue;
        const float *t = tw + half * tstride + S * xl;
        const size_t obase = (size_t)plane * HWo + xl;
        float win[K][K];                               // ring: input row r in slot r % K
#pragma unroll
        for (int r = 0; r < K - S; ++r)
#pragma unroll
            for (int kx = 0; kx < K; ++kx) win[r % K][kx] = t[r * TW + kx];
        for (int y0 = 0; y0 < a.Ho; y0 += K) {
#pragma unroll
            for (int u = 0; u < K; ++u) {
                const int y = y0 + u;
                if (y < a.Ho) {
#pragma unroll
                    for (int j = 0; j < S; ++j) {   // the S rows this output row adds
                        const int r = S * y + K - S + j;
                        const int sl = (S * u + K - S + j) % K;
#pragma unroll
                        for (int kx = 0; kx < K; ++kx) win[sl][kx] = t[r * TW + kx];
                    }
                    // one partial sum per kernel row: K independent FMA chains
                    float pr[K];
#pragma unroll
                    for (int ky = 0; ky < K; ++ky) {
                        pr[ky] = win[(S * u + ky) % K][0] * wr[ky][0];
#pragma unroll
                        for (int kx = 1; kx < K; ++kx)
                            pr[ky] = fmaf(win[(S * u + ky) % K][kx], wr[ky][kx], pr[ky]);
                    }
                    float acc = pr[0];
#pragma unroll
                    for (int ky = 1; ky < K; ++ky) acc += pr[ky];
                    st_out(out, obase + (size_t)y * a.Wo, epi_apply(a.epi, acc, bias, c, a.eps),
                           a.out_dt);
                }
            }
        }
        (void)TH;
    }
}

// Small planes, stride 1 (outputs at most 16 wide and 32 tall): the warp
// stages one or more whole (image, channel) planes in its shared memory, in
// the input's own type, inside a zero border that is written once (only the
// interiors are rewritten for each group of planes), and each thread computes
// a TY-row x 8-column block of one plane's outputs: the TY + K - 1 input rows
// of its window are read once each (8 + K - 1 values, two per 32-bit load for
// 16-bit inputs) and feed all TY output rows, so a block costs
// (TY + K - 1)(K + 7) values read for 8 TY K^2 FMAs.  The results go to a
// compact per-warp buffer in the output type, and the warp writes the group's
// outputs -- one contiguous run of the output, like its input -- with 16-byte
// stores.  The next group's planes (and weights) arrive by 4-byte cp.async
// copies into a second buffer while the current group is computed; each
// copied word (an fp32 element, or a pair of 16-bit elements where rows have
// even length) finds its place through a table built once per block, so no
// element pays for divisions.  (Measured on the 576-channel 14 x 14 5x5 layer,
// N = 64: the streaming kernel spent about 70 thread instructions per output
// for 25 FMAs; this kernel spends about 62 and takes a third less time.)
constexpr int kDwrTX = 8;
constexpr int kDwrWarps = 4;   // warps per block

// Column of a staged row where the plane's first column sits: the left border
// is K/2 wide, widened to an even count for 16-bit inputs so that pairs of
// columns stay 32-bit aligned.
__host__ __device__ constexpr int dwr_c0(int K, int es) { return es == 2 ? (K / 2 + 1) & ~1 : K / 2; }

template <int DT>
struct DwStage {                 // 16-bit inputs: raw halves, converted in pairs on use
    using T = uint16_t;
    __device__ static float2 pair(uint32_t w)
    {
        if (DT == BIGEMM_F16) return __half22float2(*reinterpret_cast<const __half2 *>(&w));
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
    }
    // one element of a pair: the low (hi = 0) or the high half
    __device__ static float half(uint32_t w, int hi)
    {
        if (DT == BIGEMM_F16) {
            const __half2 h = *reinterpret_cast<const __half2 *>(&w);
            return hi ? __high2float(h) : __low2float(h);
        }
        const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w);
        return hi ? __high2float(h) : __low2float(h);
    }
};
template <>
struct DwStage<BIGEMM_F32> {
    using T = float;
};

template <int OT>
__device__ __forceinline__ void dw_put(char *buf, int i, float v)
{
    if (OT == BIGEMM_F32) reinterpret_cast<float *>(buf)[i] = v;
    else if (OT == BIGEMM_F16) reinterpret_cast<__half *>(buf)[i] = __float2half_rn(v);
    else reinterpret_cast<__nv_bfloat16 *>(buf)[i] = __float2bfloat16_rn(v);
}

// A thread's outputs into the warp's compact output buffer (plane slot pl,
// rows oy0.., columns ox0..; those outside the plane are dropped).  With
// 16-bit outputs and rows of even length, columns go in pairs (one 32-bit
// store each: every pair starts on an even element).
template <int OT, int TY>
__device__ __forceinline__ void dw_put_block(char *ob, const float (&acc)[TY][kDwrTX], int pl,
                                             int HW, int W, int Ho, int Wo, int oy0, int ox0)
{
    if (OT != BIGEMM_F32 && (W & 1) == 0) {
#pragma unroll
        for (int oy = 0; oy < TY; ++oy)
#pragma unroll
            for (int ox = 0; ox < kDwrTX; ox += 2)
                if (oy0 + oy < Ho && ox0 + ox < Wo) {
                    uint32_t pk;
                    if (OT == BIGEMM_F16) {
                        const __half2 h = __floats2half2_rn(acc[oy][ox], acc[oy][ox + 1]);
                        pk = *reinterpret_cast<const uint32_t *>(&h);
                    } else {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[oy][ox], acc[oy][ox + 1]);
                        pk = *reinterpret_cast<const uint32_t *>(&h);
                    }
                    reinterpret_cast<uint32_t *>(ob)[(pl * HW + (oy0 + oy) * W + ox0 + ox) >> 1] = pk;
                }
        return;
    }
#pragma unroll
    for (int oy = 0; oy < TY; ++oy)
#pragma unroll
        for (int ox = 0; ox < kDwrTX; ++ox)
            if (oy0 + oy < Ho && ox0 + ox < Wo)
                dw_put<OT>(ob, pl * HW + (oy0 + oy) * W + ox0 + ox, acc[oy][ox]);
}

// Words of a warp's weight slot: one channel's K x K weights from the 32-bit
// word holding the first (16-bit weights may start mid-word).
__host__ __device__ constexpr int dwr_wslot(int K, int es) { return es == 4 ? K * K : (K * K + 1) / 2; }

template <int DT, int K, int TY>
__global__ void __launch_bounds__(kDwrWarps * 32, TY == 2 ? (K == 7 ? 6 : 8) : (K == 7 ? 4 : 6))
dw_small_kernel(SimtArgs a, int tpp, int ppw, int bxn, int pitch, int tstride, int wbytes,
                FastDiv fd_w, FastDiv fd_hw, FastDiv fd_ci, const void *__restrict__ x,
                const void *__restrict__ w, const float *__restrict__ bias, void *__restrict__ out)
{
    constexpr int P = K / 2, TX = kDwrTX, WX = TX + K - 1, KK = K * K;
    constexpr int VE = DwIn<DT>::VE;
    constexpr int ES = DT == BIGEMM_F32 ? 4 : 2;
    constexpr int C0 = dwr_c0(K, ES);
    constexpr int WS = dwr_wslot(K, ES);
    using ST = typename DwStage<DT>::T;
    extern __shared__ __align__(16) char dwr_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HW = a.H * a.W;
    // 16-bit elements of rows of even length move in pairs; 32-bit units (an
    // fp32 element or such a pair) are copied asynchronously, two groups of
    // planes in flight per warp (the one computed and the next)
    const bool pairs = ES == 2 && (a.W & 1) == 0;
    const bool async_in = ES == 4 || pairs;
    // weights too, when every channel's block lies inside the tensor's words
    const bool async_w = async_in && ((a.CI * KK * ES) & 3) == 0;
    const int tab_n = pairs ? ppw * HW / 2 : ppw * HW;
    // the staging offset of each element (or pair, in 32-bit words) of a group
    // of planes, in NCHW order
    int *tab = reinterpret_cast<int *>(dwr_smem);
    for (int e = threadIdx.x; e < tab_n; e += blockDim.x) {
        uint32_t r, ix;
        const uint32_t q = fd_divmod((uint32_t)(pairs ? 2 * e : e), fd_hw, &r);
        const uint32_t iy = fd_divmod(r, fd_w, &ix);
        const int off = (int)(q * tstride + (iy + P) * pitch + ix + C0);
        tab[e] = pairs ? off >> 1 : off;
    }
    // per warp: two staging buffers, two weight buffers, the compact outputs
    const size_t stg = ((size_t)ppw * tstride * ES + 15) & ~(size_t)15;
    const size_t wsb = ((size_t)ppw * WS * 4 + 15) & ~(size_t)15;
    char *wb = dwr_smem + (size_t)((tab_n + 3) & ~3) * 4 + (size_t)warp * wbytes;
    char *wgt = wb + 2 * stg;
    char *ob = wgt + 2 * wsb;
    // the zero borders, once: interiors are rewritten for every group of planes
    for (int i = lane; i < (int)(2 * stg / 16); i += 32)
        reinterpret_cast<uint4 *>(wb)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    griddep_enter();
    const int pl = lane / tpp, t = lane - pl * tpp;      // plane slot, thread of the plane
    const int by = t / bxn, bx = t - by * bxn;
    const int oy0 = by * TY, ox0 = bx * TX;
    const long long planes = (long long)a.N * a.CI;
    const long long step = (long long)gridDim.x * (blockDim.x >> 5) * ppw;
    const int ESO = a.out_dt == BIGEMM_F32 ? 4 : 2;
    const int cstep = (int)(step % a.CI);
    const uint32_t wwords = (uint32_t)a.CI * KK * ES / 4;
    // the copies of the group of planes from gpp (first channel gc) into buffer b
    auto issue = [&](long long gpp, int gc, int b) {
        if (gpp < planes) {
            const int gnp = (int)min((long long)ppw, planes - gpp);
            const int units = gnp * HW * ES / 4;
            const char *src = static_cast<const char *>(x) + (size_t)gpp * HW * ES;
            char *dst = wb + b * stg;
            for (int u = lane; u < units; u += 32) cp_async4(dst + 4 * tab[u], src + 4 * u);
            if (async_w)
                for (int i = lane; i < gnp * WS; i += 32) {
                    const int s = i / WS, wd = i - s * WS;
                    uint32_t ch;
                    fd_divmod((uint32_t)(gc + s), fd_ci, &ch);
                    const uint32_t w0 = ch * KK * ES / 4 + wd;
                    if (w0 < wwords)
                        cp_async4(wgt + b * wsb + 4 * i, static_cast<const uint32_t *>(w) + w0);
                }
        }
        cp_async_commit();
    };
    long long pp = ((long long)blockIdx.x * (blockDim.x >> 5) + warp) * ppw;
    int c0 = (int)(pp % a.CI);                         // channel of the group's first plane
    int buf = 0;
    if (async_in) issue(pp, c0, 0);
    for (; pp < planes; pp += step) {
        const int np = (int)min((long long)ppw, planes - pp);
        const int nel = np * HW;
        __syncwarp();                                  // the previous group is read and written out
        int cn = c0 + cstep;
        if (cn >= a.CI) cn -= a.CI;
        if (async_in) {
            issue(pp + step, cn, buf ^ 1);
            cp_async_wait<1>();                        // this lane's copies of the group
        } else {
            // 16-bit rows of odd length: the np planes (one contiguous run of
            // the input) element by element
            ST *tw = reinterpret_cast<ST *>(wb);
            const char *src = static_cast<const char *>(x) + (size_t)pp * HW * ES;
            if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && nel % VE == 0) {
                const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
                for (int v = lane; v < nel / VE; v += 32) {
                    const uint4 u = __ldg(s4 + v);
                    const int4 o0 = reinterpret_cast<const int4 *>(tab)[2 * v];
                    const int4 o1 = reinterpret_cast<const int4 *>(tab)[2 * v + 1];
                    tw[o0.x] = (ST)u.x, tw[o0.y] = (ST)(u.x >> 16);
                    tw[o0.z] = (ST)u.y, tw[o0.w] = (ST)(u.y >> 16);
                    tw[o1.x] = (ST)u.z, tw[o1.y] = (ST)(u.z >> 16);
                    tw[o1.z] = (ST)u.w, tw[o1.w] = (ST)(u.w >> 16);
                }
            } else {
                const ST *xs = reinterpret_cast<const ST *>(src);
                for (int i = lane; i < nel; i += 32) tw[tab[i]] = xs[i];
            }
        }
        __syncwarp();                                  // every lane's copies are visible
        const bool active = pl < np && t < tpp;
        uint32_t c;
        fd_divmod((uint32_t)(c0 + pl), fd_ci, &c);
        float acc[TY][TX];
#pragma unroll
        for (int oy = 0; oy < TY; ++oy)
#pragma unroll
            for (int ox = 0; ox < TX; ++ox) acc[oy][ox] = 0.f;
        if (active) {
            float wr[K][K];
            if (async_w) {
                const char *ws = wgt + buf * wsb + pl * WS * 4 + ((c * KK * ES) & 3);
#pragma unroll
                for (int k = 0; k < KK; ++k) {
                    if constexpr (ES == 4)
                        wr[k / K][k % K] = reinterpret_cast<const float *>(ws)[k];
                    else if (DT == BIGEMM_F16)
                        wr[k / K][k % K] = __half2float(reinterpret_cast<const __half *>(ws)[k]);
                    else
                        wr[k / K][k % K] =
                            __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(ws)[k]);
                }
            } else {
#pragma unroll
                for (int ky = 0; ky < K; ++ky)
#pragma unroll
                    for (int kx = 0; kx < K; ++kx)
                        wr[ky][kx] = ld_in(w, (size_t)c * KK + ky * K + kx, DT);
            }
            // padded coordinates: output (y, x) reads rows y .. y + K - 1 and
            // columns x + C0 - P .. x + C0 + P
            const ST *base = reinterpret_cast<const ST *>(wb + buf * stg) + pl * tstride +
                             oy0 * pitch + ox0;
#pragma unroll
            for (int i = 0; i < TY + K - 1; ++i) {
                float row[WX];
                if constexpr (ES == 4) {
#pragma unroll
                    for (int j = 0; j < WX; ++j) row[j] = base[i * pitch + C0 - P + j];
                } else {
                    // pairs from the even element at or before the window's first
                    // (pitch, plane stride and ox0 are even)
                    constexpr int SK = C0 - P;                  // 0 or 1 elements to skip
                    constexpr int NPR = (WX + SK + 1) / 2;
                    const uint32_t *r32 = reinterpret_cast<const uint32_t *>(base + i * pitch);
                    float e[2 * NPR];
#pragma unroll
                    for (int j = 0; j < NPR; ++j) {
                        const float2 f = DwStage<DT>::pair(r32[j]);
                        e[2 * j] = f.x, e[2 * j + 1] = f.y;
                    }
#pragma unroll
                    for (int j = 0; j < WX; ++j) row[j] = e[j + SK];
                }
#pragma unroll
                for (int oy = 0; oy < TY; ++oy) {
                    const int ky = i - oy;
                    if (ky >= 0 && ky < K) {
#pragma unroll
                        for (int ox = 0; ox < TX; ++ox)
#pragma unroll
                            for (int kx = 0; kx < K; ++kx)
                                acc[oy][ox] = fmaf(row[ox + kx], wr[ky][kx], acc[oy][ox]);
                    }
                }
            }
            if (a.epi != BIGEMM_EPI_NONE) {
                const float bv = bias[c];
                float *f = &acc[0][0];
                switch (a.epi) {
                case BIGEMM_EPI_BIAS:
#pragma unroll
                    for (int j = 0; j < TY * TX; ++j) f[j] += bv;
                    break;
                case BIGEMM_EPI_BIAS_EXP:
#pragma unroll
                    for (int j = 0; j < TY * TX; ++j) f[j] = expf(f[j] + bv);
                    break;
                case BIGEMM_EPI_BIAS_RSQRT:
#pragma unroll
                    for (int j = 0; j < TY * TX; ++j) f[j] = rsqrtf(f[j] + bv + a.eps);
                    break;
                case BIGEMM_EPI_BIAS_RELU:
#pragma unroll
                    for (int j = 0; j < TY * TX; ++j) f[j] = fmaxf(f[j] + bv, 0.f);
                    break;
                default:
#pragma unroll
                    for (int j = 0; j < TY * TX; ++j) f[j] = 1.0f / (f[j] + bv);
                }
            }
            if (a.out_dt == BIGEMM_F32)
                dw_put_block<BIGEMM_F32, TY>(ob, acc, pl, HW, a.W, a.Ho, a.Wo, oy0, ox0);
            else if (a.out_dt == BIGEMM_F16)
                dw_put_block<BIGEMM_F16, TY>(ob, acc, pl, HW, a.W, a.Ho, a.Wo, oy0, ox0);
            else
                dw_put_block<BIGEMM_BF16, TY>(ob, acc, pl, HW, a.W, a.Ho, a.Wo, oy0, ox0);
        }
        __syncwarp();
        // the group's outputs are one contiguous run too (Ho = H, Wo = W)
        char *dst = static_cast<char *>(out) + (size_t)pp * HW * ESO;
        const int nb = nel * ESO;
        if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0 && nb % 16 == 0) {
            for (int v = lane; v < nb / 16; v += 32)
                reinterpret_cast<uint4 *>(dst)[v] = reinterpret_cast<const uint4 *>(ob)[v];
        } else if (ESO == 4) {
            for (int i = lane; i < nel; i += 32)
                reinterpret_cast<float *>(dst)[i] = reinterpret_cast<const float *>(ob)[i];
        } else {
            for (int i = lane; i < nel; i += 32)
                reinterpret_cast<uint16_t *>(dst)[i] = reinterpret_cast<const uint16_t *>(ob)[i];
        }
        c0 = cn;
        if (async_in) buf ^= 1;
    }
    cp_async_wait<0>();
}

// The small-plane kernel's geometry for a shape and block height TY: threads
// per plane, planes per warp, column blocks, the staging row pitch and plane
// stride (elements), each warp's shared bytes (staging, weights, compact
// outputs) and the dynamic shared memory of a block; false when it does not
// apply.
struct DwSmallGeom {
    int tpp, ppw, bxn, pitch, tstride, wbytes;
    size_t smem;
};

constexpr size_t kDwrSmemMax = 96 * 1024;

bool dw_small_geom_search(const ConvShape &s, int TY, DwSmallGeom &g)
{
    if (!(s.groups > 1 && s.groups == s.CI && s.CO == s.CI)) return false;
    if (s.KH != s.KW || s.pad != s.KH / 2 || s.stride != 1) return false;
    if (!(s.KH == 3 || s.KH == 5 || s.KH == 7)) return false;
    if (!(TY == 2 || TY == 4)) return false;
    if (s.Wo > 2 * kDwrTX || s.Ho > 32) return false;
    const int K = s.KH;
    const int es = dtype_size(s.in_dt), eso = dtype_size(s.out_dt);
    const int step = es == 2 ? 2 : 1;        // 16-bit rows are read as pairs: even offsets
    g.bxn = (s.Wo + kDwrTX - 1) / kDwrTX;
    const int rb = (s.Ho + TY - 1) / TY;
    g.tpp = g.bxn * rb;
    if (g.tpp > 32) return false;
    // interior at column dwr_c0, right border K/2 wide; 16-bit rows keep one
    // more column, read (and dropped) by the last pair of a window
    const int c0 = dwr_c0(K, es), extra = es == 2 ? 1 : 0;
    const int pmin = (g.bxn * kDwrTX + c0 + K / 2 + extra + step - 1) / step * step;
    const int rows = rb * TY + K - 1;
    const int HW = s.H * s.W;
    // as many planes per warp as fill its lanes, fewer where a block's shared
    // memory would pass the limit
    for (g.ppw = 32 / g.tpp; g.ppw >= 1; --g.ppw) {
        // the row pitch and plane stride (padding of up to 31 elements each)
        // that put the fewest lanes of a warp on one bank when they read their
        // windows: the lanes read at the same offset from their first word, so
        // the first words' banks decide; then the smallest stride
        int best_conf = 1 << 30;
        for (int pitch = pmin; pitch < pmin + 32; pitch += step)
            for (int ts = rows * pitch; ts < rows * pitch + 32; ts += step) {
                int cnt[32] = {0}, worst = 0;
                for (int l = 0; l < g.ppw * g.tpp; ++l) {
                    const int pl = l / g.tpp, t = l - pl * g.tpp;
                    const int off = pl * ts + (t / g.bxn) * TY * pitch + (t % g.bxn) * kDwrTX;
                    worst = std::max(worst, ++cnt[(off / step) & 31]);
                }
                if (worst < best_conf || (worst == best_conf && ts < g.tstride))
                    best_conf = worst, g.pitch = pitch, g.tstride = ts;
            }
        // the element table (one int per element or pair of a group), then per
        // warp two staging buffers, two weight buffers and the compact
        // outputs, each rounded to 16 bytes
        const bool pairs = es == 2 && (s.W & 1) == 0;
        const size_t tab = (size_t)(((pairs ? g.ppw * HW / 2 : g.ppw * HW) + 3) & ~3) * 4;
        const size_t stg = ((size_t)g.ppw * g.tstride * es + 15) & ~(size_t)15;
        const size_t wsb = ((size_t)g.ppw * dwr_wslot(K, es) * 4 + 15) & ~(size_t)15;
        const size_t obuf = ((size_t)g.ppw * HW * eso + 15) & ~(size_t)15;
        g.wbytes = (int)(2 * stg + 2 * wsb + obuf);
        g.smem = tab + kDwrWarps * (size_t)g.wbytes;
        if (g.smem <= kDwrSmemMax) return true;
    }
    return false;
}

// The search above runs once per shape and TY: plans and launches look it up.
bool dw_small_geom(const ConvShape &s, int TY, DwSmallGeom &g)
{
    static std::mutex mu;
    using Key = std::tuple<int, int, int, int, int, int, int, int, int, int>;
    static std::map<Key, std::pair<bool, DwSmallGeom>> memo;
    const Key key(s.groups == s.CI && s.CO == s.CI && s.groups > 1 ? 1 : 0, s.Ho, s.Wo, s.KH,
                  s.KW, s.pad, s.stride, s.in_dt, s.out_dt, TY);
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find(key);
    if (it == memo.end()) {
        DwSmallGeom found{};
        const bool ok = dw_small_geom_search(s, TY, found);
        it = memo.emplace(key, std::make_pair(ok, found)).first;
    }
    g = it->second.second;
    return it->second.first;
}

// Bands of large planes (rows of 16-byte multiples, at most 512 bytes): a warp
// takes a run of (plane, band) items -- a band is rbw x 4 output rows of one
// plane, all its columns -- and stages each band's input rows in its shared
// memory with 16-byte cp.async copies, inside a zero border (left and right
// columns written once, rows outside the plane zeroed per band), the next
// band arriving while the current one is computed.  Each thread computes a
// 4-row x 8-column block (rbw row blocks x bxn column blocks per warp) as the
// small-plane kernel does, with stride S, and writes each output row's 8
// values with one 16-byte store (two for fp32).  A warp's items are
// consecutive, so its weights are loaded once per plane.
constexpr int kDwbTY = 4;

template <int DT, int K, int S>
__global__ void __launch_bounds__(kDwrWarps * 32, 4)
dw_band_kernel(SimtArgs a, int bxn, int rbw, int nbands, int ir, int pitch, int wbytes, int ipw,
               FastDiv fd_nb, FastDiv fd_ci, const void *__restrict__ x, const void *__restrict__ w,
               const float *__restrict__ bias, void *__restrict__ out)
{
    constexpr int P = K / 2, TX = kDwrTX, TY = kDwbTY, KK = K * K;
    constexpr int ES = DT == BIGEMM_F32 ? 4 : 2;
    constexpr int C0 = 16 / ES;                        // left border: 16 bytes
    constexpr int WXS = (TX - 1) * S + K;              // window columns of a thread
    constexpr int NR = (TY - 1) * S + K;               // window rows of a thread
    using ST = typename DwStage<DT>::T;
    extern __shared__ __align__(16) char dwb_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    char *wb = dwb_smem + (size_t)warp * wbytes;
    const int stg = (ir * pitch * ES + 15) & ~15;
    for (int i = lane; i < 2 * stg / 16; i += 32)
        reinterpret_cast<uint4 *>(wb)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    griddep_enter();
    const int cw = a.W * ES / 16;                      // 16-byte chunks of an input row
    const int rpi = 32 / cw;                           // rows copied per pass of the warp
    const int rr = lane / cw, ck = lane - rr * cw;
    const int by = lane / bxn, bx = lane - by * bxn;   // the thread's row block, column block
    const bool active = by < rbw;
    const int ox0 = bx * TX;
    const int items = a.N * a.CI * nbands;
    const int it0 = ((int)blockIdx.x * kDwrWarps + warp) * ipw;
    const int it1 = min(items, it0 + ipw);
    const size_t plane_in = (size_t)a.H * a.W, plane_out = (size_t)a.Ho * a.Wo;
    // the input rows of item `item` into buffer b
    auto issue = [&](int item, int b) {
        if (item < it1) {
            uint32_t band;
            const uint32_t plane = fd_divmod((uint32_t)item, fd_nb, &band);
            const int iy0 = (int)band * rbw * TY * S - P;
            const char *src = static_cast<const char *>(x) + plane * plane_in * ES;
            char *dst = wb + b * stg + C0 * ES + ck * 16;
            if (rr < rpi)
                for (int r = rr; r < ir; r += rpi) {
                    const int iy = iy0 + r;
                    char *d = dst + (size_t)r * pitch * ES;
                    if (iy >= 0 && iy < a.H)
                        cp_async16(d, src + (size_t)iy * a.W * ES + ck * 16);
                    else
                        *reinterpret_cast<uint4 *>(d) = make_uint4(0u, 0u, 0u, 0u);
                }
        }
        cp_async_commit();
    };
    float wr[K][K];
    int wplane = -1;
    int buf = 0;
    if (it0 < it1) issue(it0, 0);
    for (int item = it0; item < it1; ++item) {
        __syncwarp();                                  // the previous band is read
        issue(item + 1, buf ^ 1);
        cp_async_wait<1>();                            // this lane's copies of the band
        __syncwarp();                                  // every lane's copies and zeros are visible
        uint32_t band;
        const uint32_t plane = fd_divmod((uint32_t)item, fd_nb, &band);
        uint32_t c;
        fd_divmod(plane, fd_ci, &c);
        if ((int)plane != wplane) {
            wplane = (int)plane;
#pragma unroll
            for (int k = 0; k < KK; ++k) wr[k / K][k % K] = ld_in(w, (size_t)c * KK + k, DT);
        }
        const int y0 = (int)band * rbw * TY + by * TY;   // the thread's first output row
        if (active && y0 < a.Ho && ox0 < a.Wo) {
            float acc[TY][TX];
#pragma unroll
            for (int oy = 0; oy < TY; ++oy)
#pragma unroll
                for (int ox = 0; ox < TX; ++ox) acc[oy][ox] = 0.f;
            // band-local row (by * TY + oy) * S + ky, column ox * S + kx + C0 - P
            const ST *base = reinterpret_cast<const ST *>(wb + buf * stg) +
                             (size_t)by * TY * S * pitch + ox0 * S;
            // the window's row i as 16-byte chunks from the thread's first
            // column (16-byte aligned: pitch and ox0 * S are multiples of a chunk)
            constexpr int EPC = 16 / ES;                       // elements per chunk
            constexpr int LO = C0 - P;                         // first window element in the run
            constexpr int NCH = (LO + WXS + EPC - 1) / EPC;
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                float row[WXS];
                const uint4 *rc = reinterpret_cast<const uint4 *>(base + i * pitch);
                uint32_t wd[4 * NCH];
#pragma unroll
                for (int k = 0; k < NCH; ++k) {
                    const uint4 u = rc[k];
                    wd[4 * k] = u.x, wd[4 * k + 1] = u.y, wd[4 * k + 2] = u.z, wd[4 * k + 3] = u.w;
                }
#pragma unroll
                for (int j = 0; j < WXS; ++j) {
                    const int el = LO + j;
                    if constexpr (ES == 4)
                        row[j] = __uint_as_float(wd[el]);
                    else
                        row[j] = DwStage<DT>::half(wd[el >> 1], el & 1);
                }
#pragma unroll
                for (int oy = 0; oy < TY; ++oy) {
                    const int ky = i - oy * S;
                    if (ky >= 0 && ky < K) {
#pragma unroll
                        for (int ox = 0; ox < TX; ++ox)
#pragma unroll
                            for (int kx = 0; kx < K; ++kx)
                                acc[oy][ox] = fmaf(row[ox * S + kx], wr[ky][kx], acc[oy][ox]);
                    }
                }
            }
            if (a.epi != BIGEMM_EPI_NONE) {
                const float bv = bias[c];
                float *f = &acc[0][0];
                switch (a.epi) {
                case BIGEMM_EPI_BIAS:
#pragma unroll
                    for (int j = 0; j < TY * TX; ++j) f[j] += bv;
                    break;
                case BIGEMM_EPI_BIAS_EXP:
#pragma unroll
                    for (int j = 0; j < TY * TX; ++j) f[j] = expf(f[j] + bv);
                    break;
                case BIGEMM_EPI_BIAS_RSQRT:
#pragma unroll
                    for (int j = 0; j < TY * TX; ++j) f[j] = rsqrtf(f[j] + bv + a.eps);
                    break;
                case BIGEMM_EPI_BIAS_RELU:
#pragma unroll
                    for (int j = 0; j < TY * TX; ++j) f[j] = fmaxf(f[j] + bv, 0.f);
                    break;
                default:
#pragma unroll
                    for (int j = 0; j < TY * TX; ++j) f[j] = 1.0f / (f[j] + bv);
                }
            }
            const int ESO = a.out_dt == BIGEMM_F32 ? 4 : 2;
            char *orow = static_cast<char *>(out) + (plane * plane_out + (size_t)y0 * a.Wo + ox0) * ESO;
            // 16-byte stores: whole 8-column blocks of rows that keep 16-byte alignment
            const bool vec = ox0 + TX <= a.Wo && (a.Wo * ESO) % 16 == 0 &&
                             (reinterpret_cast<uintptr_t>(out) & 15) == 0;
#pragma unroll
            for (int oy = 0; oy < TY; ++oy) {
                if (y0 + oy >= a.Ho) break;
                char *o = orow + (size_t)oy * a.Wo * ESO;
                if (vec) {
                    if (a.out_dt == BIGEMM_F32) {
                        reinterpret_cast<float4 *>(o)[0] =
                            make_float4(acc[oy][0], acc[oy][1], acc[oy][2], acc[oy][3]);
                        reinterpret_cast<float4 *>(o)[1] =
                            make_float4(acc[oy][4], acc[oy][5], acc[oy][6], acc[oy][7]);
                    } else {
                        uint32_t pk[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            if (a.out_dt == BIGEMM_F16) {
                                const __half2 h = __floats2half2_rn(acc[oy][2 * k], acc[oy][2 * k + 1]);
                                pk[k] = *reinterpret_cast<const uint32_t *>(&h);
                            } else {
                                const __nv_bfloat162 h =
                                    __floats2bfloat162_rn(acc[oy][2 * k], acc[oy][2 * k + 1]);
                                pk[k] = *reinterpret_cast<const uint32_t *>(&h);
                            }
                        }
                        *reinterpret_cast<uint4 *>(o) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                } else {
#pragma unroll
                    for (int ox = 0; ox < TX; ++ox)
                        if (ox0 + ox < a.Wo)
                            st_out(out, plane * plane_out + (size_t)(y0 + oy) * a.Wo + ox0 + ox,
                                   acc[oy][ox], a.out_dt);
                }
            }
        }
        buf ^= 1;
    }
    cp_async_wait<0>();
}

// The band kernel's geometry: column blocks, row blocks per warp, bands per
// plane, input rows per band, the staging row pitch (elements), each warp's
// shared bytes (two staging buffers) and a block's; false when it does not
// apply.
struct DwBandGeom {
    int bxn, rbw, nbands, ir, pitch, wbytes;
    size_t smem;
};

bool dw_band_geom(const ConvShape &s, DwBandGeom &g)
{
    if (!(s.groups > 1 && s.groups == s.CI && s.CO == s.CI)) return false;
    if (s.KH != s.KW || s.pad != s.KH / 2 || !(s.stride == 1 || s.stride == 2)) return false;
    if (!(s.KH == 3 || s.KH == 5 || s.KH == 7)) return false;
    const int es = dtype_size(s.in_dt), K = s.KH, S = s.stride, P = K / 2;
    if ((s.W * es) % 16 != 0 || s.W * es > 512) return false;   // whole 16-byte chunks, <= 32 per row
    g.bxn = (s.Wo + kDwrTX - 1) / kDwrTX;
    if (g.bxn > 32) return false;
    g.rbw = std::min(32 / g.bxn, (s.Ho + kDwbTY - 1) / kDwbTY);
    const int rows = g.rbw * kDwbTY;
    g.nbands = (s.Ho + rows - 1) / rows;
    if ((long long)s.N * s.CI * g.nbands >= (1ll << 31)) return false;
    g.ir = (rows - 1) * S + K;
    const int c0 = 16 / es, step = 16 / es;        // rows start on 16-byte boundaries
    // the last column block's window ends at (bxn * 8 - 1) * S + P (+1 for the
    // pair read) past the left border
    const int need = c0 + std::max(s.W, (g.bxn * kDwrTX - 1) * S + P + 2);
    const int pmin = (need + step - 1) / step * step;
    // threads read their rows as 16-byte chunks, served a quarter-warp (eight
    // threads) at a time: the pitch that puts the fewest threads of a quarter
    // on one 16-byte bank group
    int best = 1 << 30;
    for (int pitch = pmin; pitch < pmin + 16 * step; pitch += step) {
        int worst = 0;
        for (int q0 = 0; q0 < g.rbw * g.bxn; q0 += 8) {
            int cnt[8] = {0};
            for (int l = q0; l < std::min(q0 + 8, g.rbw * g.bxn); ++l) {
                const int b_y = l / g.bxn, b_x = l - b_y * g.bxn;
                const int off = b_y * kDwbTY * S * pitch + b_x * kDwrTX * S;   // elements
                worst = std::max(worst, ++cnt[(off / step) & 7]);
            }
        }
        if (worst < best) best = worst, g.pitch = pitch;
    }
    const size_t stg = ((size_t)g.ir * g.pitch * es + 15) & ~(size_t)15;
    g.wbytes = (int)(2 * stg);
    g.smem = kDwrWarps * (size_t)g.wbytes;
    return g.smem <= kDwrSmemMax;
}

}  // namespace

// Resident blocks per SM of a small-plane kernel with this much
// dynamic shared memory (looked up once per kernel and size).
int dw_small_blocks_per_sm(const void *kern, size_t smem)
{
    static std::mutex mu;
    static std::map<std::pair<const void *, size_t>, int> memo;
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find({kern, smem});
    if (it != memo.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDwrWarps * 32, smem) != cudaSuccess ||
        n < 1)
        n = 1;
    memo[{kern, smem}] = n;
    return n;
}

bool dw_small_ok(const ConvShape &s, int TY)
{
    DwSmallGeom g;
    if (!dw_small_geom(s, TY, g)) return false;
    DeviceState *ds = device_state();
    return !ds || g.smem <= (size_t)ds->max_smem_optin;
}

cudaError_t launch_dw_small(const ConvShape &s, const void *x, const void *w, const float *bias,
                            float eps, void *out, int TY, cudaStream_t stream)
{
    DwSmallGeom g;
    if (!dw_small_geom(s, TY, g)) return cudaErrorInvalidValue;
    ProfScope prof("simt_conv_depthwise", stream);
    const SimtArgs a = make_args(s, eps);
    const long long planes = (long long)s.N * s.CI;
    DeviceState *ds = device_state();
    const int sms = ds ? ds->sm_count : 148;
    const long long warps_needed = (planes + g.ppw - 1) / g.ppw;
    const FastDiv fdw = make_fastdiv((uint32_t)s.W), fdhw = make_fastdiv((uint32_t)(s.H * s.W));
    const FastDiv fdci = make_fastdiv((uint32_t)s.CI);
    auto go = [&](auto kern) {
        if (g.smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)g.smem);
            if (e != cudaSuccess) return e;
        }
        // one wave of resident blocks: each warp builds its table and zero
        // border once and then takes group after group of planes
        const int bps = dw_small_blocks_per_sm(reinterpret_cast<const void *>(kern), g.smem);
        long long blocks =
            std::min<long long>((warps_needed + kDwrWarps - 1) / kDwrWarps, (long long)sms * bps);
        if (blocks < 1) blocks = 1;
        return launch_pdl(kern, dim3((unsigned)blocks), dim3(kDwrWarps * 32), g.smem, stream, a,
                          g.tpp, g.ppw,
                          g.bxn, g.pitch, g.tstride, g.wbytes, fdw, fdhw, fdci, x, w, bias, out);
    };
#define BIGEMM_DWR(DTV, TYV)                                          \
    if (s.KH == 3) return go(dw_small_kernel<DTV, 3, TYV>);           \
    if (s.KH == 5) return go(dw_small_kernel<DTV, 5, TYV>);           \
    if (s.KH == 7) return go(dw_small_kernel<DTV, 7, TYV>);           \
    return cudaErrorInvalidValue;
    if (TY == 2) {
        if (s.in_dt == BIGEMM_F32) { BIGEMM_DWR(BIGEMM_F32, 2) }
        if (s.in_dt == BIGEMM_F16) { BIGEMM_DWR(BIGEMM_F16, 2) }
        BIGEMM_DWR(BIGEMM_BF16, 2)
    }
    if (s.in_dt == BIGEMM_F32) { BIGEMM_DWR(BIGEMM_F32, 4) }
    if (s.in_dt == BIGEMM_F16) { BIGEMM_DWR(BIGEMM_F16, 4) }
    BIGEMM_DWR(BIGEMM_BF16, 4)
#undef BIGEMM_DWR
}

bool dw_band_ok(const ConvShape &s)
{
    DwBandGeom g;
    if (!dw_band_geom(s, g)) return false;
    DeviceState *ds = device_state();
    return !ds || g.smem <= (size_t)ds->max_smem_optin;
}

cudaError_t launch_dw_band(const ConvShape &s, const void *x, const void *w, const float *bias,
                           float eps, void *out, cudaStream_t stream)
{
    DwBandGeom g;
    if (!dw_band_geom(s, g)) return cudaErrorInvalidValue;
    ProfScope prof("simt_conv_depthwise", stream);
    const SimtArgs a = make_args(s, eps);
    DeviceState *ds = device_state();
    const int sms = ds ? ds->sm_count : 148;
    const long long items = (long long)s.N * s.CI * g.nbands;
    const FastDiv fdnb = make_fastdiv((uint32_t)g.nbands), fdci = make_fastdiv((uint32_t)s.CI);
    auto go = [&](auto kern) {
        if (g.smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)g.smem);
            if (e != cudaSuccess) return e;
        }
        // one wave of resident blocks; each warp takes a run of consecutive items
        const int bps = dw_small_blocks_per_sm(reinterpret_cast<const void *>(kern), g.smem);
        const long long warps = std::max<long long>(
            1, std::min<long long>((long long)sms * bps * kDwrWarps, items));
        const int ipw = (int)((items + warps - 1) / warps);
        const long long blocks = ((items + ipw - 1) / ipw + kDwrWarps - 1) / kDwrWarps;
        return launch_pdl(kern, dim3((unsigned)blocks), dim3(kDwrWarps * 32), g.smem, stream, a,
                          g.bxn, g.rbw, g.nbands, g.ir, g.pitch, g.wbytes, ipw, fdnb, fdci, x, w,
                          bias, out);
    };
#define BIGEMM_DWB(DTV, SV)                                         \
    if (s.KH == 3) return go(dw_band_kernel<DTV, 3, SV>);           \
    if (s.KH == 5) return go(dw_band_kernel<DTV, 5, SV>);           \
    if (s.KH == 7) return go(dw_band_kernel<DTV, 7, SV>);           \
    return cudaErrorInvalidValue;
    if (s.stride == 1) {
        if (s.in_dt == BIGEMM_F32) { BIGEMM_DWB(BIGEMM_F32, 1) }
        if (s.in_dt == BIGEMM_F16) { BIGEMM_DWB(BIGEMM_F16, 1) }
        BIGEMM_DWB(BIGEMM_BF16, 1)
    }
    if (s.in_dt == BIGEMM_F32) { BIGEMM_DWB(BIGEMM_F32, 2) }
    if (s.in_dt == BIGEMM_F16) { BIGEMM_DWB(BIGEMM_F16, 2) }
    BIGEMM_DWB(BIGEMM_BF16, 2)
#undef BIGEMM_DWB
}

bool dw_stream_ok(const ConvShape &s)
{
    if (!(s.groups > 1 && s.groups == s.CI && s.CO == s.CI)) return false;
    if (s.KH != s.KW || s.pad != s.KH / 2) return false;
    if (!(s.KH == 3 || s.KH == 5 || s.KH == 7)) return false;
    return s.stride == 1 || s.stride == 2;
}

size_t dw_plane_smem(const ConvShape &s, int *lp, int *tstride);

bool dw_plane_ok(const ConvShape &s)
{
    if (!(dw_stream_ok(s) && s.H <= kDwpMax && s.W <= kDwpMax && s.Wo <= 32)) return false;
    int lp = 0, ts = 0;
    return dw_plane_smem(s, &lp, &ts) <= 48 * 1024;   // static-size limit, no opt-in
}

size_t dw_plane_smem(const ConvShape &s, int *lp, int *tstride)
{
    const int P = s.KH / 2;
    const int tsz = (s.H + 2 * P) * (kDwpMax + 2 * P);   // the kernel's fixed row pitch
    // a plane's floats rounded up to 4; with two planes per warp, an odd
    // multiple of 16 so that the two half-warps' planes sit on different banks
    const int t1 = (tsz + 3) & ~3;
    const int t2 = ((t1 + 15) / 16 | 1) * 16;
    const bool two = s.Wo <= 16 && (size_t)8 * 2 * t2 * sizeof(float) <= 48 * 1024;
    *lp = two ? 16 : 32;
    *tstride = two ? t2 : t1;
    return (size_t)8 * (two ? 2 : 1) * (*tstride) * sizeof(float);
}

cudaError_t launch_dw_plane(const ConvShape &s, const void *x, const void *w, const float *bias,
                            float eps, void *out, cudaStream_t stream)
{
    if (!dw_plane_ok(s)) return cudaErrorInvalidValue;
    ProfScope prof("simt_conv_depthwise", stream);
    const SimtArgs a = make_args(s, eps);
    int lp = 32, tstride = 0;
    const size_t smem = dw_plane_smem(s, &lp, &tstride);
    const long long planes = (long long)s.N * s.CI;
    DeviceState *ds = device_state();
    const int sms = ds ? ds->sm_count : 148;
    const long long warps_needed = (planes + (32 / lp) - 1) / (32 / lp);
    long long blocks = std::min<long long>((warps_needed + 7) / 8, (long long)sms * 8);
    if (blocks < 1) blocks = 1;
    const FastDiv fdw = make_fastdiv((uint32_t)s.W);
    auto go = [&](auto kern) {
        return launch_pdl(kern, dim3((unsigned)blocks), dim3(256), smem, stream, a, lp, tstride, fdw,
                          x, w, bias, out);
    };
#define BIGEMM_DWP(DTV, KV, SV) \
    if (s.KH == KV && s.stride == SV) return go(dw_plane_kernel<DTV, KV, SV>);
#define BIGEMM_DWPS(DTV)                                                                 \
    BIGEMM_DWP(DTV, 3, 1) BIGEMM_DWP(DTV, 3, 2) BIGEMM_DWP(DTV, 5, 1) BIGEMM_DWP(DTV, 5, 2) \
    BIGEMM_DWP(DTV, 7, 1) BIGEMM_DWP(DTV, 7, 2) return cudaErrorInvalidValue;
    if (s.in_dt == BIGEMM_F32) { BIGEMM_DWPS(BIGEMM_F32) }
    if (s.in_dt == BIGEMM_F16) { BIGEMM_DWPS(BIGEMM_F16) }
    BIGEMM_DWPS(BIGEMM_BF16)
#undef BIGEMM_DWPS
#undef BIGEMM_DWP
}

cudaError_t launch_dw_stream(const ConvShape &s, const void *x, const void *w, const float *bias,
                             float eps, void *out, int rows, cudaStream_t stream)
{
    if (!dw_stream_ok(s)) return cudaErrorInvalidValue;
    // rows per thread: 2, 4 or 8 (8 only at stride 1 with K <= 5)
    const int R = rows >= 8 && s.stride == 1 && s.KH <= 5 ? 8 : rows >= 4 ? 4 : 2;
    ProfScope prof("simt_conv_depthwise", stream);
    const SimtArgs a = make_args(s, eps);
    const int gx = (s.Wo + kDwsXO - 1) / kDwsXO;
    const int nrr = (s.Ho + R - 1) / R;
    const long long units = (long long)s.N * s.CI * nrr;
    // whole row units per warp when a row's groups fit in one warp
    const int rpw = gx <= 32 ? 32 / gx : 0;
    const long long threads = rpw > 0 ? (units + rpw - 1) / rpw * 32 : units * gx;
    const long long blocks = (threads + 127) / 128;
    if (threads + 128 >= (1ll << 31) || units >= (1ll << 31)) return cudaErrorInvalidValue;
    const int ve = s.in_dt == BIGEMM_F32 ? 4 : 8;
    // the vector paths take their halos from neighbouring lanes: 16-byte
    // vectors when rows are 16-byte aligned, else 4-byte words when they are
    // 4-byte aligned
    const size_t esz = dtype_size(s.in_dt);
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x);
    const int vec_in = rpw == 0                                    ? 0
                       : (s.W % ve == 0 && (xa & 15) == 0)          ? 1
                       : ((s.W * esz) % 4 == 0 && (xa & 3) == 0) ? 2
                                                                   : 0;
    const int vo = s.out_dt == BIGEMM_F32 ? 4 : 8;
    const int vec_out = (s.Wo % vo == 0) && ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    auto go = [&](auto kern) {
        return launch_pdl(kern, dim3((unsigned)blocks), dim3(128), 0, stream, a, gx, nrr, rpw,
                          make_fastdiv((uint32_t)gx), make_fastdiv((uint32_t)nrr),
                          make_fastdiv((uint32_t)s.CI), x, w, bias, out, vec_in, vec_out);
    };
#define BIGEMM_DWK(DTV, KV, SV)                                                           \
    if (s.KH == KV && s.stride == SV) {                                                   \
        if (R == 8) return go(dw_stream_kernel<DTV, KV, SV, (SV == 1 && KV <= 5) ? 8 : 4>); \
        if (R == 4) return go(dw_stream_kernel<DTV, KV, SV, 4>);                          \
        return go(dw_stream_kernel<DTV, KV, SV, 2>);                                      \
    }
#define BIGEMM_DWS(DTV)                                                                   \
    BIGEMM_DWK(DTV, 3, 1) BIGEMM_DWK(DTV, 3, 2) BIGEMM_DWK(DTV, 5, 1)                     \
    BIGEMM_DWK(DTV, 5, 2) BIGEMM_DWK(DTV, 7, 1) BIGEMM_DWK(DTV, 7, 2)                     \
    return cudaErrorInvalidValue;
    if (s.in_dt == BIGEMM_F32) { BIGEMM_DWS(BIGEMM_F32) }
    if (s.in_dt == BIGEMM_F16) { BIGEMM_DWS(BIGEMM_F16) }
    BIGEMM_DWS(BIGEMM_BF16)
#undef BIGEMM_DWS
#undef BIGEMM_DWK
}



}  // namespace bigemm
