// pack.cu -- operand layouts for the implicit GEMM, and the split-K reduction.
//
//  pack_nhwc     data [N][C][H*W] -> [N][H*W][Ch] (channels innermost, zero
//                padded to Ch), so that every (ry, rx) tap of a pixel box is one
//                TMA box whose innermost coordinate is a channel offset (always
//                16-byte aligned) and whose spatial coordinates may be negative
//                (zero fill = the conv's inlined padding).
//  pack_operands the same transpose into a per-image grid [Hop][Wop] whose
//                pixel (yo, xo) takes input pixel (s*yo, s*xo), zero where that
//                lies outside the image -- plus the kernel re-layout, in one
//                launch.  Hop = H, Wop = W, s = 1 is the plain copy; Hop > H
//                appends zero rows below each image (images stacked with a
//                padding gap, read by one tensor map over all rows); s > 1
//                keeps only the pixels a strided 1x1 conv reads.
//  weights       kernel [CO][CI][KH*KW] -> [CO][KH*KW][cip]: the reduction
//                order (ry, rx, ci) of the packed data, channels zero padded to
//                whole 128-byte K blocks (part of pack_operands).
//  splitk_reduce out = op(sum_s ws[s] + bias[f]) with the K slices added in
//                index order (deterministic), then rounded to the output type.
#include <algorithm>
#include <climits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace bigemm {

namespace {

template <typename T>
__global__ void pack_nhwc_kernel(const T *__restrict__ x, T *__restrict__ xh, int C, int HW,
                                 int Ch)
{
    griddep_enter();
    __shared__ T tile[32][33];
    const int n = blockIdx.z;
    const int p0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
    const T *xs = x + (size_t)n * C * HW;
    T *xd = xh + (size_t)n * HW * Ch;
    for (int i = threadIdx.y; i < 32; i += 8) {
        const int c = c0 + i, p = p0 + threadIdx.x;
        T v;
        if (c < C && p < HW)
            v = xs[(size_t)c * HW + p];
        else
            v = T(0);
        tile[i][threadIdx.x] = v;
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
        const int p = p0 + i, c = c0 + threadIdx.x;
        if (p < HW && c < Ch) xd[(size_t)p * Ch + c] = tile[threadIdx.x][i];
    }
}

// 16-byte vectors on both sides: a tile of TILE channels x TILE pixels is read
// as rows of pixels and written as rows of channels.  The odd row pitch keeps
// the column reads of the transpose free of bank conflicts.
template <typename T>
__global__ void __launch_bounds__(256) pack_nhwc_vec_kernel(const T *__restrict__ x,
                                                            T *__restrict__ xh, int C, int HW,
                                                            int Ch)
{
    griddep_enter();
    constexpr int VEC = 16 / sizeof(T);
    constexpr int TILE = 8 * VEC;
    __shared__ T tile[TILE][TILE + 1];
    const int n = blockIdx.z;
    const int p0 = blockIdx.x * TILE, c0 = blockIdx.y * TILE;
    const T *xs = x + (size_t)n * C * HW;
    T *xd = xh + (size_t)n * HW * Ch;
    for (int v = threadIdx.x; v < TILE * 8; v += blockDim.x) {
        const int cr = v >> 3, pv = v & 7;
        const int c = c0 + cr, pix = p0 + pv * VEC;
        union {
            uint4 u;
            T e[VEC];
        } val;
        val.u = make_uint4(0, 0, 0, 0);
        if (c < C && pix < HW) val.u = *reinterpret_cast<const uint4 *>(xs + (size_t)c * HW + pix);
#pragma unroll
        for (int i = 0; i < VEC; ++i) tile[cr][pv * VEC + i] = val.e[i];
    }
    __syncthreads();
    for (int v = threadIdx.x; v < TILE * 8; v += blockDim.x) {
        const int pr = v >> 3, cv = v & 7;
        const int pix = p0 + pr, c = c0 + cv * VEC;
        if (pix < HW && c < Ch) {
            union {
                uint4 u;
                T e[VEC];
            } val;
#pragma unroll
            for (int i = 0; i < VEC; ++i) val.e[i] = tile[cv * VEC + i][pr];
            *reinterpret_cast<uint4 *>(xd + (size_t)pix * Ch + c) = val.u;
        }
    }
}

// Shared memory of a pack_operands block: a data tile, or the weight buffer
// (16 KB, so that a run of input channels x taps of one output channel fits).
constexpr int kPackSmemBytes = 16384;

// The kernel re-layout [CO][CI][KHKW] -> [CO][KHKW][cip] by blocks
// first, first + nblocks, ...: each work item is one output channel f and a
// run of cc input channels, whose cc * KHKW source elements are contiguous.
// They are read coalesced into the shared buffer `buf` (cap elements) and
// written back as KHKW runs of cc channels, zero past CI.
template <typename T>
__device__ __forceinline__ void pack_weight_part(const T *__restrict__ w, T *__restrict__ wp,
                                                 int CO, int CI, int KHKW, int cip, int first,
                                                 int nblocks, T *buf, int cap)
{
    int cc = cap / KHKW;
    if (cc >= 32) cc &= ~31;
    if (cc < 1) {   // a kernel too large for the buffer: element by element
        const long long total = (long long)CO * KHKW * cip;
        const long long nthreads = (long long)nblocks * blockDim.x;
        for (long long i = (long long)first * blockDim.x + threadIdx.x; i < total; i += nthreads) {
            const int c = (int)(i % cip);
            const long long r = i / cip;
            const int t = (int)(r % KHKW);
            const int f = (int)(r / KHKW);
            wp[i] = c < CI ? w[((size_t)f * CI + c) * KHKW + t] : T(0);
        }
        return;
    }
    const int runs = (cip + cc - 1) / cc;
    const long long items = (long long)CO * runs;
    for (long long it = first; it < items; it += nblocks) {
        const int f = (int)(it / runs);
        const int c0 = (int)(it - (long long)f * runs) * cc;
        const int nc = min(cc, CI - c0);   // source channels in this run (may be <= 0)
        const T *src = w + ((size_t)f * CI + c0) * KHKW;
        const int nsrc = nc > 0 ? nc * KHKW : 0;
        constexpr int VEC = 16 / sizeof(T);
        if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && nsrc % VEC == 0) {
            const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
            for (int i = threadIdx.x; i < nsrc / VEC; i += blockDim.x)
                reinterpret_cast<uint4 *>(buf)[i] = __ldg(s4 + i);
        } else {
            for (int i = threadIdx.x; i < nsrc; i += blockDim.x) buf[i] = __ldg(src + i);
        }
        __syncthreads();
        const int wc = min(cc, cip - c0);  // destination channels in this run
        T *dst = wp + (size_t)f * KHKW * cip + c0;
        if (wc % VEC == 0 && (cip * sizeof(T)) % 16 == 0 && ((c0 * sizeof(T)) & 15) == 0) {
            // runs of VEC channels of one tap per 16-byte store
            const int wv = wc / VEC;
            for (int i = threadIdx.x; i < KHKW * wv; i += blockDim.x) {
                const int t = i / wv, c = (i - t * wv) * VEC;
                union {
                    uint4 u;
                    T e[VEC];
                } o;
                if (c + VEC <= nc) {
                    // all VEC source channels present: a strided gather, no tests
                    const T *col = buf + c * KHKW + t;
#pragma unroll
                    for (int j = 0; j < VEC; ++j) o.e[j] = col[j * KHKW];
                } else {
#pragma unroll
                    for (int j = 0; j < VEC; ++j) o.e[j] = c + j < nc ? buf[(c + j) * KHKW + t] : T(0);
                }
                *reinterpret_cast<uint4 *>(dst + (size_t)t * cip + c) = o.u;
            }
        } else {
            for (int i = threadIdx.x; i < KHKW * wc; i += blockDim.x) {
                const int t = i / wc, c = i - t * wc;
                dst[(size_t)t * cip + c] = c < nc ? buf[c * KHKW + t] : T(0);
            }
        }
        __syncthreads();
    }
}

// Blocks [0, zblocks) of a zero-fill part: n floats at z (16-byte aligned) set to 0.
__device__ __forceinline__ void zero_part(float *__restrict__ z, long long n, int blk, int nblk)
{
    const long long nv = n >> 2;
    uint4 *zv = reinterpret_cast<uint4 *>(z);
    for (long long i = (long long)blk * blockDim.x + threadIdx.x; i < nv;
         i += (long long)nblk * blockDim.x)
        zv[i] = make_uint4(0, 0, 0, 0);
    if (blk == 0 && threadIdx.x < (n & 3)) z[(nv << 2) + threadIdx.x] = 0.f;
}

// Both operands in one launch: blocks [0, wblocks) re-lay out the kernel
// (first, so that this work overlaps the data tiles), the last zblocks blocks
// zero zn floats at z, and the blocks between transpose data tiles (tile index
// flattened as (pixel tile, channel tile, image)).  Output pixel p of an image
// copies input pixel p when p < HWi and is zero up to HWo (the zero rows below
// a stacked image).  wblocks = 0: no kernel re-layout.
//
// Large planes (HWi a whole number of 16-byte runs): a data tile is 128
// pixels x 128 bytes of channels.  Each thread keeps four 16-byte loads in
// flight (four channel rows of one pixel run), regroups them into 32-bit
// words -- channel pairs of one pixel for 16-bit types, single channels for
// fp32 -- in a [128 pixels][32 words] shared array whose 16-byte chunks are
// XOR-swizzled by pixel group, and the block then writes each pixel's 128
// bytes of channels as 16-byte stores.  (Measured on the 64-channel 56 x 56
// fp16 layer: 83% of the copy bandwidth, against 65% for a 64 x 64 tile
// transposed element by element.)
template <typename T>
__global__ void __launch_bounds__(256) pack_operands_kernel(const T *__restrict__ x,
                                                            T *__restrict__ xh, int C, int HWi,
                                                            int HWo, int Ch, int ptiles,
                                                            int ctiles, int wblocks,
                                                            const T *__restrict__ w,
                                                            T *__restrict__ wp, int CO, int CI,
                                                            int KHKW, int cip, float *z,
                                                            long long zn, int zblocks)
{
    griddep_enter();
    constexpr int E = sizeof(T);
    constexpr int VEC = 16 / E;          // elements per 16 bytes
    constexpr int TP = 128;              // pixels per tile
    constexpr int TC = 128 / E;          // channels per tile
    constexpr int PV = TP / VEC;         // 16-byte pixel runs per channel row
    static_assert(PV * (TC / 4) == 256, "one thread per (pixel run, channel quad)");
    static_assert(TP * 32 * 4 == kPackSmemBytes, "the word array is the block's buffer");
    __shared__ __align__(16) uint32_t wsm[TP * 32];
    if ((int)blockIdx.x < wblocks) {
        pack_weight_part(w, wp, CO, CI, KHKW, cip, (int)blockIdx.x, wblocks,
                         reinterpret_cast<T *>(wsm), (int)(kPackSmemBytes / E));
        return;
    }
    if ((int)blockIdx.x >= (int)gridDim.x - zblocks) {
        zero_part(z, zn, (int)blockIdx.x - ((int)gridDim.x - zblocks), zblocks);
        return;
    }
    const int t = (int)blockIdx.x - wblocks;
    const int pt = t % ptiles, r = t / ptiles;
    const int ct = r % ctiles, n = r / ctiles;
    const int p0 = pt * TP, c0 = ct * TC;
    const T *xs = x + (size_t)n * C * HWi;
    T *xd = xh + (size_t)n * HWo * Ch;
    const int pv = threadIdx.x % PV, cq = threadIdx.x / PV;
    const int pix = p0 + pv * VEC;
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int c = c0 + cq * 4 + k;
        v[k] = make_uint4(0, 0, 0, 0);
        if (c < C && pix < HWi) v[k] = __ldg(reinterpret_cast<const uint4 *>(xs + (size_t)c * HWi + pix));
    }
    if (E == 2) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int p = pv * 8 + i;
            const uint32_t sw = (uint32_t)((p >> 3) & 7) << 2;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const uint32_t a = (&v[2 * m].x)[i >> 1], b = (&v[2 * m + 1].x)[i >> 1];
                wsm[p * 32 + ((uint32_t)(cq * 2 + m) ^ sw)] = __byte_perm(a, b, (i & 1) ? 0x7632 : 0x5410);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int p = pv * 4 + i;
            const uint32_t sw = (uint32_t)((p >> 3) & 7) << 2;
#pragma unroll
            for (int k = 0; k < 4; ++k) wsm[p * 32 + ((uint32_t)(cq * 4 + k) ^ sw)] = (&v[k].x)[i];
        }
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < TP * 8 / 256; ++it) {
        const int q = it * 256 + (int)threadIdx.x;
        const int p = q >> 3, kc = q & 7;
        const int op = p0 + p, c = c0 + kc * VEC;
        if (op < HWo && c < Ch) {
            const uint32_t ph = (uint32_t)(kc ^ ((p >> 3) & 7));
            *reinterpret_cast<uint4 *>(xd + (size_t)op * Ch + c) =
                *reinterpret_cast<const uint4 *>(&wsm[p * 32 + ph * 4]);
        }
    }
}

// Small planes (HWi <= kPlaneMax): a data tile is the whole plane of one image
// for ipb x 128 bytes of channels (ipb channel tiles, ipb * HWi <= kPlaneMax),
// which is one contiguous run of the input.  The run is copied to shared
// memory (16-byte loads where it is aligned), then each thread writes 16-byte
// channel runs of output pixels gathered from the plane rows.  Tile index
// flattened as (channel group, image).  (Several tiles per block: each block
// keeps more bytes in flight and the grid fits one wave; one 128-byte tile per
// block left the 512-channel 7 x 7 layer's pack at half the copy bandwidth.)
constexpr int kPlaneMax = 256;
// the whole-plane kernels' shared buffer (128 bytes of channels x kPlaneMax
// pixels), which their weight blocks use whole: twice the channel run of the
// other kernels, so a large kernel takes half the weight blocks
constexpr int kPlaneBufBytes = 128 * kPlaneMax;

template <typename T>
__global__ void __launch_bounds__(256) pack_plane_kernel(const T *__restrict__ x,
                                                         T *__restrict__ xh, int C, int HWi,
                                                         int HWo, int Ch, int cgroups, int ipb,
                                                         int wblocks,
                                                         const T *__restrict__ w,
                                                         T *__restrict__ wp, int CO, int CI,
                                                         int KHKW, int cip, float *z,
                                                         long long zn, int zblocks)
{
    griddep_enter();
    constexpr int E = sizeof(T);
    constexpr int VEC = 16 / E;
    constexpr int TC = 128 / E;
    constexpr int KC = TC / VEC;         // 16-byte channel runs per pixel (8)
    static_assert(TC * kPlaneMax * E == kPlaneBufBytes, "the weight blocks use the whole buffer");
    __shared__ __align__(16) T sp[TC * kPlaneMax];
    if ((int)blockIdx.x < wblocks) {
        pack_weight_part(w, wp, CO, CI, KHKW, cip, (int)blockIdx.x, wblocks, sp,
                         (int)(kPlaneBufBytes / E));
        return;
    }
    if ((int)blockIdx.x >= (int)gridDim.x - zblocks) {
        zero_part(z, zn, (int)blockIdx.x - ((int)gridDim.x - zblocks), zblocks);
        return;
    }
    const int t = (int)blockIdx.x - wblocks;
    const int g = t % cgroups, n = t / cgroups;
    const int c0 = g * ipb * TC;
    const int nc = min(ipb * TC, C - c0);  // channels of the input in this group (<= 0: padding)
    const int kcb = ipb * KC;              // 16-byte channel runs per pixel of the group
    const T *src = x + ((size_t)n * C + c0) * HWi;
    const int cnt = nc > 0 ? nc * HWi : 0;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0 && cnt % VEC == 0) {
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
        for (int i = threadIdx.x; i < cnt / VEC; i += blockDim.x)
            reinterpret_cast<uint4 *>(sp)[i] = __ldg(s4 + i);
    } else {
        for (int i = threadIdx.x; i < cnt; i += blockDim.x) sp[i] = __ldg(src + i);
    }
    __syncthreads();
    T *xd = xh + (size_t)n * HWo * Ch;
    for (int q = threadIdx.x; q < HWo * kcb; q += blockDim.x) {
        // q = (tile, pixel, run): the eight lanes of a pixel gather eight
        // channel rows from distinct bank groups, as with one tile per block
        const int r = q / KC, kt = r / HWo;
        const int p = r - kt * HWo, k = kt * KC + (q - r * KC);
        const int c = c0 + k * VEC;
        if (c >= Ch) continue;
        union {
            uint4 u;
            T e[VEC];
        } o;
        if (p < HWi && (k + 1) * VEC <= nc) {
            // a pixel of the plane with all VEC channels present: one strided
            // gather down the channel planes, no per-element tests
            const T *col = sp + k * VEC * HWi + p;
#pragma unroll
            for (int j = 0; j < VEC; ++j) o.e[j] = col[j * HWi];
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const int ch = k * VEC + j;
                o.e[j] = (p < HWi && ch < nc) ? sp[ch * HWi + p] : T(0);
            }
        }
        *reinterpret_cast<uint4 *>(xd + (size_t)p * Ch + c) = o.u;
    }
}

// Subsampling over small planes (Hop * Wop <= kPlaneMax, input rows a whole
// number of 8-byte words): output pixel (yo, xo) of an image takes input pixel
// (s*yo, s*xo), zero past the image.  A data tile is the whole output plane of
// one image for 128 bytes of channels: the threads read the input rows s*yo
// as 8-byte words (the rows the conv skips are never read), keep the pixels
// at multiples of s in shared memory as [channel][output pixel] with an odd
// row pitch (so that the gather below reads eight channel rows from eight
// bank groups), and write 16-byte channel runs per output pixel as the plane
// kernel does.  Each word finds its first output column with one
// multiply-high division (a per-element remainder test had made the kernel
// ALU-bound).  Tile index flattened as (channel tile, image).
template <typename T>
__global__ void __launch_bounds__(256) pack_subplane_kernel(const T *__restrict__ x,
                                                            T *__restrict__ xh, int C, int H,
                                                            int W, int Hop, int Wop, int s,
                                                            int Ch, int ctiles, int wblocks,
                                                            FastDiv fd_wpr, FastDiv fd_rows,
                                                            FastDiv fd_wop, FastDiv fd_s,
                                                            const T *__restrict__ w,
                                                            T *__restrict__ wp, int CO, int CI,
                                                            int KHKW, int cip, float *z,
                                                            long long zn, int zblocks)
{
    griddep_enter();
    constexpr int E = sizeof(T);
    constexpr int VEC = 16 / E;
    constexpr int TC = 128 / E;
    constexpr int KC = TC / VEC;
    constexpr int G = 8 / E;             // elements per 8-byte word
    // item indices are split with multiply-high divisions by the launch's fixed
    // row length, row count and output width (runtime divisions dominated)
    static_assert(TC * kPlaneMax * E == kPlaneBufBytes, "the weight blocks use the whole buffer");
    __shared__ __align__(16) T sp[TC * kPlaneMax];
    if ((int)blockIdx.x < wblocks) {
        pack_weight_part(w, wp, CO, CI, KHKW, cip, (int)blockIdx.x, wblocks, sp,
                         (int)(kPlaneBufBytes / E));
        return;
    }
    if ((int)blockIdx.x >= (int)gridDim.x - zblocks) {
        zero_part(z, zn, (int)blockIdx.x - ((int)gridDim.x - zblocks), zblocks);
        return;
    }
    const int t = (int)blockIdx.x - wblocks;
    const int ct = t % ctiles, n = t / ctiles;
    const int c0 = ct * TC;
    const int nc = min(TC, C - c0);
    const int hwo = Hop * Wop;
    const int pitch = ((hwo | 1) <= kPlaneMax) ? (hwo | 1) : hwo;   // shared row pitch
    const int wpr = W / G;                               // words per input row
    // rows actually read: s*yo < H
    const int rows = min(Hop, (H + s - 1) / s);
    const long long hw = (long long)H * W;
    const int items = (nc > 0 ? nc : 0) * rows * wpr;    // (channel, output row, word)
    // eight words per thread in flight, then their pixels to shared memory; the
    // first pass keeps each word's shared-memory row offset and first column
    constexpr int UN = 8;
    for (int i0 = threadIdx.x; i0 < items; i0 += UN * (int)blockDim.x) {
        uint2 u[UN];
        int off[UN], x0s[UN];
#pragma unroll
        for (int k = 0; k < UN; ++k) {
            const int i = i0 + k * (int)blockDim.x;
            off[k] = -1;
            x0s[k] = 0;
            if (i < items) {
                uint32_t wd, yo;
                const uint32_t r = fd_divmod((uint32_t)i, fd_wpr, &wd);
                const uint32_t c = fd_divmod(r, fd_rows, &yo);
                u[k] = __ldg(reinterpret_cast<const uint2 *>(
                                 x + ((size_t)n * C + c0 + c) * hw + (size_t)(s * yo) * W) + wd);
                off[k] = (int)c * pitch + (int)yo * Wop;
                x0s[k] = (int)wd * G;
            }
        }
#pragma unroll
        for (int k = 0; k < UN; ++k) {
            if (off[k] < 0) continue;
            const T *e = reinterpret_cast<const T *>(&u[k]);
            T *dst = sp + off[k];
            const int x0 = x0s[k];
            if (s == 2) {
                // a word starts at an even column: its even pixels are outputs x0/2, x0/2 + 1, ...
                const int xo0 = x0 >> 1;
#pragma unroll
                for (int j = 0; j < G / 2; ++j)
                    if (xo0 + j < Wop) dst[xo0 + j] = e[2 * j];
            } else {
                // output columns xo0, xo0 + 1, ... read pixels (xo0 + j) * s of this word
                const int xo0 = (int)fd_div((uint32_t)(x0 + s - 1), fd_s);
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const int d = (xo0 + j) * s - x0;
                    if (d < G && xo0 + j < Wop) {
                        T val = e[0];
#pragma unroll
                        for (int g = 1; g < G; ++g)
                            if (d == g) val = e[g];
                        dst[xo0 + j] = val;
                    }
                }
            }
        }
    }
    __syncthreads();
    T *xd = xh + (size_t)n * hwo * Ch;
    for (int q = threadIdx.x; q < hwo * KC; q += blockDim.x) {
        const int pix = q / KC, k = q - pix * KC;
        const int c = c0 + k * VEC;
        if (c >= Ch) continue;
        uint32_t xo;
        const int yo = (int)fd_divmod((uint32_t)pix, fd_wop, &xo);
        const bool inside = yo < rows && (int)xo * s < W;
        union {
            uint4 u;
            T e[VEC];
        } o;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const int ch = k * VEC + j;
            o.e[j] = (inside && ch < nc) ? sp[ch * pitch + pix] : T(0);
        }
        *reinterpret_cast<uint4 *>(xd + (size_t)pix * Ch + c) = o.u;
    }
}

// The general form: output pixel (yo, xo) of the [Hop][Wop] grid takes input
// pixel (s*yo, s*xo), zero outside the image.  Element reads (any alignment,
// any stride), 16-byte channel-row writes.
template <typename T>
__global__ void __launch_bounds__(256) pack_remap_kernel(const T *__restrict__ x,
                                                         T *__restrict__ xh, int C, int H, int W,
                                                         int Hop, int Wop, int s, int Ch,
                                                         int ptiles, int ctiles, int wblocks,
                                                         const T *__restrict__ w,
                                                         T *__restrict__ wp, int CO, int CI,
                                                         int KHKW, int cip, float *z,
                                                         long long zn, int zblocks)
{
    griddep_enter();
    constexpr int VEC = 16 / sizeof(T);
    constexpr int TILE = 8 * VEC;
    static_assert(256 % TILE == 0, "a thread keeps one pixel column");
    static_assert(TILE * (TILE + 1) * sizeof(T) <= kPackSmemBytes, "tile fits the buffer");
    __shared__ __align__(16) T sbuf[kPackSmemBytes / sizeof(T)];
    T(*tile)[TILE + 1] = reinterpret_cast<T(*)[TILE + 1]>(sbuf);
    if ((int)blockIdx.x < wblocks) {
        pack_weight_part(w, wp, CO, CI, KHKW, cip, (int)blockIdx.x, wblocks, sbuf,
                         (int)(kPackSmemBytes / sizeof(T)));
        return;
    }
    if ((int)blockIdx.x >= (int)gridDim.x - zblocks) {
        zero_part(z, zn, (int)blockIdx.x - ((int)gridDim.x - zblocks), zblocks);
        return;
    }
    {
        const int t = (int)blockIdx.x - wblocks;
        const int pt = t % ptiles, r = t / ptiles;
        const int ct = r % ctiles, n = r / ctiles;
        const int p0 = pt * TILE, c0 = ct * TILE;
        const long long hwi = (long long)H * W, hwo = (long long)Hop * Wop;
        const T *xs = x + (size_t)n * C * hwi;
        T *xd = xh + (size_t)n * hwo * Ch;
        const int pc = threadIdx.x % TILE;
        const long long pix = (long long)p0 + pc;
        long long src = -1;
        if (pix < hwo) {
            const long long yo = pix / Wop, xo = pix - yo * Wop;
            const long long yi = yo * s, xi = xo * s;
            if (yi < H && xi < W) src = yi * W + xi;
        }
        // all of the thread's loads first, so that they are in flight together
        constexpr int kRows = 256 / TILE, kPer = TILE / kRows;
        T val[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int c = c0 + threadIdx.x / TILE + k * kRows;
            val[k] = (c < C && src >= 0) ? __ldg(xs + (size_t)c * hwi + src) : T(0);
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) tile[threadIdx.x / TILE + k * kRows][pc] = val[k];
        __syncthreads();
        for (int v = threadIdx.x; v < TILE * 8; v += blockDim.x) {
            const int pr = v >> 3, cv = v & 7;
            const long long op = (long long)p0 + pr;
            const int c = c0 + cv * VEC;
            if (op < hwo && c < Ch) {
                union {
                    uint4 u;
                    T e[VEC];
                } val;
#pragma unroll
                for (int i = 0; i < VEC; ++i) val.e[i] = tile[cv * VEC + i][pr];
                *reinterpret_cast<uint4 *>(xd + (size_t)op * Ch + c) = val.u;
            }
        }
    }
}

__device__ __forceinline__ float epi_apply(int epi, float acc, float b, float eps)
{
    switch (epi) {
    case BIGEMM_EPI_NONE: return acc;
    case BIGEMM_EPI_BIAS: return acc + b;
    case BIGEMM_EPI_BIAS_EXP: return expf(acc + b);
    case BIGEMM_EPI_BIAS_RSQRT: return rsqrtf(acc + b + eps);
    case BIGEMM_EPI_BIAS_RELU: return fmaxf(acc + b, 0.f);
    default: return 1.0f / (acc + b);
    }
}

template <typename TO>
__device__ __forceinline__ TO to_out(float v);
template <>
__device__ __forceinline__ float to_out<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half to_out<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float v)
{
    return __float2bfloat16_rn(v);
}

template <typename TO>
__global__ void splitk_reduce_kernel(const float *__restrict__ ws, int split, long long elems,
                                     int CO, int HoWo, int epi, const float *__restrict__ bias,
                                     float eps, TO *__restrict__ out)
{
    griddep_enter();
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < elems;
         i += (long long)gridDim.x * blockDim.x) {
        float s = ws[i];
        for (int k = 1; k < split; ++k) s += ws[(long long)k * elems + i];
        const int f = (int)((i / HoWo) % CO);
        out[i] = to_out<TO>(epi_apply(epi, s, epi ? bias[f] : 0.f, eps));
    }
}

int grid_for(long long work, int per_block)
{
    long long g = (work + per_block - 1) / per_block;
    DeviceState *ds = device_state();
    const long long cap = (long long)(ds ? ds->sm_count : 148) * 16;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_pack_nhwc(const void *x, void *xh, int N, int C, int HW, int Ch, int dt,
                             cudaStream_t stream)
{
    ProfScope prof("pack_nhwc", stream);
    const int vec = (int)(16 / dtype_size(dt));
    const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(xh)) & 15) == 0;
    if (aligned && HW % vec == 0 && Ch % vec == 0) {
        const int tile = 8 * vec;
        dim3 g((HW + tile - 1) / tile, (Ch + tile - 1) / tile, N);
        if (dtype_size(dt) == 4)
            return launch_pdl(pack_nhwc_vec_kernel<uint32_t>, g, dim3(256), 0, stream,
                              static_cast<const uint32_t *>(x), static_cast<uint32_t *>(xh), C, HW, Ch);
        return launch_pdl(pack_nhwc_vec_kernel<uint16_t>, g, dim3(256), 0, stream,
                          static_cast<const uint16_t *>(x), static_cast<uint16_t *>(xh), C, HW, Ch);
    }
    dim3 grid((HW + 31) / 32, (Ch + 31) / 32, N), block(32, 8);
    if (dtype_size(dt) == 4)
        return launch_pdl(pack_nhwc_kernel<uint32_t>, grid, block, 0, stream,
                          static_cast<const uint32_t *>(x), static_cast<uint32_t *>(xh), C, HW, Ch);
    return launch_pdl(pack_nhwc_kernel<uint16_t>, grid, block, 0, stream,
                      static_cast<const uint16_t *>(x), static_cast<uint16_t *>(xh), C, HW, Ch);
}

cudaError_t launch_pack_operands(const void *x, void *xh, int N, int C, int H, int W, int Hop,
                                 int Wop, int s, int Ch, const void *w, void *wp, int CO, int CI,
                                 int KHKW, int cip, int dt, cudaStream_t stream, float *zero,
                                 long long zero_elems)
{
    const int vec = (int)(16 / dtype_size(dt));
    if (Ch % vec || (reinterpret_cast<uintptr_t>(xh) & 15)) return cudaErrorInvalidValue;
    const bool aligned = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    const long long hwi = (long long)H * W, hwo = (long long)Hop * Wop;
    // pixel p of the output is pixel p of the input (or zero below it)
    const bool linear = s == 1 && Wop == W && Hop >= H;
    // the subsampled copy of small planes, rows read as 8-byte words
    const bool subplane = !linear && s > 1 && hwo <= kPlaneMax &&
                          ((long long)W * dtype_size(dt)) % 8 == 0 &&
                          (reinterpret_cast<uintptr_t>(x) & 7) == 0;
    const int kind = (linear && hwi <= kPlaneMax) ? 0                                  // plane
                     : (linear && aligned && hwi % vec == 0 && hwo % vec == 0) ? 1    // rows
                     : subplane ? 3                                                    // subsampled planes
                                : 2;                                                   // remap
    const int tile = 8 * vec;                          // remap tiles: tile x tile
    const long long tc = 128 / (long long)dtype_size(dt);   // plane / rows tiles: 128 B of channels
    const long long ptiles = (kind == 0 || kind == 3) ? 1 : kind == 1 ? (hwo + 127) / 128 : (hwo + tile - 1) / tile;
    const long long ctiles = kind == 2 ? (Ch + tile - 1) / tile : (Ch + tc - 1) / tc;
    // whole planes: ipb channel tiles per block, as many as the buffer holds
    // while every SM still gets two data blocks, then as few as give the same
    // number of groups (balanced groups)
    long long ipb = 1;
    if (kind == 0) {
        DeviceState *ds = device_state();
        const long long want = 2ll * (ds ? ds->sm_count : 148);
        const long long maxb = std::max<long long>(1, std::min<long long>(kPlaneMax / hwi, ctiles));
        for (long long b = maxb; b > 1; --b)
            if ((long long)N * ((ctiles + b - 1) / b) >= want) {
                ipb = b;
                break;
            }
        const long long groups = (ctiles + ipb - 1) / ipb;
        while (ipb > 1 && (ctiles + ipb - 2) / (ipb - 1) == groups) --ipb;
    }
    const long long cgroups = (ctiles + ipb - 1) / ipb;
    const long long data_blocks = ptiles * (kind == 0 ? cgroups : ctiles) * N;
    // weight blocks: one per (output channel, channel run) item of pack_weight_part;
    // none when w is null (the conv reads the caller's kernel as it is)
    const long long cap = ((kind == 0 || kind == 3) ? kPlaneBufBytes : kPackSmemBytes) /
                          (long long)dtype_size(dt);
    long long cc = cap / KHKW;
    if (cc >= 32) cc &= ~31ll;
    const long long witems = cc >= 1 ? (long long)CO * ((cip + cc - 1) / cc)
                                     : ((long long)CO * KHKW * cip + 255) / 256;
    const long long wblocks = w ? std::max<long long>(1, std::min<long long>(witems, 2048)) : 0;
    if (zero && (reinterpret_cast<uintptr_t>(zero) & 15)) return cudaErrorInvalidValue;
    const long long zblocks =
        zero && zero_elems > 0 ? std::min<long long>((zero_elems / 4 + 255) / 256 + 1, 1024) : 0;
    if (data_blocks + wblocks + zblocks > INT32_MAX || hwo > INT32_MAX) return cudaErrorInvalidValue;
    ProfScope prof("pack_operands", stream);
    const int grid = (int)(data_blocks + wblocks + zblocks);
    if (kind == 0) {
        if (dtype_size(dt) == 4)
            return launch_pdl(pack_plane_kernel<uint32_t>, dim3(grid), dim3(256), 0, stream,
                              static_cast<const uint32_t *>(x), static_cast<uint32_t *>(xh), C,
                              (int)hwi, (int)hwo, Ch, (int)cgroups, (int)ipb, (int)wblocks,
                              static_cast<const uint32_t *>(w), static_cast<uint32_t *>(wp), CO, CI,
                              KHKW, cip, zero, zero_elems, (int)zblocks);
        return launch_pdl(pack_plane_kernel<uint16_t>, dim3(grid), dim3(256), 0, stream,
                          static_cast<const uint16_t *>(x), static_cast<uint16_t *>(xh), C,
                          (int)hwi, (int)hwo, Ch, (int)cgroups, (int)ipb, (int)wblocks,
                          static_cast<const uint16_t *>(w), static_cast<uint16_t *>(wp), CO, CI,
                          KHKW, cip, zero, zero_elems, (int)zblocks);
    }
    if (kind == 3) {
        const FastDiv fd_wpr = make_fastdiv((uint32_t)(W * dtype_size(dt) / 8));
        const FastDiv fd_rows = make_fastdiv((uint32_t)std::min<long long>(Hop, (H + s - 1) / s));
        const FastDiv fd_wop = make_fastdiv((uint32_t)Wop);
        const FastDiv fd_s = make_fastdiv((uint32_t)s);
        if (dtype_size(dt) == 4)
            return launch_pdl(pack_subplane_kernel<uint32_t>, dim3(grid), dim3(256), 0, stream,
                              static_cast<const uint32_t *>(x), static_cast<uint32_t *>(xh), C, H, W,
                              Hop, Wop, s, Ch, (int)ctiles, (int)wblocks, fd_wpr, fd_rows, fd_wop, fd_s,
                              static_cast<const uint32_t *>(w), static_cast<uint32_t *>(wp), CO, CI,
                              KHKW, cip, zero, zero_elems, (int)zblocks);
        return launch_pdl(pack_subplane_kernel<uint16_t>, dim3(grid), dim3(256), 0, stream,
                          static_cast<const uint16_t *>(x), static_cast<uint16_t *>(xh), C, H, W,
                          Hop, Wop, s, Ch, (int)ctiles, (int)wblocks, fd_wpr, fd_rows, fd_wop, fd_s,
                          static_cast<const uint16_t *>(w), static_cast<uint16_t *>(wp), CO, CI,
                          KHKW, cip, zero, zero_elems, (int)zblocks);
    }
    if (kind == 1) {
        if (dtype_size(dt) == 4)
            return launch_pdl(pack_operands_kernel<uint32_t>, dim3(grid), dim3(256), 0, stream,
                              static_cast<const uint32_t *>(x), static_cast<uint32_t *>(xh), C,
                              (int)hwi, (int)hwo, Ch, (int)ptiles, (int)ctiles, (int)wblocks,
                              static_cast<const uint32_t *>(w), static_cast<uint32_t *>(wp), CO, CI,
                              KHKW, cip, zero, zero_elems, (int)zblocks);
        return launch_pdl(pack_operands_kernel<uint16_t>, dim3(grid), dim3(256), 0, stream,
                          static_cast<const uint16_t *>(x), static_cast<uint16_t *>(xh), C,
                          (int)hwi, (int)hwo, Ch, (int)ptiles, (int)ctiles, (int)wblocks,
                          static_cast<const uint16_t *>(w), static_cast<uint16_t *>(wp), CO, CI,
                          KHKW, cip, zero, zero_elems, (int)zblocks);
    }
    if (dtype_size(dt) == 4)
        return launch_pdl(pack_remap_kernel<uint32_t>, dim3(grid), dim3(256), 0, stream,
                          static_cast<const uint32_t *>(x), static_cast<uint32_t *>(xh), C, H, W,
                          Hop, Wop, s, Ch, (int)ptiles, (int)ctiles, (int)wblocks,
                          static_cast<const uint32_t *>(w), static_cast<uint32_t *>(wp), CO, CI,
                          KHKW, cip, zero, zero_elems, (int)zblocks);
    return launch_pdl(pack_remap_kernel<uint16_t>, dim3(grid), dim3(256), 0, stream,
                      static_cast<const uint16_t *>(x), static_cast<uint16_t *>(xh), C, H, W, Hop,
                      Wop, s, Ch, (int)ptiles, (int)ctiles, (int)wblocks,
                      static_cast<const uint16_t *>(w), static_cast<uint16_t *>(wp), CO, CI, KHKW,
                      cip, zero, zero_elems, (int)zblocks);
}

cudaError_t launch_splitk_reduce(const float *ws, int split, long long elems, int CO, int HoWo,
                                 int epi, const float *bias, float eps, void *out, int out_dt,
                                 cudaStream_t stream)
{
    ProfScope prof("splitk_reduce", stream);
    const int grid = grid_for(elems, 256);
    switch (out_dt) {
    case BIGEMM_F32:
        return launch_pdl(splitk_reduce_kernel<float>, dim3(grid), dim3(256), 0, stream, ws, split,
                          elems, CO, HoWo, epi, bias, eps, static_cast<float *>(out));
    case BIGEMM_F16:
        return launch_pdl(splitk_reduce_kernel<__half>, dim3(grid), dim3(256), 0, stream, ws, split,
                          elems, CO, HoWo, epi, bias, eps, static_cast<__half *>(out));
    default:
        return launch_pdl(splitk_reduce_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream, ws,
                          split, elems, CO, HoWo, epi, bias, eps, static_cast<__nv_bfloat16 *>(out));
    }
}

}  // namespace bigemm
