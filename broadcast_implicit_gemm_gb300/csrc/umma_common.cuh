// umma_common.cuh -- pieces shared by the implicit-GEMM conv kernels
// (umma_conv.cu: per-tap and direct operand modes; halo_conv.cu: halo mode):
// tile constants, the work-unit decode, and the epilogue warps that drain the
// TMEM accumulators into NCHW outputs.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace bigemm {
namespace {

constexpr int kThreads = 320;                  // producer, MMA, 8 epilogue warps
constexpr int kEpiWarps = 8;
constexpr int kTileM = 128;
constexpr int kRowBytes = 128;                  // one K block: a 128-byte swizzle row
constexpr int kABytes = kTileM * kRowBytes;     // 16 KB of A per stage

template <int BN>
struct Cfg {
    static constexpr int stages = BN <= 64 ? 8 : (BN <= 128 ? 6 : 4);
    static constexpr int b_bytes = BN * kRowBytes;
    static constexpr int ring = stages * (kABytes + b_bytes);
    static constexpr int staging = kEpiWarps * 4096;          // 4 KB output staging per epilogue warp
    static constexpr int bars = (2 * stages + 5) * 8;
    static constexpr int smem = ring + staging + bars + 16 + 16 + 1024;   // + alignment slack
    static constexpr uint32_t tmem_cols = (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                         : (2 * BN <= 256) ? 256 : 512;
};

struct Unit {
    int ct, pt, sp, kb0, kb1;
};

__device__ __forceinline__ Unit decode(const UmmaParams &p, int u)
{
    Unit w;
    uint32_t rem;
    const int r = (int)fd_divmod((uint32_t)u, p.fd_co, &rem);
    w.ct = (int)rem;
    w.sp = (int)fd_divmod((uint32_t)r, p.fd_pix, &rem);
    w.pt = (int)rem;
    w.kb0 = w.sp * p.kb_per_split;
    w.kb1 = min(p.k_blocks, w.kb0 + p.kb_per_split);
    return w;
}

constexpr int kMaxBoxes = 16;   // boxes per tile: 128 rows / at least 8 pixels per box (< 32 lanes)

// Epilogue warp groups that take alternate units (epilogue_warp): two for 16
// warps over 64-channel tiles, else one.  An accumulator is handed back by the
// NEPI / groups warps that drain it.
__host__ __device__ constexpr int epi_groups(int bn, int nepi) { return (nepi == 16 && bn == 64) ? 2 : 1; }

// Two floats rounded to nearest-even 16-bit values (fp16 or bf16), a in the
// low half: one packed conversion instruction for the pair.
__device__ __forceinline__ uint32_t pack2_16(float a, float b, bool f16)
{
    if (f16) {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// tcgen05.wait::ld that also names the loaded registers, so that no use of
// them can be scheduled above the wait.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Epilogue of one warp (warps 2 .. 2 + NEPI - 1 of the block).  NEPI = 8: two
// warps per TMEM lane quadrant, each taking every other 32-channel chunk of
// the accumulator; NEPI = 16: four per quadrant, each taking every fourth
// (BN = 128), or, with BN = 64 (two chunks), two groups of eight warps that
// take alternate units -- group g the block's units that use accumulator g --
// so that each warp drains half as many units (the per-unit work, not the
// chunks, paces 64-channel tiles); NEPI = 4: one warp per quadrant takes every
// chunk.  MT = 2:
// a unit is two 128-pixel M tiles stacked vertically (box_h = 32 rows of a
// halo tile), with accumulators at TMEM columns acc * 2BN and acc * 2BN + BN.
// BOXED: the tile's pixels are 2-D boxes (box_w x box_h) of one image (or of
// the stacked images); otherwise runs of box_w consecutive flattened pixels
// (the direct mode).
// STG: bytes of output staging per warp, used as STG / 2 KB buffers in turn.
// A store box is 2 KB: 32 channels x 32 pixels of 16-bit output, or 16
// channels of fp32 (the store map's box is 16 channels deep for 4-byte
// outputs), so a 32-channel chunk of fp32 leaves as two boxes.
// FORM narrows what the launch's tiles can need, so that the kernel carries
// only that code: 0 any output (every case decided at run time); 1 a 16-bit
// output written in place by TMA stores, with no epilogue op; 2 the same
// written from registers; 3 an fp32 output written in place by TMA stores,
// the epilogue op chosen at run time; 4 K slices added into an fp32 output
// (TMA reduce-add boxes or atomic adds), no op but the first slice's bias.
// (Measured on the 1x1 ResNet-50 layers: the general form's unused paths cost
// a third of the epilogue's time per tile.)
// PAIR: the block is one of a cluster's CTA pair sharing each MMA (M = 256);
// a pair runs units blockIdx.x / 2, + gridDim.x / 2, ..., this CTA holding
// pixel tile 2 * pt + rank of each, and the accumulator is handed back to the
// MMA thread of the pair's even CTA.
template <int BN, bool BOXED, int NEPI = kEpiWarps, int MT = 1, int STG = 4096, int FORM = 0,
          bool PAIR = false>
__device__ __forceinline__ void epilogue_warp(const UmmaParams &p, const CUtensorMap *map_c,
                                              uint32_t tmem_base, uint64_t *tfull,
                                              uint64_t *tempty, uint8_t *stage_out,
                                              volatile int *abort_flag, int warp, int lane,
                                              int box_px)
{
    // The warp owns TMEM lanes 32q..32q+31 (32 pixels of the tile) and the
    // chunks h, h + NEPI/4, ... of the BN accumulator columns.  Lane 0 waits
    // for the accumulator and shares the outcome, so the warp stays converged.
    // The load of the warp's next chunk is issued before the current one is
    // processed.  With TMA stores the warp stages its 32 pixels x 32 channels
    // in its own STG bytes of shared memory and lane 0 writes them as one box.
    static_assert(NEPI == 4 || NEPI == 8 || NEPI == 16, "one, two or four warps per TMEM lane quadrant");
    constexpr int kGroups = epi_groups(BN, NEPI);   // unit-interleaved warp groups
    static_assert(BN / 32 >= NEPI / 4 / kGroups, "every warp of a quadrant takes at least one chunk");
    static_assert(kGroups == 1 || (!PAIR && MT == 1), "unit groups: single blocks, one M tile");
    constexpr int kSplit = NEPI / 4 / kGroups;  // warps of a group sharing a quadrant
    constexpr int kChunks = BN / 32;            // 2, 4 or 8
    constexpr int kMine = kChunks / kSplit;     // chunks per warp
    const int q = warp & 3;                     // TMEM lane quadrant of this warp
    const int h4 = (warp - 2) >> 2;             // 0 .. NEPI/4 - 1
    const int grp = kGroups > 1 ? h4 / kSplit : 0;   // the warp's unit group
    const int h = h4 - grp * kSplit;            // which share of the chunks (0 when NEPI = 4)
    const int row = q * 32 + lane;              // tile row = pixel
    const int bi = row / box_px, bj = row - bi * box_px;
    const int wbi = (q * 32) / box_px;          // the warp's box
    const int wj0 = (q * 32) - wbi * box_px;    // its first pixel in the box
    const int bj_y = bj / p.box_w, bj_x = bj - bj_y * p.box_w;
    const int wj0_y = wj0 / p.box_w, wj0_x = wj0 - wj0_y * p.box_w;
    const long long howo = (long long)p.Ho * p.Wo;
    static_assert(FORM >= 0 && FORM <= 4, "output form");
    constexpr bool kPlain = FORM == 1 || FORM == 2;   // 16-bit, in place, no epilogue op
    constexpr bool kInPlace = FORM != 0;              // no workspace
    const bool red = FORM == 4 || (FORM == 0 && p.red_add);   // adds into an fp32 output
    const int ec = (FORM == 3 || FORM == 4) ? 4 : kPlain ? 2 : ((p.ws || p.out_dt == BIGEMM_F32) ? 4 : 2);
    const bool tma_out = (FORM == 1 || FORM == 3) ? true : FORM == 2 ? false : p.store_tma != 0;
    // 4-pixel register stores need the output itself (stored into, or added into
    // by K slices; not the workspace), planes of a whole number of 4-element
    // groups and an output base on a 4-element boundary
    const bool vec_static = (FORM == 0 || FORM == 2 || FORM == 4) && !tma_out && (kInPlace || !p.ws) &&
                            howo % 4 == 0 &&
                            (reinterpret_cast<uintptr_t>(p.out) & (uintptr_t)(4 * ec - 1)) == 0;
    uint8_t *wstage = stage_out + (warp - 2) * STG;
    constexpr int kNB = STG / 2048;             // 2 KB store buffers of the warp
    static_assert(kNB >= 1, "at least one 2 KB buffer per warp");
    int piece = 0;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    // with unit groups, group g takes the block's units g, g + 2, ... (in the
    // block's order), all of which use accumulator g
    int acc = grp;
    uint32_t acc_phase = 0;
    bool alive = true;
    const int u_first = PAIR ? (int)(blockIdx.x >> 1) : (int)(blockIdx.x + grp * gridDim.x);
    const int u_step = PAIR ? (int)(gridDim.x >> 1) : (int)(kGroups * gridDim.x);
    const int pair_rank = PAIR ? (int)cluster_ctarank() : 0;
    for (int u = u_first; alive && u < p.units; u += u_step) {
        Unit w = decode(p, u);
        if (PAIR) w.pt = 2 * w.pt + pair_rank;
        // partial sums take no epilogue, except the bias that the first of the
        // slices adding into the output brings.  Lane l fetches channel l of each
        // of the warp's chunks now, before the accumulator is ready; the chunk
        // loop hands the values round with shuffles (a per-chunk load of all 32
        // biases cost a DRAM round trip per chunk after a cold start).
        const bool use_bias = !kPlain && (kInPlace || !p.ws) && p.epi != BIGEMM_EPI_NONE &&
                              !(red && w.sp != 0);
        float bl[kMine];
#pragma unroll
        for (int i = 0; i < kMine; ++i) {
            const int c = w.ct * BN + (h + kSplit * i) * 32 + lane;
            bl[i] = (use_bias && c < p.CO) ? __ldg(p.bias + c) : 0.f;
        }
#pragma unroll 1
      for (int m = 0; m < MT; ++m) {
        // where this lane's pixel and this warp's store box go: computed
        // before the accumulator is ready
        const int b = w.pt * p.bpt + bi;
        bool valid = bi < p.bpt && b < p.total_boxes;
        long long base = 0;
        if (valid) {
            uint32_t urem;
            int n = (int)fd_divmod((uint32_t)b, p.fd_bpi, &urem);
            const int rem = (int)urem;
            long long pix;
            if (BOXED && p.im2col) {
                // the tile is 128 consecutive pixels of the flattened N x Ho x Wo
                const long long g = (long long)w.pt * 128 + row;
                n = (int)fd_divmod((uint32_t)g, p.fd_howo, &urem);
                pix = urem;
                valid = g < (long long)p.N * howo;
            } else if (BOXED) {
                const int byi = (int)fd_divmod((uint32_t)rem, p.fd_bx, &urem), bxi = (int)urem;
                int y = byi * p.box_h + m * 16 + bj_y;
                const int x = bxi * p.box_w + bj_x;
                if (p.hp) {                     // stacked images: row -> (image, row)
                    n = (int)fd_divmod((uint32_t)y, p.fd_hp, &urem);
                    y = (int)urem;
                }
                valid = n < p.N && y < p.Ho && x < p.Wo;
                pix = (long long)y * p.Wo + x;
            } else {
                pix = (long long)rem * p.box_w + bj;
                valid = pix < howo;
            }
            base = ((!kInPlace && p.ws) ? (long long)w.sp * p.out_elems : 0ll) + (long long)n * p.CO * howo + pix;
        }
        // the warp's store box (TMA mode): origin and image index
        const int wb = w.pt * p.bpt + wbi;
        const bool wbox = tma_out && wbi < p.bpt && wb < p.total_boxes;
        int sx = 0, sy = 0, sn = 0;
        if (wbox) {
            uint32_t urem;
            int n = (int)fd_divmod((uint32_t)wb, p.fd_bpi, &urem);
            const int rem = (int)urem;
            if (BOXED) {
                const int byi = (int)fd_divmod((uint32_t)rem, p.fd_bx, &urem), bxi = (int)urem;
                sx = bxi * p.box_w + wj0_x;
                sy = byi * p.box_h + m * 16 + wj0_y;
                if (p.hp) {                     // the warp's rows lie in one image (hp % rows == 0)
                    n = (int)fd_divmod((uint32_t)sy, p.fd_hp, &urem);
                    sy = (int)urem;
                }
            } else {
                sx = rem * p.box_w + wj0;
            }
            sn = n;
        }
        const bool wstore = wbox && sn < p.N;
        if (!kInPlace && p.ws) sn += w.sp * p.N;   // K slice w.sp's plane of the workspace
        // Stores from registers (no TMA box fits the output rows): where every
        // group of four lanes holds four consecutive pixels of one plane, at a
        // 4-element boundary, or no valid pixel at all, the warp regroups each
        // 32 x 32 block through its staging buffer and a lane writes 4-pixel
        // runs of one channel (8 or 16 bytes; K slices add them with one
        // 16-byte vector atomic) instead of single elements.
        bool vec4 = false, gok = false;
        long long gbase = 0;
        if (vec_static) {
            const long long lead = __shfl_sync(0xffffffffu, base, lane & ~3);
            const bool mine = valid && base == lead + (lane & 3) && (lead & 3) == 0;
            const unsigned okm = __ballot_sync(0xffffffffu, mine);
            const unsigned vm = __ballot_sync(0xffffffffu, valid);
            bool uniform = true;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                const unsigned no = (okm >> (4 * g)) & 0xFu, nv = (vm >> (4 * g)) & 0xFu;
                uniform = uniform && (no == 0xFu || nv == 0u);
            }
            vec4 = uniform;
            gbase = __shfl_sync(0xffffffffu, base, (lane & 7) * 4);
            gok = ((okm >> ((lane & 7) * 4)) & 0xFu) == 0xFu;
        }
        if (m == 0) {
            int okw = 0;
            if (lane == 0) okw = mbar_wait(&tfull[acc], acc_phase, p.timeout_ns, abort_flag, p.err);
            if (!__shfl_sync(0xffffffffu, okw, 0)) {
                alive = false;
                break;
            }
            tc_fence_after();
        }
        const uint32_t acc_col = lane_base + (uint32_t)(acc * MT * BN + m * BN);
        uint32_t ra[32], rb[32];
        tmem_ld_32x32b_x32(acc_col + (uint32_t)(h * 32), ra);
        const int co0 = w.ct * BN;
#pragma unroll
        for (int i = 0; i < kMine; ++i) {
            uint32_t(&cur)[32] = (i & 1) ? rb : ra;
            uint32_t(&nxt)[32] = (i & 1) ? ra : rb;
            tmem_wait_ld_regs(cur);
            if (i + 1 < kMine) {
                tmem_ld_32x32b_x32(acc_col + (uint32_t)((h + kSplit * (i + 1)) * 32), nxt);
            } else if (m == MT - 1) {           // accumulator drained by this warp: hand it back
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR)
                        mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
                    else
                        mbar_arrive(&tempty[acc]);
                }
            }
            const int cb = co0 + (h + kSplit * i) * 32;
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(cur[j]);
            if (use_bias) {
                float bv[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) bv[j] = __shfl_sync(0xffffffffu, bl[i], j);
                if (FORM == 4 || p.epi == BIGEMM_EPI_BIAS) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] += bv[j];
                } else if (p.epi == BIGEMM_EPI_BIAS_EXP) {
                    // the hardware exp2 with one multiply (a few ulp): far inside the
                    // conv's own error bound, and half the instructions of expf
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __expf(v[j] + bv[j]);
                } else if (p.epi == BIGEMM_EPI_BIAS_RSQRT) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = rsqrtf(v[j] + bv[j] + p.eps);
                } else if (p.epi == BIGEMM_EPI_BIAS_RELU) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = fmaxf(v[j] + bv[j], 0.f);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 1.0f / (v[j] + bv[j]);
                }
            }
            if (wstore) {
                // 2 KB pieces (32 channels of 16-bit output, or 16 of fp32), each
                // written to the next of the warp's NB staging buffers and sent as
                // one TMA box; a buffer is rewritten once the store that last used
                // it has read it, so NB - 1 stores stay in flight
#pragma unroll
                for (int hh = 0; hh < (ec == 4 ? 2 : 1); ++hh) {
                    uint8_t *buf = wstage + (piece % kNB) * 2048;
                    ++piece;
                    if (lane == 0) bulk_wait_read<kNB - 1>();
                    __syncwarp();
                    if (ec == 4) {
                        uint8_t *dst = buf + lane * 4;
#pragma unroll
                        for (int j = 0; j < 16; ++j) *reinterpret_cast<float *>(dst + j * 128) = v[hh * 16 + j];
                    } else {
                        // two channels per conversion (cvt.rn.{f16,bf16}x2.f32), one per 16-bit store
                        uint8_t *dst = buf + lane * 2;
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const uint32_t pk = pack2_16(v[j], v[j + 1], p.out_dt == BIGEMM_F16);
                            *reinterpret_cast<uint16_t *>(dst + j * 64) = (uint16_t)(pk & 0xFFFFu);
                            *reinterpret_cast<uint16_t *>(dst + (j + 1) * 64) = (uint16_t)(pk >> 16);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int cc = cb + hh * 16;
                        if (red) {
                            if (BOXED)
                                tma_reduce_add_4d(map_c, buf, sx, sy, cc, sn);
                            else
                                tma_reduce_add_3d(map_c, buf, sx, cc, sn);
                        } else if (BOXED) {
                            tma_store_4d(map_c, buf, sx, sy, cc, sn);
                        } else {
                            tma_store_3d(map_c, buf, sx, cc, sn);
                        }
                        bulk_commit();
                    }
                }
            } else if (vec4) {
                // the block of 32 pixels x 32 channels goes through the first
                // 2 KB of the warp's staging as [channel][pixel] (16 channels at a
                // time for fp32); lane l then takes pixel group l % 8 of channels
                // l / 8, l / 8 + 4, ... and writes each as one 4-pixel run
                const int g = lane & 7, c0 = lane >> 3;
                if (ec == 4) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            *reinterpret_cast<float *>(wstage + j * 128 + lane * 4) = v[hh * 16 + j];
                        __syncwarp();
                        if (gok) {
                            float *o = static_cast<float *>(p.out) + gbase + (long long)(cb + hh * 16) * howo;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int c = c0 + 4 * k;
                                if (cb + hh * 16 + c < p.CO) {
                                    const float4 val = *reinterpret_cast<const float4 *>(wstage + c * 128 + g * 16);
                                    if (red)   // a K slice: one 16-byte vector add per run
                                        atomicAdd(reinterpret_cast<float4 *>(o + c * howo), val);
                                    else
                                        *reinterpret_cast<float4 *>(o + c * howo) = val;
                                }
                            }
                        }
                    }
                } else {
                    const bool f16 = p.out_dt == BIGEMM_F16;
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const uint32_t pk = pack2_16(v[j], v[j + 1], f16);
                        *reinterpret_cast<uint16_t *>(wstage + j * 64 + lane * 2) = (uint16_t)(pk & 0xFFFFu);
                        *reinterpret_cast<uint16_t *>(wstage + (j + 1) * 64 + lane * 2) = (uint16_t)(pk >> 16);
                    }
                    __syncwarp();
                    if (gok) {
                        uint16_t *o = static_cast<uint16_t *>(p.out) + gbase + (long long)cb * howo;
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int c = c0 + 4 * k;
                            if (cb + c < p.CO)
                                *reinterpret_cast<uint2 *>(o + c * howo) =
                                    *reinterpret_cast<const uint2 *>(wstage + c * 64 + g * 8);
                        }
                    }
                }
            } else if ((FORM == 0 || FORM == 2 || FORM == 4) && !tma_out && valid) {
                const long long o0 = base + (long long)cb * howo;
                const int jn = min(32, p.CO - cb);
                if (!kInPlace && p.ws) {
                    float *o = p.ws + o0;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < jn) o[j * howo] = v[j];
                } else if (red) {
                    float *o = static_cast<float *>(p.out) + o0;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < jn) atomicAdd(o + j * howo, v[j]);
                } else if (FORM == 0 && p.out_dt == BIGEMM_F32) {
                    float *o = static_cast<float *>(p.out) + o0;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < jn) o[j * howo] = v[j];
                } else {
                    uint16_t *o = static_cast<uint16_t *>(p.out) + o0;
                    const bool f16 = p.out_dt == BIGEMM_F16;
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const uint32_t pk = pack2_16(v[j], v[j + 1], f16);
                        if (j < jn) o[j * howo] = (uint16_t)(pk & 0xFFFFu);
                        if (j + 1 < jn) o[(j + 1) * howo] = (uint16_t)(pk >> 16);
                    }
                }
            }
        }
      }
        if (kGroups > 1) {
            acc_phase ^= 1u;                    // the group's next use of its accumulator
        } else {
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    if (lane == 0) bulk_wait<0>();              // stores complete before the block exits
}


}  // namespace
}  // namespace bigemm
