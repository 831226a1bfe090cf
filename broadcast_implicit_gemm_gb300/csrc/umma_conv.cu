// umma_conv.cu -- implicit-GEMM NCHW convolution on the sm_103a tensor cores.
//
// The convolution of "Tuning High Performance Convolution on NVIDIA GPUs"
// (TVM v0.5 autotvm tutorial, Step 1: conv2d_nchw with inlined padding) is
// computed as one GEMM per launch:
//     D[pixel, f] = sum_k A[pixel, k] * B[f, k]
// with pixel = (n, y, x) on the MMA's M axis (128 TMEM lanes), the output
// channel f on its N axis (tile of BN), and k = (ry, rx, ci) on the reduction
// axis.  The padded tensor is never built: TMA reads each tap's box at the
// shifted (possibly negative) coordinates and fills out-of-range elements
// with zeros, which is the tutorial's inlined padding done by the copy engine.
//
// Structure (one persistent CTA per SM, 10 warps):
//   warp 0    TMA producer: for each K block loads the A box(es) and the B tile
//             into a STAGES-deep shared-memory ring (mbarrier full/empty).
//   warp 1    allocates TMEM, and one lane issues tcgen05.mma (4 per K block,
//             128-byte swizzled operands) into one of two TMEM accumulators.
//   warps 2-9 epilogue, two warps per TMEM lane quadrant (a warp may only
//             read the 32 lanes of quadrant warp % 4), each taking every other
//             32-channel chunk: tcgen05.ld the accumulator (lane = pixel),
//             apply the fused per-channel epilogue op(acc + bias[f]) and store
//             NCHW, through a TMA tensor store of a staged 32 x 32 box or, where
//             TMA cannot address the output rows, directly: for a fixed
//             channel the 32 lanes of a warp write 32 neighbouring pixels.
// The two accumulators let the epilogue of one tile overlap the MMAs of the
// next.  Split-K writes fp32 partial sums to a workspace instead; a separate
// kernel adds them in a fixed order and applies the epilogue.
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

// Epilogue of one warp (warps 2..9 of the block: two warps per TMEM lane
// quadrant, each taking every other 32-channel chunk of the accumulator).
// BOXED: the tile's pixels are 2-D boxes (box_w x box_h) of one image (or of
// the stacked images); otherwise runs of box_w consecutive flattened pixels
// (the direct mode).
template <int BN, bool BOXED>
__device__ __forceinline__ void epilogue_warp(const UmmaParams &p, const CUtensorMap *map_c,
                                              uint32_t tmem_base, uint64_t *tfull,
                                              uint64_t *tempty, uint8_t *stage_out,
                                              volatile int *abort_flag, int warp, int lane,
                                              int box_px)
{
    // The warp owns TMEM lanes 32q..32q+31 (32 pixels of the tile) and the
    // chunks h, h+2, ... of the BN accumulator columns.  Lane 0 waits for the
    // accumulator and shares the outcome, so the warp stays converged.  The
    // load of the warp's next chunk is issued before the current one is
    // processed.  With TMA stores the warp stages its 32 pixels x 32 channels
    // in its own 4 KB of shared memory and lane 0 writes them as one box.
    constexpr int kChunks = BN / 32;            // 2, 4 or 8
    constexpr int kMine = kChunks / 2;          // chunks per warp
    const int q = warp & 3;                     // TMEM lane quadrant of this warp
    const int h = (warp - 2) >> 2;              // which half of the chunks
    const int row = q * 32 + lane;              // tile row = pixel
    const int bi = row / box_px, bj = row - bi * box_px;
    const int wbi = (q * 32) / box_px;          // the warp's box
    const int wj0 = (q * 32) - wbi * box_px;    // its first pixel in the box
    const int bj_y = bj / p.box_w, bj_x = bj - bj_y * p.box_w;
    const int wj0_y = wj0 / p.box_w, wj0_x = wj0 - wj0_y * p.box_w;
    const long long howo = (long long)p.Ho * p.Wo;
    const int ec = p.ws ? 4 : (p.out_dt == BIGEMM_F32 ? 4 : 2);
    uint8_t *wstage = stage_out + (warp - 2) * 4096;
    const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        const Unit w = decode(p, u);
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
            if (BOXED) {
                const int byi = (int)fd_divmod((uint32_t)rem, p.fd_bx, &urem), bxi = (int)urem;
                int y = byi * p.box_h + bj_y;
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
            base = (long long)w.sp * p.out_elems + (long long)n * p.CO * howo + pix;
        }
        // the warp's store box (TMA mode): origin and image index
        const int wb = w.pt * p.bpt + wbi;
        const bool wbox = p.store_tma && wbi < p.bpt && wb < p.total_boxes;
        int sx = 0, sy = 0, sn = 0;
        if (wbox) {
            uint32_t urem;
            int n = (int)fd_divmod((uint32_t)wb, p.fd_bpi, &urem);
            const int rem = (int)urem;
            if (BOXED) {
                const int byi = (int)fd_divmod((uint32_t)rem, p.fd_bx, &urem), bxi = (int)urem;
                sx = bxi * p.box_w + wj0_x;
                sy = byi * p.box_h + wj0_y;
                if (p.hp) {                     // the warp's rows lie in one image (hp % rows == 0)
                    n = (int)fd_divmod((uint32_t)sy, p.fd_hp, &urem);
                    sy = (int)urem;
                }
            } else {
                sx = rem * p.box_w + wj0;
            }
            sn = w.sp * p.N + n;
        }
        const bool wstore = wbox && sn < (w.sp + 1) * p.N;
        int okw = 0;
        if (lane == 0) okw = mbar_wait(&tfull[acc], acc_phase, p.timeout_ns, abort_flag, p.err);
        if (!__shfl_sync(0xffffffffu, okw, 0)) break;
        tc_fence_after();
        const uint32_t acc_col = lane_base + (uint32_t)(acc * BN);
        uint32_t ra[32], rb[32];
        tmem_ld_32x32b_x32(acc_col + (uint32_t)(h * 32), ra);
        const int co0 = w.ct * BN;
#pragma unroll
        for (int i = 0; i < kMine; ++i) {
            uint32_t(&cur)[32] = (i & 1) ? rb : ra;
            uint32_t(&nxt)[32] = (i & 1) ? ra : rb;
            tmem_wait_ld_regs(cur);
            if (i + 1 < kMine) {
                tmem_ld_32x32b_x32(acc_col + (uint32_t)((h + 2 * (i + 1)) * 32), nxt);
            } else {                            // accumulator drained by this warp: hand it back
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[acc]);
            }
            const int cb = co0 + (h + 2 * i) * 32;
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(cur[j]);
            if (!p.ws && p.epi != BIGEMM_EPI_NONE) {
                float bv[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) bv[j] = cb + j < p.CO ? __ldg(p.bias + cb + j) : 0.f;
                if (p.epi == BIGEMM_EPI_BIAS) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] += bv[j];
                } else if (p.epi == BIGEMM_EPI_BIAS_EXP) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = expf(v[j] + bv[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = rsqrtf(v[j] + bv[j] + p.eps);
                }
            }
            if (wstore) {
                if (lane == 0) bulk_wait_read<0>();   // the previous store has read the buffer
                __syncwarp();
                uint8_t *dst = wstage + lane * ec;
                if (ec == 4) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) *reinterpret_cast<float *>(dst + j * 128) = v[j];
                } else {
                    // two channels per conversion (cvt.rn.{f16,bf16}x2.f32), one per 16-bit store
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
                    if (BOXED)
                        tma_store_4d(map_c, wstage, sx, sy, cb, sn);
                    else
                        tma_store_3d(map_c, wstage, sx, cb, sn);
                    bulk_commit();
                }
            } else if (!p.store_tma && valid) {
                const long long o0 = base + (long long)cb * howo;
                const int jn = min(32, p.CO - cb);
                if (p.ws) {
                    float *o = p.ws + o0;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < jn) o[j * howo] = v[j];
                } else if (p.out_dt == BIGEMM_F32) {
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
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait<0>();              // stores complete before the block exits
}

template <int BN, int AMODE, int FMT>
__global__ void __launch_bounds__(kThreads, 1)
    umma_conv_kernel(const __grid_constant__ CUtensorMap map_a,
                     const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_c, const UmmaParams p)
{
    using C = Cfg<BN>;
    constexpr int S = C::stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sa = smem;
    uint8_t *sb = smem + S * kABytes;
    uint8_t *stage_out = sb + S * C::b_bytes;               // 8 warps x 4 KB output staging
    uint64_t *full = reinterpret_cast<uint64_t *>(stage_out + C::staging);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int box_px = p.box_w * p.box_h;           // rows of A filled by one box
    const uint32_t box_bytes = (uint32_t)box_px * kRowBytes;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kEpiWarps);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
        if (p.store_tma) tma_prefetch_desc(&map_c);
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(tmem_holder, C::tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    griddep_wait();   // the set-up above overlapped the previous kernel; its data is ready now

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // The warp walks the loop together: lane 0 waits for a free slot and
        // arms its barrier, then lanes 0..nbox-1 each issue one A box and lane
        // nbox the B tile, so the copies of a K block leave in one instruction.
        {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            uint32_t last_parity[S];
            bool issued[S];
            for (int i = 0; i < S; ++i) issued[i] = false, last_parity[i] = 0;
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                const Unit w = decode(p, u);
                const int box0 = w.pt * p.bpt;
                const int nbox = min(p.bpt, p.total_boxes - box0);
                const uint32_t tx = (uint32_t)nbox * box_bytes + (uint32_t)C::b_bytes;
                int mbx = 0, mby = 0, mbn = 0;
                if (lane < nbox) {
                    const int bb = box0 + lane;
                    uint32_t urem;
                    const int n = (int)fd_divmod((uint32_t)bb, p.fd_bpi, &urem);
                    const int rem = (int)urem;
                    mbn = n;
                    if (AMODE == A_NHWC) {
                        const int byi = (int)fd_divmod((uint32_t)rem, p.fd_bx, &urem), bxi = (int)urem;
                        mbx = bxi * p.box_w * p.stride - p.pad;
                        mby = byi * p.box_h * p.stride - p.pad;
                    } else {
                        mbx = rem * p.box_w;
                    }
                }
                uint32_t urem;
                const int tap = (int)fd_divmod((uint32_t)w.kb0, p.fd_cib, &urem);
                int cb = (int)urem;
                int ry = (int)fd_divmod((uint32_t)tap, p.fd_kw, &urem), rx = (int)urem;
                const int ncol = w.ct * BN;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    int okw = 1;
                    if (lane == 0) {
                        okw = mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag, p.err);
                        if (okw) mbar_arrive_expect_tx(&full[stage], tx);
                    }
                    if (!__shfl_sync(0xffffffffu, okw, 0)) { ok = false; break; }
                    issued[stage] = true;
                    last_parity[stage] = phase;
                    uint8_t *a_dst = sa + stage * kABytes;
                    uint8_t *b_dst = sb + stage * C::b_bytes;
                    if (lane < nbox) {
                        if (AMODE == A_NHWC)
                            tma_load_4d(a_dst + lane * box_bytes, &map_a, &full[stage], cb * p.bk,
                                        mbx + rx, mby + ry, mbn);
                        else
                            tma_load_3d(a_dst + lane * box_bytes, &map_a, &full[stage], mbx, kb * p.bk, mbn);
                    } else if (lane == nbox) {
                        if (AMODE == A_NHWC)
                            tma_load_2d(b_dst, &map_b, &full[stage], (ry * p.KW + rx) * p.cip + cb * p.bk, ncol);
                        else
                            tma_load_2d(b_dst, &map_b, &full[stage], kb * p.bk, ncol);
                    }
                    if (++stage == S) stage = 0, phase ^= 1u;
                    if (++cb == p.ci_blocks) {
                        cb = 0;
                        if (++rx == p.KW) rx = 0, ++ry;
                    }
                }
            }
            if (!ok && lane == 0) {
                int local_abort = 0;
                for (int i = 0; i < S; ++i)
                    if (issued[i]) mbar_wait(&full[i], last_parity[i], p.timeout_ns, &local_abort, p.err);
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc =
                make_idesc(FMT == 2 ? 2u : (uint32_t)FMT, AMODE == A_DIRECT ? 1u : 0u, 0u,
                           kTileM, BN);
            // Byte step of the A start address per MMA (K = 32 bytes of each row):
            // K-major rows advance inside the swizzle row; MN-major advances by
            // whole 8-row groups (16 rows for 16-bit types, 8 rows for tf32).
            constexpr uint32_t a_kstep = AMODE == A_NHWC ? 32u : (FMT == 2 ? 1024u : 2048u);
            const uint32_t a_hi = desc_hi(1024u, 2u), b_hi = desc_hi(1024u, 2u);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true, any = false;
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                const Unit w = decode(p, u);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.timeout_ns, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_lo = desc_lo(smem_u32(sa + stage * kABytes),
                                                  AMODE == A_NHWC ? 16u : box_bytes);
                    const uint32_t b_lo = desc_lo(smem_u32(sb + stage * C::b_bytes), 16u);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_lohi<FMT == 2>(d_tmem, a_lo + k * (a_kstep >> 4), a_hi, b_lo + k * 2u,
                                            b_hi, idesc, (kb > w.kb0 || k > 0) ? 1u : 0u);
                    any = true;
                    umma_commit(&empty[stage]);
                    if (++stage == S) stage = 0, phase ^= 1u;
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && any) {
                // Wait for every MMA issued so far before TMEM is released.
                int local_abort = 0;
                umma_commit(drain);
                mbar_wait(drain, 0, p.timeout_ns, &local_abort, p.err);
            }
        }
    } else {
        // --------------------------------------------------------- epilogue
        epilogue_warp<BN, AMODE != A_DIRECT>(p, &map_c, tmem_base, tfull, tempty, stage_out,
                                             abort_flag, warp, lane, box_px);
    }

    griddep_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, C::tmem_cols);
    }
}


// ------------------------------------------------------------------ halo mode
// Stride-1 K x K convolutions: the tile is 16 output rows x 8 output columns of
// one image.  For each 128-byte channel block one TMA box brings the tile's
// input halo, (16 + KH - 1) rows x 16 pixels, into shared memory with a row
// pitch of 16 pixels (2 KB, a whole number of 1 KB swizzle periods).  The A
// operand of tap (ry, rx) is then this halo read from row ry, column rx: a
// descriptor start (ry*16 + rx) rows in and the 8-row groups (output rows) 2 KB
// apart.  The 128-byte swizzle is a function of the shared-memory address bits
// (measured: the descriptor's base offset must stay 0 for such starts), and
// both TMA and the MMA see the same address for each halo pixel.  The
// B operand (packed weights) arrives TB taps per copy from a (channel, output
// channel, tap) view, so a 3x3 tile needs 1 A copy and 9/TB B copies per
// channel block instead of 9 of each.
constexpr int kHaloPitch = 16;
constexpr int kHaloRowBytes = kHaloPitch * kRowBytes;        // 2 KB
constexpr int kHaloMaxKH = 7;
constexpr int kHaloBytes = (16 + kHaloMaxKH - 1) * kHaloRowBytes;   // 44 KB

template <int BN>
struct HaloCfg {
    static constexpr int a_stages = 2;
    static constexpr int b_bytes = 32768;
    static constexpr int tb = b_bytes / (BN * kRowBytes);    // taps per B copy: 4, 2, 1
    static constexpr int b_stages = 3;
    static constexpr int staging = kEpiWarps * 4096;
    static constexpr int bars = (2 * a_stages + 2 * b_stages + 5) * 8;
    static constexpr int smem = a_stages * kHaloBytes + b_stages * b_bytes + staging + bars + 16 + 1024;
    static constexpr uint32_t tmem_cols = Cfg<BN>::tmem_cols;
};

// Resident-weights form (RES): when one output-channel tile covers CO and all
// of its taps fit in shared memory, the producer loads B once (one tap per
// copy, every channel block) and only the halos stream; up to kResMaxA halo
// stages then fit beside it.  The host sizes the layout (p.res_sa stages of
// (16 + KH - 1) rows, p.res_b_bytes of weights) within the shared-memory limit.
constexpr int kResMaxA = 4;

template <int BN, bool RES>
struct HaloBars {
    static constexpr int a = RES ? kResMaxA : HaloCfg<BN>::a_stages;
    static constexpr int b = RES ? 1 : HaloCfg<BN>::b_stages;
    static constexpr int bytes = (2 * a + 2 * b + 5) * 8;
};

template <int BN>
size_t halo_res_smem(int sa, int kh, size_t b_bytes)
{
    return (size_t)sa * (16 + kh - 1) * kHaloRowBytes + b_bytes + HaloCfg<BN>::staging +
           HaloBars<BN, true>::bytes + 16 + 1024;
}

template <int BN, int FMT, bool RES>
__global__ void __launch_bounds__(kThreads, 1)
    umma_conv_halo_kernel(const __grid_constant__ CUtensorMap map_a,
                          const __grid_constant__ CUtensorMap map_b,
                          const __grid_constant__ CUtensorMap map_c, const UmmaParams p)
{
    using C = HaloCfg<BN>;
    using BARS = HaloBars<BN, RES>;
    constexpr int SAMAX = BARS::a, SB = BARS::b;
    constexpr int TB = RES ? 1 : C::tb;
    const int SA = RES ? p.res_sa : C::a_stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t halo_bytes = (uint32_t)(16 + p.KH - 1) * kHaloRowBytes;
    const uint32_t a_stride = RES ? halo_bytes : (uint32_t)kHaloBytes;
    uint8_t *sa = smem;
    uint8_t *sb = sa + SA * a_stride;
    uint8_t *stage_out = sb + (RES ? (uint32_t)p.res_b_bytes : (uint32_t)(SB * C::b_bytes));
    uint64_t *a_full = reinterpret_cast<uint64_t *>(stage_out + C::staging);
    uint64_t *a_empty = a_full + SAMAX;
    uint64_t *b_full = a_empty + SAMAX;
    uint64_t *b_empty = b_full + SB;
    uint64_t *tfull = b_empty + SB;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KK = p.KH * p.KW;

    if (threadIdx.x == 0) {
        for (int i = 0; i < SA; ++i) mbar_init(&a_full[i], 1), mbar_init(&a_empty[i], 1);
        for (int i = 0; i < SB; ++i) mbar_init(&b_full[i], 1), mbar_init(&b_empty[i], 1);
        for (int i = 0; i < 2; ++i) mbar_init(&tfull[i], 1), mbar_init(&tempty[i], kEpiWarps);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
        if (p.store_tma) tma_prefetch_desc(&map_c);
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(tmem_holder, C::tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    griddep_wait();   // the set-up above overlapped the previous kernel; its data is ready now

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int as = 0, bs = 0;
            uint32_t aph = 0, bph = 0;
            uint32_t a_par[SAMAX], b_par[SB];
            bool a_iss[SAMAX], b_iss[SB];
            for (int i = 0; i < SAMAX; ++i) a_iss[i] = false, a_par[i] = 0;
            for (int i = 0; i < SB; ++i) b_iss[i] = false, b_par[i] = 0;
            bool ok = true;
            if (RES) {
                // every tap of every channel block, once, on b_full[0]
                mbar_arrive_expect_tx(&b_full[0], (uint32_t)p.res_b_bytes);
                b_iss[0] = true;
                for (int cb = 0; cb < p.ci_blocks; ++cb)
                    for (int t = 0; t < KK; ++t)
                        tma_load_3d(sb + (size_t)(cb * KK + t) * (BN * kRowBytes), &map_b, &b_full[0],
                                    cb * p.bk, 0, t);
            }
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                const Unit w = decode(p, u);
                uint32_t urem;
                const int n = (int)fd_divmod((uint32_t)w.pt, p.fd_bpi, &urem);
                const int byi = (int)fd_divmod(urem, p.fd_bx, &urem), bxi = (int)urem;
                const int x0 = bxi * 8 - p.pad, y0 = byi * 16 - p.pad;
                const int ncol = w.ct * BN;
                for (int cb = w.kb0; ok && cb < w.kb1; ++cb) {
                    if (!mbar_wait(&a_empty[as], aph ^ 1u, p.timeout_ns, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&a_full[as], halo_bytes);
                    a_iss[as] = true, a_par[as] = aph;
                    tma_load_4d(sa + as * a_stride, &map_a, &a_full[as], cb * p.bk, x0, y0, n);
                    if (++as == SA) as = 0, aph ^= 1u;
                    if (RES) continue;
                    for (int t0 = 0; t0 < KK; t0 += TB) {
                        if (!mbar_wait(&b_empty[bs], bph ^ 1u, p.timeout_ns, abort_flag, p.err)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&b_full[bs], (uint32_t)C::b_bytes);
                        b_iss[bs] = true, b_par[bs] = bph;
                        tma_load_3d(sb + bs * C::b_bytes, &map_b, &b_full[bs], cb * p.bk, ncol, t0);
                        if (++bs == SB) bs = 0, bph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let every copy already issued land before the block exits.
                int local_abort = 0;
                for (int i = 0; i < SA; ++i)
                    if (a_iss[i]) mbar_wait(&a_full[i], a_par[i], p.timeout_ns, &local_abort, p.err);
                for (int i = 0; i < SB; ++i)
                    if (b_iss[i]) mbar_wait(&b_full[i], b_par[i], p.timeout_ns, &local_abort, p.err);
            } else if (RES) {
                // the weights may still be in flight if this block had no unit to run
                int local_abort = 0;
                mbar_wait(&b_full[0], 0, p.timeout_ns, &local_abort, p.err);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(FMT == 2 ? 2u : (uint32_t)FMT, 0u, 0u, kTileM, BN);
            const uint32_t a_hi = desc_hi((uint32_t)kHaloRowBytes, 2u), b_hi = desc_hi(1024u, 2u);
            int as = 0, bs = 0, acc = 0;
            uint32_t aph = 0, bph = 0, acc_phase = 0;
            bool ok = true, any = false;
            if (RES && blockIdx.x < p.units)
                ok = mbar_wait(&b_full[0], 0, p.timeout_ns, abort_flag, p.err);
            const uint32_t b_res0 = desc_lo(smem_u32(sb), 16u);
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                const Unit w = decode(p, u);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.timeout_ns, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                uint32_t accum = 0;
                for (int cb = w.kb0; ok && cb < w.kb1; ++cb) {
                    if (!mbar_wait(&a_full[as], aph, p.timeout_ns, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_lo0 = desc_lo(smem_u32(sa + as * a_stride), 16u);
                    int ry = 0, rx = 0;
                    if (RES) {
                        tc_fence_after();
                        uint32_t b_lo = b_res0 + (uint32_t)(cb * KK) * ((uint32_t)(BN * kRowBytes) >> 4);
                        for (int t = 0; t < KK; ++t) {
                            const uint32_t a_lo =
                                a_lo0 + (uint32_t)(ry * kHaloPitch + rx) * (kRowBytes >> 4);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                umma_lohi<FMT == 2>(d_tmem, a_lo + k * 2u, a_hi, b_lo + k * 2u, b_hi,
                                                    idesc, accum);
                                accum = 1u;
                            }
                            b_lo += (uint32_t)(BN * kRowBytes) >> 4;
                            if (++rx == p.KW) rx = 0, ++ry;
                        }
                        any = true;
                    } else {
                        for (int t0 = 0; t0 < KK; t0 += TB) {
                            if (!mbar_wait(&b_full[bs], bph, p.timeout_ns, abort_flag, p.err)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            uint32_t b_lo = desc_lo(smem_u32(sb + bs * C::b_bytes), 16u);
                            const int nt = min(TB, KK - t0);
                            for (int tt = 0; tt < nt; ++tt) {
                                const uint32_t a_lo =
                                    a_lo0 + (uint32_t)(ry * kHaloPitch + rx) * (kRowBytes >> 4);
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    umma_lohi<FMT == 2>(d_tmem, a_lo + k * 2u, a_hi, b_lo + k * 2u,
                                                        b_hi, idesc, accum);
                                    accum = 1u;
                                }
                                b_lo += (uint32_t)(BN * kRowBytes) >> 4;
                                if (++rx == p.KW) rx = 0, ++ry;
                            }
                            any = true;
                            umma_commit(&b_empty[bs]);
                            if (++bs == SB) bs = 0, bph ^= 1u;
                        }
                    }
                    umma_commit(&a_empty[as]);
                    if (++as == SA) as = 0, aph ^= 1u;
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && any) {
                int local_abort = 0;
                umma_commit(drain);
                mbar_wait(drain, 0, p.timeout_ns, &local_abort, p.err);
            }
        }
    } else {
        epilogue_warp<BN, true>(p, &map_c, tmem_base, tfull, tempty, stage_out, abort_flag, warp,
                                lane, 128);
    }

    griddep_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, C::tmem_cols);
    }
}

template <int BN, int FMT>
cudaError_t launch_halo(const UmmaParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                        const CUtensorMap &mc, int grid, cudaStream_t stream)
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (p.res_sa > 0) {
        auto kern = umma_conv_halo_kernel<BN, FMT, true>;
        const size_t smem = halo_res_smem<BN>(p.res_sa, p.KH, (size_t)p.res_b_bytes);
        static unsigned long long attr_set = 0;
        if (dev >= 64 || !(attr_set >> dev & 1ull)) {
            DeviceState *ds = device_state();
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 ds ? ds->max_smem_optin : (int)smem);
            if (e != cudaSuccess) return e;
            if (dev < 64) attr_set |= 1ull << dev;
        }
        return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, stream, ma, mb, mc, p);
    }
    auto kern = umma_conv_halo_kernel<BN, FMT, false>;
    static unsigned long long attr_set = 0;   // bit per device: smem opt-in done
    if (dev >= 64 || !(attr_set >> dev & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             HaloCfg<BN>::smem);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set |= 1ull << dev;
    }
    return launch_pdl(kern, dim3(grid), dim3(kThreads), (size_t)HaloCfg<BN>::smem, stream, ma, mb, mc,
                      p);
}

template <int FMT>
cudaError_t dispatch_halo_bn(int bn, const UmmaParams &p, const CUtensorMap &ma,
                             const CUtensorMap &mb, const CUtensorMap &mc, int grid, cudaStream_t s)
{
    switch (bn) {
    case 64: return launch_halo<64, FMT>(p, ma, mb, mc, grid, s);
    case 128: return launch_halo<128, FMT>(p, ma, mb, mc, grid, s);
    case 256: return launch_halo<256, FMT>(p, ma, mb, mc, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

template <int BN, int AMODE, int FMT>
cudaError_t launch_one(const UmmaParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                       const CUtensorMap &mc, int grid, cudaStream_t stream)
{
    auto kern = umma_conv_kernel<BN, AMODE, FMT>;
    static unsigned long long attr_set = 0;   // bit per device: smem opt-in done
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(attr_set >> dev & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg<BN>::smem);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set |= 1ull << dev;
    }
    return launch_pdl(kern, dim3(grid), dim3(kThreads), (size_t)Cfg<BN>::smem, stream, ma, mb, mc, p);
}

template <int AMODE, int FMT>
cudaError_t dispatch_bn(int bn, const UmmaParams &p, const CUtensorMap &ma,
                        const CUtensorMap &mb, const CUtensorMap &mc, int grid, cudaStream_t s)
{
    switch (bn) {
    case 64: return launch_one<64, AMODE, FMT>(p, ma, mb, mc, grid, s);
    case 128: return launch_one<128, AMODE, FMT>(p, ma, mb, mc, grid, s);
    case 256: return launch_one<256, AMODE, FMT>(p, ma, mb, mc, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

template <int AMODE>
cudaError_t dispatch_fmt(int fmt, int bn, const UmmaParams &p, const CUtensorMap &ma,
                         const CUtensorMap &mb, const CUtensorMap &mc, int grid, cudaStream_t s)
{
    switch (fmt) {
    case 0: return dispatch_bn<AMODE, 0>(bn, p, ma, mb, mc, grid, s);
    case 1: return dispatch_bn<AMODE, 1>(bn, p, ma, mb, mc, grid, s);
    case 2: return dispatch_bn<AMODE, 2>(bn, p, ma, mb, mc, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

int fmt_of(int in_dt) { return in_dt == BIGEMM_F16 ? 0 : in_dt == BIGEMM_BF16 ? 1 : 2; }

}  // namespace

int halo_res_stages(int bn, int kh, size_t b_bytes, int smem_limit)
{
    for (int sa = kResMaxA; sa >= 2; --sa) {
        size_t need = 0;
        switch (bn) {
        case 64: need = halo_res_smem<64>(sa, kh, b_bytes); break;
        case 128: need = halo_res_smem<128>(sa, kh, b_bytes); break;
        case 256: need = halo_res_smem<256>(sa, kh, b_bytes); break;
        default: return 0;
        }
        if (need <= (size_t)smem_limit) return sa;
    }
    return 0;
}

size_t umma_smem_bytes(const UmmaTiling &t)
{
    if (t.amode == A_HALO) {
        switch (t.bn) {
        case 64: return HaloCfg<64>::smem;
        case 128: return HaloCfg<128>::smem;
        case 256: return HaloCfg<256>::smem;
        default: return 0;
        }
    }
    switch (t.bn) {
    case 64: return Cfg<64>::smem;
    case 128: return Cfg<128>::smem;
    case 256: return Cfg<256>::smem;
    default: return 0;
    }
}

bool umma_tiling_compiled(const UmmaTiling &t, int in_dt)
{
    (void)in_dt;
    return (t.bn == 64 || t.bn == 128 || t.bn == 256) &&
           (t.amode == A_NHWC || t.amode == A_DIRECT || t.amode == A_HALO);
}

cudaError_t launch_umma_conv(const UmmaTiling &t, int in_dt, const UmmaParams &p0,
                             const CUtensorMap &map_a, const CUtensorMap &map_b,
                             const CUtensorMap &map_c, int grid, cudaStream_t stream)
{
    UmmaParams p = p0;
    p.fd_co = make_fastdiv((uint32_t)p.co_tiles);
    p.fd_pix = make_fastdiv((uint32_t)p.pix_tiles);
    p.fd_bpi = make_fastdiv((uint32_t)p.boxes_per_img);
    p.fd_bx = make_fastdiv((uint32_t)p.boxes_x);
    p.fd_hp = make_fastdiv((uint32_t)p.hp);
    p.fd_cib = make_fastdiv((uint32_t)p.ci_blocks);
    p.fd_kw = make_fastdiv((uint32_t)p.KW);
    ProfScope prof(t.amode == A_NHWC ? "umma_conv_nhwc"
                   : t.amode == A_HALO ? "umma_conv_halo"
                                       : "umma_conv_direct",
                   stream);
    const int fmt = fmt_of(in_dt);
    if (t.amode == A_HALO) {
        switch (fmt) {
        case 0: return dispatch_halo_bn<0>(t.bn, p, map_a, map_b, map_c, grid, stream);
        case 1: return dispatch_halo_bn<1>(t.bn, p, map_a, map_b, map_c, grid, stream);
        default: return dispatch_halo_bn<2>(t.bn, p, map_a, map_b, map_c, grid, stream);
        }
    }
    if (t.amode == A_NHWC)
        return dispatch_fmt<A_NHWC>(fmt, t.bn, p, map_a, map_b, map_c, grid, stream);
    return dispatch_fmt<A_DIRECT>(fmt, t.bn, p, map_a, map_b, map_c, grid, stream);
}

}  // namespace bigemm
