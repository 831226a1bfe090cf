// strided_main.cuh -- the implicit-GEMM kernel of the strided operand mode: a
// 1x1 convolution with stride 2 and no padding on 16-bit NCHW data, read in
// place.  Included by strided_conv.cu (every output form) and
// strided_plain.cu (the narrowed 16-bit forms); everything is internal.
//
// Output pixel (yo, xo) reads input pixel (2 yo, 2 xo).  TMA cannot skip
// elements of a tensor's innermost dimension, and NCHW rows of W 16-bit
// elements are not a valid TMA row pitch unless W is a multiple of 8, so the
// data is viewed as rows of 2W elements (an even input row followed by the
// odd one below it): in that view output row yo is row yo, and output column
// xo is element 2 xo.  A staging box of 32 elements x 4 rows x 64 channels
// (16 KB) then holds the inputs of 16 output columns x 4 output rows, at the
// even elements of each row (the last of the 16 columns can fall on the odd
// input row or past the tensor: they are then output columns >= Wo, which
// the epilogue never stores).  A tile is two boxes: 4 output rows each, or
// two column boxes of wider images.  Four compaction warps keep the even
// elements: each 16-byte piece of staging gives four of them, written as 8
// bytes of the MN-major operand [channel][64 pixels] in the 128-byte swizzle,
// the layout TMA gives the direct mode.  The MMA issue, the accumulators and
// the epilogue are those of the direct mode and of the per-tap mode's 16 x 4
// pixel boxes.
//
// Measured (per-K-block clock stamps, ResNet-50's 28 x 28 layer): a staging
// copy takes 1.3 - 3.8 us to land under load and the MMAs of a K block
// 0.25 us, so the staging ring, not the MMA, sets the pace: it is as deep as
// shared memory allows (three or four slots), and its copies are issued by a
// producer that waits for nothing else.  The weight tiles, whose ring slots
// free up only as the MMAs finish, are issued by the first compaction warp
// once the slot it is about to fill is free (a single producer issuing both
// let the weight ring hold back the staging copies).
#pragma once
#include "umma_common.cuh"

namespace bigemm {

namespace {

constexpr int kStridedThreads = 64 + 32 * kEpiWarps + 128;   // producer, MMA, epilogue, compaction
constexpr int kStridedStage = 2 * 16384;                    // staging of one K block: two boxes
constexpr int kStridedMaxS = 6;                              // A / B ring slots at most
constexpr int kStridedMaxSS = 4;                             // staging slots at most
constexpr int kStridedEpiStage = 2048;                       // output staging per epilogue warp

// Keep the even 16-bit elements of 16 bytes (8 elements): 4 elements, 8 bytes.
__device__ __forceinline__ uint2 even_halves(uint4 v)
{
    uint2 r;
    r.x = __byte_perm(v.x, v.y, 0x5410);
    r.y = __byte_perm(v.z, v.w, 0x5410);
    return r;
}

// FMT: 0 f16, 1 bf16.  FORM: the epilogue's output form (epilogue_warp).
template <int BN, int FMT, int FORM>
__global__ void __launch_bounds__(kStridedThreads, 1)
    umma_conv_strided_kernel(const __grid_constant__ CUtensorMap map_a,
                             const __grid_constant__ CUtensorMap map_b,
                             const __grid_constant__ CUtensorMap map_c, const UmmaParams p)
{
    constexpr int BB = BN * kRowBytes;                 // one weight K block
    const int S = p.halo_sa, SS = p.halo_sb;           // ring and staging slots (strided_layout)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sa = smem;                                // S x 16 KB: the compacted operand
    uint8_t *stg = smem + S * kABytes;                 // SS x 32 KB: staging
    uint8_t *sb = smem + p.halo_b_off;                 // S x BB: weights
    uint8_t *stage_out = smem + p.halo_stage_off;
    uint64_t *stg_full = reinterpret_cast<uint64_t *>(smem + p.halo_bar_off);
    uint64_t *stg_empty = stg_full + kStridedMaxSS;
    uint64_t *a_full = stg_empty + kStridedMaxSS;
    uint64_t *b_full = a_full + kStridedMaxS;
    uint64_t *ab_empty = b_full + kStridedMaxS;
    uint64_t *tfull = ab_empty + kStridedMaxS;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kCompWarp0 = 2 + kEpiWarps;

    if (threadIdx.x == 0) {
        for (int i = 0; i < SS; ++i) mbar_init(&stg_full[i], 1), mbar_init(&stg_empty[i], 4);
        for (int i = 0; i < S; ++i) {
            mbar_init(&a_full[i], 4);
            mbar_init(&b_full[i], 1);
            mbar_init(&ab_empty[i], 1);
        }
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
        tmem_alloc(tmem_holder, Cfg<BN>::tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    griddep_enter();   // the set-up above overlapped the previous kernel; its data is ready now

    if (warp == 0) {
        // ------------------------------------------------- staging producer
        // Lane 0 waits and arms the barrier; lanes 0..nbox-1 issue the staging
        // boxes of a K block in one instruction.
        int t = 0;
        uint32_t tph = 0;
        bool ok = true;
        uint32_t t_par[kStridedMaxSS];
        bool t_iss[kStridedMaxSS];
        for (int i = 0; i < kStridedMaxSS; ++i) t_iss[i] = false, t_par[i] = 0;
        for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
            const Unit w = decode(p, u);
            const int box0 = w.pt * p.bpt;
            const int nbox = min(p.bpt, p.total_boxes - box0);
            int bx = 0, by = 0, bn = 0;
            if (lane < nbox) {
                uint32_t urem;
                bn = (int)fd_divmod((uint32_t)(box0 + lane), p.fd_bpi, &urem);
                const int byi = (int)fd_divmod(urem, p.fd_bx, &urem), bxi = (int)urem;
                bx = bxi * 2 * p.box_w;     // element 2 xo of the row-pair view
                by = byi * p.box_h;         // row pair = output row
            }
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                int okw = 1;
                if (lane == 0) {
                    okw = mbar_wait(&stg_empty[t], tph ^ 1u, p.timeout_ns, abort_flag, p.err);
                    if (okw) mbar_arrive_expect_tx(&stg_full[t], (uint32_t)nbox * 16384u);
                }
                if (!__shfl_sync(0xffffffffu, okw, 0)) { ok = false; break; }
                t_iss[t] = true, t_par[t] = tph;
                if (lane < nbox)
                    tma_load_4d(stg + t * kStridedStage + lane * 16384, &map_a, &stg_full[t], bx, by,
                                kb * p.bk, bn);
                if (++t == SS) t = 0, tph ^= 1u;
            }
        }
        if (!ok && lane == 0) {
            // every copy already issued lands before the block exits
            int local_abort = 0;
            for (int i = 0; i < SS; ++i)
                if (t_iss[i]) mbar_wait(&stg_full[i], t_par[i], p.timeout_ns, &local_abort, p.err);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc((uint32_t)FMT, 1u, 0u, kTileM, BN);
            // MN-major A: 64-pixel halves 8 KB apart (LBO), 8-channel groups 1 KB
            // apart (SBO); one MMA takes 16 channels = 2 KB of A
            const uint32_t a_hi = desc_hi(1024u, 2u), b_hi = desc_hi(1024u, 2u);
            int s = 0, acc = 0;
            uint32_t sph = 0, acc_phase = 0;
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
                    if (!mbar_wait(&b_full[s], sph, p.timeout_ns, abort_flag, p.err) ||
                        !mbar_wait(&a_full[s], sph, p.timeout_ns, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_lo = desc_lo(smem_u32(sa + s * kABytes), 8192u);
                    const uint32_t b_lo = desc_lo(smem_u32(sb + s * BB), 16u);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_lohi<false>(d_tmem, a_lo + k * (2048u >> 4), a_hi, b_lo + k * 2u, b_hi,
                                         idesc, (kb > w.kb0 || k > 0) ? 1u : 0u);
                    any = true;
                    umma_commit(&ab_empty[s]);
                    if (++s == S) s = 0, sph ^= 1u;
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && any) {
                // every MMA issued so far completes before TMEM is released
                int local_abort = 0;
                umma_commit(drain);
                mbar_wait(drain, 0, p.timeout_ns, &local_abort, p.err);
            }
        }
    } else if (warp < kCompWarp0) {
        // --------------------------------------------------------- epilogue
        epilogue_warp<BN, true, kEpiWarps, 1, kStridedEpiStage, FORM>(
            p, &map_c, tmem_base, tfull, tempty, stage_out, abort_flag, warp, lane, 64);
    } else {
        // ------------------------------------------------------- compaction
        // Item q (16 per thread) is the 16-byte piece q of the staging, read
        // in order (no bank conflicts): box q / 1024, channel (q / 16) % 64,
        // output row (q / 4) % 4 of the box, half (q / 2) % 2 of the row's 16
        // columns, quarter q % 2 of that half; its 4 even elements are the 8
        // bytes at quarter * 8 of 16-byte chunk (row * 2 + half) of the
        // channel's 128-byte operand line, whose chunks the 128-byte swizzle
        // permutes by the line index (channel % 8).  The mapping is the same
        // for every K block, so each thread keeps its 16 destinations.
        const int tc = threadIdx.x - kCompWarp0 * 32;   // 0 .. 127
        uint32_t dst_off[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int q = tc + 128 * j;
            const int b = q >> 10, c = (q >> 4) & 63, k = (q >> 1) & 7;
            dst_off[j] = (uint32_t)(b * 8192 + c * 128 + ((k ^ (c & 7)) << 4) + (q & 1) * 8);
        }
        const bool b_issuer = tc == 0;                  // lane 0 of the first compaction warp
        int t = 0, s = 0;
        uint32_t tph = 0, sph = 0;
        bool ok = true;
        uint32_t s_par[kStridedMaxS];
        bool s_iss[kStridedMaxS];
        for (int i = 0; i < kStridedMaxS; ++i) s_iss[i] = false, s_par[i] = 0;
        for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
            const Unit w = decode(p, u);
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                if (!mbar_wait_warp(&ab_empty[s], sph ^ 1u, p.timeout_ns, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                if (b_issuer) {
                    // the slot is free: its weight tile goes out first
                    mbar_arrive_expect_tx(&b_full[s], (uint32_t)BB);
                    tma_load_2d(sb + s * BB, &map_b, &b_full[s], kb * p.bk, w.ct * BN);
                    s_iss[s] = true, s_par[s] = sph;
                }
                if (!mbar_wait_warp(&stg_full[t], tph, p.timeout_ns, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                const uint8_t *src = stg + t * kStridedStage + tc * 16;
                uint8_t *dst = sa + s * kABytes;
                uint4 v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = *reinterpret_cast<const uint4 *>(src + j * 2048);
                // the staging slot is free as soon as the warp holds its pieces
                __syncwarp();
                if (lane == 0) mbar_arrive(&stg_empty[t]);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    *reinterpret_cast<uint2 *>(dst + dst_off[j]) = even_halves(v[j]);
                // the operand's generic-proxy writes become visible to the MMA
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[s]);
                if (++t == SS) t = 0, tph ^= 1u;
                if (++s == S) s = 0, sph ^= 1u;
            }
        }
        if (!ok && b_issuer) {
            // every weight copy already issued lands before the block exits
            int local_abort = 0;
            for (int i = 0; i < S; ++i)
                if (s_iss[i]) mbar_wait(&b_full[i], s_par[i], p.timeout_ns, &local_abort, p.err);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, Cfg<BN>::tmem_cols);
    }
}

template <int BN, int FMT, int FORM>
cudaError_t launch_strided_one(const UmmaParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                               const CUtensorMap &mc, int grid, cudaStream_t stream)
{
    auto kern = umma_conv_strided_kernel<BN, FMT, FORM>;
    static unsigned long long attr_set = 0;   // bit per device: smem opt-in done
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !(attr_set >> dev & 1ull)) {
        DeviceState *ds = device_state();
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ds ? ds->max_smem_optin : p.halo_smem);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set |= 1ull << dev;
    }
    return launch_pdl(kern, dim3(grid), dim3(kStridedThreads), (size_t)p.halo_smem, stream, ma, mb,
                      mc, p);
}

template <int FORM>
cudaError_t dispatch_strided(int bn, int fmt, const UmmaParams &p, const CUtensorMap &ma,
                             const CUtensorMap &mb, const CUtensorMap &mc, int grid, cudaStream_t s)
{
    if (fmt != 0 && fmt != 1) return cudaErrorInvalidValue;   // 16-bit operands only
    switch (bn) {
    case 64:
        return fmt ? launch_strided_one<64, 1, FORM>(p, ma, mb, mc, grid, s)
                   : launch_strided_one<64, 0, FORM>(p, ma, mb, mc, grid, s);
    case 128:
        return fmt ? launch_strided_one<128, 1, FORM>(p, ma, mb, mc, grid, s)
                   : launch_strided_one<128, 0, FORM>(p, ma, mb, mc, grid, s);
    case 256:
        return fmt ? launch_strided_one<256, 1, FORM>(p, ma, mb, mc, grid, s)
                   : launch_strided_one<256, 0, FORM>(p, ma, mb, mc, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

}  // namespace bigemm
