// halo_main.cuh -- the halo-mode implicit-GEMM kernel and its launch
// dispatch, shared by halo_conv.cu (every output, FORM 0) and halo_forms.cu
// (the narrowed output forms of epilogue_warp).  Included once per
// translation unit; everything is internal.
#pragma once
#include "umma_common.cuh"

namespace bigemm {

namespace {

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
// copy, every channel block) and only the input halos stream.
constexpr int kHaloMaxA = 4;   // halo stages at most
constexpr int kHaloMaxB = 6;   // streamed weight stages at most
// Epilogue warps of the halo kernels: two per TMEM lane quadrant (measured:
// with one, the 256-channel exp epilogue of the fused layer limits the kernel),
// each staging 2 KB of output at a time, so that the room goes to the weight
// ring (measured: the MMA thread waited on weight tiles for a third of its loop
// with three 32 KB stages).
constexpr int kHaloEpi = kEpiWarps;
constexpr int kHaloStage = 2048;

// MT = 2: a unit is two 16-row tiles stacked vertically (32 output rows x 8
// columns) that share every weight tile, so the weights cost half as many
// bytes per MMA; the two 128-pixel accumulators sit BN columns apart.
template <int BN, int MT>
struct HaloTmem {
    static constexpr uint32_t cols = (2 * MT * BN <= 64) ? 64 : (2 * MT * BN <= 128) ? 128
                                     : (2 * MT * BN <= 256) ? 256 : 512;
    static_assert(2 * MT * BN <= 512, "two accumulators of MT tiles must fit TMEM");
};

// FORM: the epilogue's output form (epilogue_warp).
template <int BN, int FMT, bool RES, int MT, int FORM>
__global__ void __launch_bounds__(kThreads, 1)
    umma_conv_halo_kernel(const __grid_constant__ CUtensorMap map_a,
                          const __grid_constant__ CUtensorMap map_b,
                          const __grid_constant__ CUtensorMap map_c, const UmmaParams p)
{
    using C = HaloCfg<BN>;
    constexpr int SAMAX = kHaloMaxA, SBMAX = RES ? 1 : kHaloMaxB;
    const int SB = RES ? 1 : p.halo_sb;
    // taps per weight copy: 32 KB copies, or one tap with resident weights or two M tiles
    constexpr int TB = (RES || MT == 2) ? 1 : C::tb;
    constexpr int BB = TB * BN * kRowBytes;   // bytes of one streamed weight stage
    // shared-memory layout computed on the host (halo_layout): halo stages,
    // weights, output staging, barriers
    const int SA = p.halo_sa;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t halo_bytes = (uint32_t)(16 * MT + p.KH - 1) * kHaloRowBytes;
    const uint32_t a_stride = halo_bytes;
    uint8_t *sa = smem;
    uint8_t *sb = smem + p.halo_b_off;
    uint8_t *stage_out = smem + p.halo_stage_off;
    uint64_t *a_full = reinterpret_cast<uint64_t *>(smem + p.halo_bar_off);
    uint64_t *a_empty = a_full + SAMAX;
    uint64_t *b_full = a_empty + SAMAX;
    uint64_t *b_empty = b_full + SBMAX;
    uint64_t *tfull = b_empty + SBMAX;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KK = p.KH * p.KW;

    if (threadIdx.x == 0) {
        for (int i = 0; i < SA; ++i) mbar_init(&a_full[i], 1), mbar_init(&a_empty[i], 1);
        for (int i = 0; i < SB; ++i) mbar_init(&b_full[i], 1), mbar_init(&b_empty[i], 1);
        for (int i = 0; i < 2; ++i) mbar_init(&tfull[i], 1), mbar_init(&tempty[i], kHaloEpi);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
        if (p.store_tma) tma_prefetch_desc(&map_c);
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(tmem_holder, HaloTmem<BN, MT>::cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    griddep_enter();   // the set-up above overlapped the previous kernel; its data is ready now

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int as = 0, bs = 0;
            uint32_t aph = 0, bph = 0;
            uint32_t a_par[SAMAX], b_par[SBMAX];
            bool a_iss[SAMAX], b_iss[SBMAX];
            for (int i = 0; i < SAMAX; ++i) a_iss[i] = false, a_par[i] = 0;
            for (int i = 0; i < SBMAX; ++i) b_iss[i] = false, b_par[i] = 0;
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
                const int x0 = bxi * 8 - p.pad, y0 = byi * (16 * MT) - p.pad;
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
                    for (int t0 = 0; !RES && t0 < KK; t0 += TB) {
                        if (!mbar_wait(&b_empty[bs], bph ^ 1u, p.timeout_ns, abort_flag, p.err)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&b_full[bs], (uint32_t)BB);
                        b_iss[bs] = true, b_par[bs] = bph;
                        tma_load_3d(sb + bs * BB, &map_b, &b_full[bs], cb * p.bk, ncol, t0);
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
            const uint32_t b_res0 = desc_lo(smem_u32(sb), 16u);   // resident weights
            const uint32_t b_ring0 = b_res0;                        // or the first ring slot
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                const Unit w = decode(p, u);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.timeout_ns, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * MT * BN);
                uint32_t accum = 0;
                for (int cb = w.kb0; ok && cb < w.kb1; ++cb) {
                    if (!mbar_wait(&a_full[as], aph, p.timeout_ns, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_lo0 = desc_lo(smem_u32(sa + as * a_stride), 16u);
                    const uint32_t acc_cb = accum;   // accumulate into the tile from the first MMA on?
                    accum = 1u;
                    if (p.KH == 3 && p.KW == 3) {
                        // 3x3: every tap's A start and B slot are constants, the loop unrolls
                        constexpr uint32_t kTapOff[9] = {0, 8, 16, 128, 136, 144, 256, 264, 272};
                        constexpr uint32_t kBStep = (uint32_t)(BN * kRowBytes) >> 4;
                        constexpr uint32_t kMStep = (16u * kHaloRowBytes) >> 4;   // 16 rows down
                        if (RES) {
                            tc_fence_after();
                            const uint32_t b_lo = b_res0 + (uint32_t)(cb * 9) * kBStep;
#pragma unroll
                            for (int t = 0; t < 9; ++t)
#pragma unroll
                                for (int m = 0; m < MT; ++m)
                                    umma4_kmajor<FMT == 2>(d_tmem + m * BN, a_lo0 + kTapOff[t] + m * kMStep,
                                                           a_hi, b_lo + (uint32_t)t * kBStep, b_hi,
                                                           idesc, t == 0 ? acc_cb : 1u);
                            any = true;
                        } else {
                            constexpr int NST = (9 + TB - 1) / TB;   // weight stages per channel block
#pragma unroll
                            for (int g = 0; g < NST; ++g) {
                                if (!mbar_wait(&b_full[bs], bph, p.timeout_ns, abort_flag, p.err)) {
                                    ok = false;
                                    break;
                                }
                                tc_fence_after();
                                const uint32_t b_lo = b_ring0 + (uint32_t)bs * ((uint32_t)BB >> 4);
#pragma unroll
                                for (int tt = 0; tt < TB; ++tt) {
                                    const int t = g * TB + tt;
                                    if (t < 9)
#pragma unroll
                                        for (int m = 0; m < MT; ++m)
                                            umma4_kmajor<FMT == 2>(
                                                d_tmem + m * BN, a_lo0 + kTapOff[t] + m * kMStep, a_hi,
                                                b_lo + (uint32_t)tt * kBStep, b_hi, idesc,
                                                t == 0 ? acc_cb : 1u);
                                }
                                any = true;
                                umma_commit(&b_empty[bs]);
                                if (++bs == SB) bs = 0, bph ^= 1u;
                            }
                        }
                    } else if (RES) {
                        int ry = 0, rx = 0;
                        tc_fence_after();
                        uint32_t b_lo = b_res0 + (uint32_t)(cb * KK) * ((uint32_t)(BN * kRowBytes) >> 4);
                        for (int t = 0; t < KK; ++t) {
                            const uint32_t a_lo =
                                a_lo0 + (uint32_t)(ry * kHaloPitch + rx) * (kRowBytes >> 4);
                            for (int m = 0; m < MT; ++m)
                                umma4_kmajor<FMT == 2>(d_tmem + m * BN,
                                                       a_lo + m * ((16u * kHaloRowBytes) >> 4), a_hi,
                                                       b_lo, b_hi, idesc, t == 0 ? acc_cb : 1u);
                            b_lo += (uint32_t)(BN * kRowBytes) >> 4;
                            if (++rx == p.KW) rx = 0, ++ry;
                        }
                        any = true;
                    } else {
                        int ry = 0, rx = 0, t = 0;
                        for (int t0 = 0; t0 < KK; t0 += TB) {
                            if (!mbar_wait(&b_full[bs], bph, p.timeout_ns, abort_flag, p.err)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            uint32_t b_lo = b_ring0 + (uint32_t)bs * ((uint32_t)BB >> 4);
                            const int nt = min(TB, KK - t0);
                            for (int tt = 0; tt < nt; ++tt, ++t) {
                                const uint32_t a_lo =
                                    a_lo0 + (uint32_t)(ry * kHaloPitch + rx) * (kRowBytes >> 4);
                                for (int m = 0; m < MT; ++m)
                                    umma4_kmajor<FMT == 2>(d_tmem + m * BN,
                                                           a_lo + m * ((16u * kHaloRowBytes) >> 4),
                                                           a_hi, b_lo, b_hi, idesc,
                                                           t == 0 ? acc_cb : 1u);
                                b_lo += (uint32_t)(BN * kRowBytes) >> 4;
                                if (++rx == p.KW) rx = 0, ++ry;
                            }
                            any = true;
                            umma_commit(&b_empty[bs]);
                            if (++bs == SB) bs = 0, bph ^= 1u;
                        }
                    }
                    if (!ok) break;
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
    } else if (warp < 2 + kHaloEpi) {
        epilogue_warp<BN, true, kHaloEpi, MT, kHaloStage, FORM>(p, &map_c, tmem_base, tfull, tempty,
                                                                stage_out, abort_flag, warp, lane, 128);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, HaloTmem<BN, MT>::cols);
    }
}

template <int BN, int FMT, int FORM>
cudaError_t launch_halo(const UmmaParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                        const CUtensorMap &mc, int grid, cudaStream_t stream)
{
    int dev = 0;
    cudaGetDevice(&dev);
    // resident weights take one M tile; two M tiles need 2 x 2 x BN <= 512 TMEM columns
    const int mt = (p.box_h == 32 && BN <= 128) ? 2 : 1;
    const int which = p.res_b_bytes > 0 ? 0 : mt;
    auto kern = which == 0   ? umma_conv_halo_kernel<BN, FMT, true, 1, FORM>
                : which == 1 ? umma_conv_halo_kernel<BN, FMT, false, 1, FORM>
                             : umma_conv_halo_kernel<BN, FMT, false, (BN <= 128 ? 2 : 1), FORM>;
    static unsigned long long attr_set[3] = {0, 0, 0};   // bit per device: smem opt-in done
    if (dev >= 64 || !(attr_set[which] >> dev & 1ull)) {
        DeviceState *ds = device_state();
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ds ? ds->max_smem_optin : (int)p.halo_smem);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set[which] |= 1ull << dev;
    }
    return launch_pdl(kern, dim3(grid), dim3(kThreads), (size_t)p.halo_smem, stream, ma, mb, mc, p);
}

template <int FMT, int FORM = 0>
cudaError_t dispatch_halo_bn(int bn, const UmmaParams &p, const CUtensorMap &ma,
                             const CUtensorMap &mb, const CUtensorMap &mc, int grid, cudaStream_t s)
{
    switch (bn) {
    case 64: return launch_halo<64, FMT, FORM>(p, ma, mb, mc, grid, s);
    case 128: return launch_halo<128, FMT, FORM>(p, ma, mb, mc, grid, s);
    case 256: return launch_halo<256, FMT, FORM>(p, ma, mb, mc, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

}  // namespace bigemm
