// halo_pair_main.cuh -- the halo-mode implicit-GEMM kernel for a CTA pair:
// a cluster of two CTAs shares each MMA (tcgen05.mma.cta_group::2, M = 256).
// Included by halo_pair.cu (every output form) and halo_pair_plain.cu (the
// narrowed 16-bit forms); everything is internal.
//
// Why: a 128 x N x 16 MMA reads its A rows (4 KB) and its B rows (N x 32 bytes)
// from the SM's shared memory, and at N = 64 those reads, not the arithmetic,
// set its pace (measured: 52 cycles per MMA against 32 of arithmetic; 69 when
// the A start moves every four MMAs, as the halo taps do).  With a CTA pair
// each SM reads its own 128 rows of A and only half of B, the two halves
// meeting in both SMs' tensor cores, so the operand bytes per MMA fall from
// 6 KB to 5 KB at N = 64.
//
// Layout and protocol (resident weights, one 128-pixel halo tile per CTA):
//  * each CTA keeps output channels [rank * BN/2, (rank + 1) * BN/2) of every
//    tap's weights (K-major, 128-byte swizzle) and loads its own halo tile
//    (tile 2u + rank of pair unit u) into the same shared-memory offsets as its
//    partner;
//  * its TMA copies complete on the even CTA's barriers (the cta_group::2 form
//    of the copy, addressed through mapa), where the even CTA's producer arms
//    the bytes of both;
//  * the even CTA's MMA lane issues the pair's MMAs; each commit is multicast
//    to the same barrier in both CTAs (halo slot free, accumulator ready);
//  * each CTA's epilogue drains its own TMEM lanes (its 128 pixels, all BN
//    channels) and hands the accumulator back on the even CTA's barrier, which
//    counts both CTAs' epilogue warps;
//  * TMEM is allocated and freed by one warp of each CTA together, and the two
//    CTAs meet at a cluster barrier after set-up and before exit (so neither
//    leaves while the other may still touch its shared memory).  Every other
//    wait is bounded like mbar_wait.
#pragma once
#include "halo_main.cuh"

namespace bigemm {

namespace {

template <int BN, int FMT, int FORM>
__global__ void __launch_bounds__(kThreads, 1)
    umma_conv_halo_pair_kernel(const __grid_constant__ CUtensorMap map_a,
                               const __grid_constant__ CUtensorMap map_b,
                               const __grid_constant__ CUtensorMap map_c, const UmmaParams p)
{
    constexpr int BH = BN / 2;                        // output channels of B this CTA holds
    constexpr uint32_t kBHalf = (uint32_t)BH * kRowBytes;   // one tap's weight half
    constexpr uint32_t kCols = HaloTmem<BN, 1>::cols;
    const int SA = p.halo_sa;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t halo_bytes = (uint32_t)(16 + p.KH - 1) * kHaloRowBytes;
    const uint32_t a_stride = halo_bytes;
    uint8_t *sa = smem;
    uint8_t *sb = smem + p.halo_b_off;
    uint8_t *stage_out = smem + p.halo_stage_off;
    uint64_t *a_full = reinterpret_cast<uint64_t *>(smem + p.halo_bar_off);
    uint64_t *a_empty = a_full + kHaloMaxA;
    uint64_t *b_full = a_empty + kHaloMaxA;
    uint64_t *tfull = b_full + 1;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KK = p.KH * p.KW;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int u_first = (int)(blockIdx.x >> 1), u_step = (int)(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int i = 0; i < SA; ++i) mbar_init(&a_full[i], 1), mbar_init(&a_empty[i], 1);
        mbar_init(b_full, 1);
        // the accumulator comes back from both CTAs' epilogue warps
        for (int i = 0; i < 2; ++i) mbar_init(&tfull[i], 1), mbar_init(&tempty[i], 2 * kHaloEpi);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
        if (p.store_tma) tma_prefetch_desc(&map_c);
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc_pair(tmem_holder, kCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync_all();   // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    griddep_enter();   // the set-up above overlapped the previous kernel; its data is ready now

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t a_full_even = mapa_shared(smem_u32(a_full), 0);
            const uint32_t b_full_even = mapa_shared(smem_u32(b_full), 0);
            int as = 0;
            uint32_t aph = 0;
            uint32_t a_par[kHaloMaxA];
            bool a_iss[kHaloMaxA];
            for (int i = 0; i < kHaloMaxA; ++i) a_iss[i] = false, a_par[i] = 0;
            bool ok = true;
            // this CTA's half of every tap of every channel block, once; the
            // even CTA arms the bytes of both halves
            if (leader) mbar_arrive_expect_tx(b_full, 2u * (uint32_t)p.res_b_bytes);
            for (int cb = 0; cb < p.ci_blocks; ++cb)
                for (int t = 0; t < KK; ++t)
                    tma_load_3d_pair(sb + (size_t)(cb * KK + t) * kBHalf, &map_b, b_full_even,
                                     cb * p.bk, (int)rank * BH, t);
            for (int u = u_first; ok && u < p.units; u += u_step) {
                const Unit w = decode(p, u);
                const int pt = 2 * w.pt + (int)rank;   // this CTA's tile (past the last: zeros)
                uint32_t urem;
                const int n = (int)fd_divmod((uint32_t)pt, p.fd_bpi, &urem);
                const int byi = (int)fd_divmod(urem, p.fd_bx, &urem), bxi = (int)urem;
                const int x0 = bxi * 8 - p.pad, y0 = byi * 16 - p.pad;
                for (int cb = w.kb0; cb < w.kb1; ++cb) {
                    if (!mbar_wait(&a_empty[as], aph ^ 1u, p.timeout_ns, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(&a_full[as], 2u * halo_bytes);
                    a_iss[as] = true, a_par[as] = aph;
                    tma_load_4d_pair(sa + as * a_stride, &map_a, a_full_even + (uint32_t)as * 8u,
                                     cb * p.bk, x0, y0, n);
                    if (++as == SA) as = 0, aph ^= 1u;
                }
            }
            if (leader) {
                // the even CTA's barriers count both CTAs' copies: let every
                // armed round land (the weights too) before the pair exits
                int local_abort = 0;
                if (!ok)
                    for (int i = 0; i < SA; ++i)
                        if (a_iss[i]) mbar_wait(&a_full[i], a_par[i], p.timeout_ns, &local_abort, p.err);
                mbar_wait(b_full, 0, p.timeout_ns, &local_abort, p.err);
            } else if (!ok) {
                // the odd CTA cannot wait on the even CTA's barriers: give the
                // copies it issued a bounded time to land
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 20000ull) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (leader && lane == 0) {
            constexpr uint32_t idesc =
                make_idesc(FMT == 2 ? 2u : (uint32_t)FMT, 0u, 0u, 2 * kTileM, BN);
            const uint32_t a_hi = desc_hi((uint32_t)kHaloRowBytes, 2u), b_hi = desc_hi(1024u, 2u);
            constexpr uint32_t kBStep = kBHalf >> 4;
            int as = 0, acc = 0;
            uint32_t aph = 0, acc_phase = 0;
            bool ok = true, any = false;
            if (u_first < p.units) ok = mbar_wait(b_full, 0, p.timeout_ns, abort_flag, p.err);
            const uint32_t b_res0 = desc_lo(smem_u32(sb), 16u);
            for (int u = u_first; ok && u < p.units; u += u_step) {
                const Unit w = decode(p, u);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.timeout_ns, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                uint32_t accum = 0;
                for (int cb = w.kb0; cb < w.kb1; ++cb) {
                    if (!mbar_wait(&a_full[as], aph, p.timeout_ns, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_lo0 = desc_lo(smem_u32(sa + as * a_stride), 16u);
                    const uint32_t acc_cb = accum;   // accumulate into the tile from the first MMA on?
                    accum = 1u;
                    const uint32_t b_lo = b_res0 + (uint32_t)(cb * KK) * kBStep;
                    if (p.KH == 3 && p.KW == 3) {
                        // 3x3: every tap's A start and B slot are constants, the loop unrolls
                        constexpr uint32_t kTapOff[9] = {0, 8, 16, 128, 136, 144, 256, 264, 272};
#pragma unroll
                        for (int t = 0; t < 9; ++t)
                            umma4_kmajor_pair<FMT == 2>(d_tmem, a_lo0 + kTapOff[t], a_hi,
                                                        b_lo + (uint32_t)t * kBStep, b_hi, idesc,
                                                        t == 0 ? acc_cb : 1u);
                    } else {
                        int ry = 0, rx = 0;
                        for (int t = 0; t < KK; ++t) {
                            const uint32_t a_lo =
                                a_lo0 + (uint32_t)(ry * kHaloPitch + rx) * (kRowBytes >> 4);
                            umma4_kmajor_pair<FMT == 2>(d_tmem, a_lo, a_hi,
                                                        b_lo + (uint32_t)t * kBStep, b_hi, idesc,
                                                        t == 0 ? acc_cb : 1u);
                            if (++rx == p.KW) rx = 0, ++ry;
                        }
                    }
                    any = true;
                    umma_commit_pair_mc(&a_empty[as], (uint16_t)3u);
                    if (++as == SA) as = 0, aph ^= 1u;
                }
                if (!ok) break;
                umma_commit_pair_mc(&tfull[acc], (uint16_t)3u);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && any) {
                // every MMA issued so far completes before the pair's TMEM is freed
                int local_abort = 0;
                umma_commit_pair(drain);
                mbar_wait(drain, 0, p.timeout_ns, &local_abort, p.err);
            }
        }
    } else if (warp < 2 + kHaloEpi) {
        epilogue_warp<BN, true, kHaloEpi, 1, kHaloStage, FORM, true>(
            p, &map_c, tmem_base, tfull, tempty, stage_out, abort_flag, warp, lane, 128);
    }

    tc_fence_before();
    __syncwarp();
    cluster_sync_all();   // neither CTA leaves while its partner may still use its memory
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc_pair(tmem_base, kCols);
    }
}

template <int BN, int FMT, int FORM>
cudaError_t launch_halo_pair_one(const UmmaParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                                 const CUtensorMap &mc, int grid, cudaStream_t stream)
{
    if (grid < 2 || grid % 2) return cudaErrorInvalidValue;
    auto kern = umma_conv_halo_pair_kernel<BN, FMT, FORM>;
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)p.halo_smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, p);
}

template <int FORM>
cudaError_t dispatch_halo_pair(int bn, int fmt, const UmmaParams &p, const CUtensorMap &ma,
                               const CUtensorMap &mb, const CUtensorMap &mc, int grid,
                               cudaStream_t s)
{
    switch (bn) {
    case 64:
        return fmt == 0   ? launch_halo_pair_one<64, 0, FORM>(p, ma, mb, mc, grid, s)
               : fmt == 1 ? launch_halo_pair_one<64, 1, FORM>(p, ma, mb, mc, grid, s)
                          : launch_halo_pair_one<64, 2, FORM>(p, ma, mb, mc, grid, s);
    case 128:
        return fmt == 0   ? launch_halo_pair_one<128, 0, FORM>(p, ma, mb, mc, grid, s)
               : fmt == 1 ? launch_halo_pair_one<128, 1, FORM>(p, ma, mb, mc, grid, s)
                          : launch_halo_pair_one<128, 2, FORM>(p, ma, mb, mc, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

}  // namespace bigemm
