// umma_main.cuh -- the implicit-GEMM kernel of the per-tap (nhwc) and direct
// operand modes, and its launch dispatch, shared by umma_conv.cu (weights
// streamed through the ring) and umma_res.cu (weights resident in shared
// memory).  Included once per translation unit; everything is internal.
#pragma once
#include "umma_common.cuh"

namespace bigemm {

namespace {

constexpr int kResMaxA = 10;   // A stages at most with resident weights

// RB (resident weights, split 1): the block's output-channel tile is the
// same for all its units (the grid is a multiple of the tile count, and units
// advance by the grid), so the producer loads every K block of that tile's
// weights once, into shared memory laid out by main_res_layout, and the ring
// carries only the A boxes.
// NEPI: epilogue warps, 8 (two per TMEM lane quadrant) or 16 (four, for
// BN = 128: each warp then drains one 32-channel chunk per tile; for BN = 64:
// two groups of eight take alternate units), so the quadrant's stores and
// address arithmetic run in more warps at once.  The 16
// warps stage 2 KB each, so the shared-memory layout is the same.  (At
// BN = 256 the 576-thread block's register budget would spill.)
template <int NEPI>
constexpr int main_threads() { return 64 + 32 * NEPI; }

// FORM: the epilogue's output form (epilogue_warp).
template <int BN, int AMODE, int FMT, bool RB, int NEPI, int FORM>
__global__ void __launch_bounds__(main_threads<NEPI>(), 1)
    umma_conv_kernel(const __grid_constant__ CUtensorMap map_a,
                     const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_c, const UmmaParams p)
{
    using C = Cfg<BN>;
    constexpr int SMAX = RB ? kResMaxA : C::stages;
    const int S = RB ? p.halo_sa : C::stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sa = smem;
    uint8_t *sb = RB ? smem + p.halo_b_off : smem + S * kABytes;
    uint8_t *stage_out = RB ? smem + p.halo_stage_off : sb + S * C::b_bytes;   // 32 KB of staging
    uint64_t *full = reinterpret_cast<uint64_t *>(RB ? smem + p.halo_bar_off : stage_out + C::staging);
    uint64_t *empty = full + SMAX;
    uint64_t *tfull = empty + SMAX;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *b_full = drain + 1;                 // RB: the resident weights have landed
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(b_full + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    // RB: the block's output-channel tile
    const int ct_res = RB ? (int)(blockIdx.x % (unsigned)p.co_tiles) : 0;

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
            mbar_init(&tempty[i], NEPI / epi_groups(BN, NEPI));
        }
        mbar_init(drain, 1);
        mbar_init(b_full, 1);
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
    griddep_enter();   // the set-up above overlapped the previous kernel; its data is ready now

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // The warp walks the loop together: lane 0 waits for a free slot and
        // arms its barrier, then lanes 0..nbox-1 each issue one A box and lane
        // nbox the B tile, so the copies of a K block leave in one instruction.
        {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            uint32_t last_parity[SMAX];
            bool issued[SMAX];
            for (int i = 0; i < SMAX; ++i) issued[i] = false, last_parity[i] = 0;
            const bool res_load = RB && (int)blockIdx.x < p.units;
            if (res_load && lane == 0) {
                // every K block of the tile's weights, once
                mbar_arrive_expect_tx(b_full, (uint32_t)p.res_b_bytes);
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    uint32_t urem;
                    const int tap = (int)fd_divmod((uint32_t)kb, p.fd_cib, &urem);
                    const int bx = AMODE == A_NHWC ? tap * p.cip + (int)urem * p.bk : kb * p.bk;
                    tma_load_2d(sb + (size_t)kb * C::b_bytes, &map_b, b_full, bx, ct_res * BN);
                }
            }
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                const Unit w = decode(p, u);
                const int box0 = w.pt * p.bpt;
                const int nbox = min(p.bpt, p.total_boxes - box0);
                const uint32_t tx = (uint32_t)nbox * box_bytes + (RB ? 0u : (uint32_t)C::b_bytes);
                int mbx = 0, mby = 0, mbn = 0;
                if (AMODE == A_NHWC && p.im2col) {
                    // the tile's first output pixel, as its window's base position
                    uint32_t r, x;
                    mbn = (int)fd_divmod((uint32_t)box0 * 128u, p.fd_howo, &r);
                    const int y = (int)fd_divmod(r, p.fd_wo, &x);
                    mbx = (int)x * p.stride - p.pad;
                    mby = y * p.stride - p.pad;
                } else if (lane < nbox) {
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
                        if (AMODE == A_NHWC && p.im2col)
                            tma_load_im2col_4d(a_dst, &map_a, &full[stage], cb * p.bk, mbx, mby, mbn,
                                               (uint16_t)rx, (uint16_t)ry);
                        else if (AMODE == A_NHWC)
                            tma_load_4d(a_dst + lane * box_bytes, &map_a, &full[stage], cb * p.bk,
                                        mbx + rx, mby + ry, mbn);
                        else
                            tma_load_3d(a_dst + lane * box_bytes, &map_a, &full[stage], mbx, kb * p.bk, mbn);
                    } else if (!RB && lane == nbox) {
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
            if (res_load && lane == 0) {
                // the weights land before the block exits, consumed or not
                int local_abort = 0;
                mbar_wait(b_full, 0, p.timeout_ns, &local_abort, p.err);
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
            if (RB && (int)blockIdx.x < p.units)
                ok = mbar_wait(b_full, 0, p.timeout_ns, abort_flag, p.err);
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                const Unit w = decode(p, u);
                if (RB && w.ct != ct_res) {   // the grid keeps each block on one tile
                    atomicExch(p.err, 1 /* BIGEMM_ERR_INVALID_ARG */);
                    ok = false;
                    break;
                }
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
                    const uint32_t b_lo =
                        desc_lo(smem_u32(sb + (size_t)(RB ? kb : stage) * C::b_bytes), 16u);
                    if (AMODE == A_NHWC) {
                        umma4_kmajor<FMT == 2>(d_tmem, a_lo, a_hi, b_lo, b_hi, idesc,
                                               kb > w.kb0 ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_lohi<FMT == 2>(d_tmem, a_lo + k * (a_kstep >> 4), a_hi,
                                                b_lo + k * 2u, b_hi, idesc,
                                                (kb > w.kb0 || k > 0) ? 1u : 0u);
                    }
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
        static_assert(NEPI == kEpiWarps || (NEPI == 16 && (BN == 128 || BN == 64)),
                      "16 epilogue warps need BN = 128 or 64");
        epilogue_warp<BN, AMODE != A_DIRECT, NEPI, 1, kEpiWarps * 4096 / NEPI, FORM>(
            p, &map_c, tmem_base, tfull, tempty, stage_out, abort_flag, warp, lane, box_px);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, C::tmem_cols);
    }
}


template <int BN, int AMODE, int FMT, bool RB, int NEPI, int FORM>
cudaError_t launch_one(const UmmaParams &p, const CUtensorMap &ma, const CUtensorMap &mb,
                       const CUtensorMap &mc, int grid, cudaStream_t stream)
{
    auto kern = umma_conv_kernel<BN, AMODE, FMT, RB, NEPI, FORM>;
    static unsigned long long attr_set = 0;   // bit per device: smem opt-in done
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = RB ? (size_t)p.halo_smem : (size_t)Cfg<BN>::smem;
    if (dev >= 64 || !(attr_set >> dev & 1ull)) {
        DeviceState *ds = device_state();
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             RB ? (ds ? ds->max_smem_optin : (int)smem) : (int)smem);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr_set |= 1ull << dev;
    }
    return launch_pdl(kern, dim3(grid), dim3(main_threads<NEPI>()), smem, stream, ma, mb, mc, p);
}

template <int AMODE, int FMT, bool RB, int FORM>
cudaError_t dispatch_bn(int bn, bool epi16, const UmmaParams &p, const CUtensorMap &ma,
                        const CUtensorMap &mb, const CUtensorMap &mc, int grid, cudaStream_t s)
{
    switch (bn) {
    case 64:
        if (epi16) return launch_one<64, AMODE, FMT, RB, 16, FORM>(p, ma, mb, mc, grid, s);
        return launch_one<64, AMODE, FMT, RB, kEpiWarps, FORM>(p, ma, mb, mc, grid, s);
    case 128:
        if (epi16) return launch_one<128, AMODE, FMT, RB, 16, FORM>(p, ma, mb, mc, grid, s);
        return launch_one<128, AMODE, FMT, RB, kEpiWarps, FORM>(p, ma, mb, mc, grid, s);
    case 256:
        if (epi16) return cudaErrorInvalidValue;
        return launch_one<256, AMODE, FMT, RB, kEpiWarps, FORM>(p, ma, mb, mc, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

// FORM 0 for every operand format; the narrowed forms only where the
// launching translation unit asks for them (umma_plain_*.cu: 16-bit outputs,
// 16-bit operands; umma_add.cu: split-K adds into fp32, any operand format).
template <int AMODE, bool RB, int FORM = 0>
cudaError_t dispatch_fmt(int fmt, int bn, bool epi16, const UmmaParams &p, const CUtensorMap &ma,
                         const CUtensorMap &mb, const CUtensorMap &mc, int grid, cudaStream_t s)
{
    switch (fmt) {
    case 0: return dispatch_bn<AMODE, 0, RB, FORM>(bn, epi16, p, ma, mb, mc, grid, s);
    case 1: return dispatch_bn<AMODE, 1, RB, FORM>(bn, epi16, p, ma, mb, mc, grid, s);
    case 2:
        if constexpr (FORM == 1 || FORM == 2)
            return cudaErrorInvalidValue;   // 16-bit output forms take 16-bit operands
        else
            return dispatch_bn<AMODE, 2, RB, FORM>(bn, epi16, p, ma, mb, mc, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

}  // namespace bigemm
