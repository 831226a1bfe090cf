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
#include "umma_common.cuh"

namespace bigemm {

namespace {

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
        epilogue_warp<BN, AMODE != A_DIRECT>(p, &map_c, tmem_base, tfull, tempty, stage_out,
                                             abort_flag, warp, lane, box_px);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem_base, C::tmem_cols);
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

size_t umma_smem_bytes(const UmmaTiling &t)
{
    if (t.amode == A_HALO) return halo_smem_bytes(t.bn);
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
    if (t.amode == A_HALO) return launch_halo_conv(t.bn, fmt, p, map_a, map_b, map_c, grid, stream);
    if (t.amode == A_NHWC)
        return dispatch_fmt<A_NHWC>(fmt, t.bn, p, map_a, map_b, map_c, grid, stream);
    return dispatch_fmt<A_DIRECT>(fmt, t.bn, p, map_a, map_b, map_c, grid, stream);
}

}  // namespace bigemm
