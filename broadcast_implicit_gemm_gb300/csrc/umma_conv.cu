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
// next.  Split-K slices add their partial tiles into a zeroed fp32 output, or
// write them to a workspace that a separate kernel sums in a fixed order
// before the epilogue.  The kernel itself is in umma_main.cuh; this file
// launches the form that streams the weights through the ring, umma_res.cu
// the form that keeps them resident.
#include "umma_main.cuh"

namespace bigemm {

namespace {

int fmt_of(int in_dt) { return in_dt == BIGEMM_F16 ? 0 : in_dt == BIGEMM_BF16 ? 1 : 2; }

}  // namespace

size_t umma_smem_bytes(const UmmaTiling &t)
{
    if (t.amode == A_HALO) return halo_smem_bytes(t.bn);
    if (t.amode == A_STRIDED) return strided_smem_bytes(t.bn);
    switch (t.bn) {
    case 64: return Cfg<64>::smem;
    case 128: return Cfg<128>::smem;
    case 256: return Cfg<256>::smem;
    default: return 0;
    }
}

bool umma_tiling_compiled(const UmmaTiling &t, int in_dt)
{
    return (t.bn == 64 || t.bn == 128 || t.bn == 256) &&
           (t.amode == A_NHWC || t.amode == A_DIRECT || t.amode == A_HALO ||
            (t.amode == A_STRIDED && in_dt != BIGEMM_F32));
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
    p.fd_howo = make_fastdiv((uint32_t)((long long)p.Ho * p.Wo));
    p.fd_wo = make_fastdiv((uint32_t)p.Wo);
    ProfScope prof(t.amode == A_NHWC      ? "umma_conv_nhwc"
                   : t.amode == A_HALO    ? (t.pair ? "umma_conv_halo_pair" : "umma_conv_halo")
                   : t.amode == A_STRIDED ? "umma_conv_strided"
                                          : "umma_conv_direct",
                   stream);
    const int fmt = fmt_of(in_dt);
    if (t.amode == A_HALO && t.pair)
        return launch_halo_pair(t.bn, fmt, p, map_a, map_b, map_c, grid, stream);
    if (t.amode == A_HALO) return launch_halo_conv(t.bn, fmt, p, map_a, map_b, map_c, grid, stream);
    const bool e16 = t.epi16 != 0;
    // a 16-bit output written in place with no epilogue op takes the kernel
    // whose epilogue carries only that path
    const bool plain = fmt != 2 && !p.ws && !p.red_add && p.epi == BIGEMM_EPI_NONE &&
                       p.out_dt != BIGEMM_F32;
    if (t.amode == A_STRIDED) {
        if (t.bres || e16) return cudaErrorInvalidValue;
        if (plain)
            return launch_strided_plain(t.bn, fmt, p.store_tma != 0, p, map_a, map_b, map_c, grid,
                                        stream);
        return launch_strided_conv(t.bn, fmt, p, map_a, map_b, map_c, grid, stream);
    }
    // split-K slices adding into an fp32 output take the kernel narrowed to that
    if (p.red_add && !p.ws && !t.bres && t.amode != A_HALO)
        return launch_umma_add(t.amode, fmt, t.bn, e16, p, map_a, map_b, map_c, grid, stream);
    if (plain && t.amode != A_HALO) {
        // the checks launch_umma_res makes for resident weights
        if (t.bres && (p.split != 1 || grid % p.co_tiles != 0 || p.res_b_bytes <= 0))
            return cudaErrorInvalidValue;
        if (p.store_tma)
            return launch_umma_plain_tma(t.amode, t.bres != 0, fmt, t.bn, e16, p, map_a, map_b,
                                         map_c, grid, stream);
        return launch_umma_plain_reg(t.amode, t.bres != 0, fmt, t.bn, e16, p, map_a, map_b, map_c,
                                     grid, stream);
    }
    if (t.bres) return launch_umma_res(t.amode, fmt, t.bn, e16, p, map_a, map_b, map_c, grid, stream);
    if (t.amode == A_NHWC)
        return dispatch_fmt<A_NHWC, false>(fmt, t.bn, e16, p, map_a, map_b, map_c, grid, stream);
    return dispatch_fmt<A_DIRECT, false>(fmt, t.bn, e16, p, map_a, map_b, map_c, grid, stream);
}

}  // namespace bigemm
