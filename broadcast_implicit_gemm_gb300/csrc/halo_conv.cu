// halo_conv.cu -- the halo operand mode of the implicit-GEMM convolution
// (stride-1 K x K kernels): one input halo per channel block serves every tap.
#include "halo_main.cuh"

namespace bigemm {

bool halo_layout(int bn, bool res, int rows, int kh, int kk, int ci_blocks, int smem_limit,
                 UmmaParams &p)
{
    const uint32_t a_stride = (uint32_t)(rows + kh - 1) * kHaloRowBytes;
    const long long res_ll = (long long)ci_blocks * kk * bn * kRowBytes;
    if (res && res_ll >= (1ll << 20)) return false;
    // one streamed weight stage: 32 KB, or a single tap for two-tile units
    const uint32_t stage_b = rows == 32 ? (uint32_t)bn * kRowBytes : (uint32_t)HaloCfg<64>::b_bytes;
    const uint32_t staging = (uint32_t)kHaloEpi * kHaloStage;
    const uint32_t bars = (2 * kHaloMaxA + 2 * kHaloMaxB + 5) * 8 + 16;
    const uint32_t fixed = staging + bars + 1024;
    // resident weights: as many halo stages as fit; streamed: two halo stages
    // and as deep a weight ring as fits (then a third halo stage if room is left)
    int best_sa = 0, best_sb = 0;
    uint32_t b_bytes = 0;
    if (res) {
        for (int sa = kHaloMaxA; sa >= 2 && !best_sa; --sa)
            if ((uint32_t)sa * a_stride + (uint32_t)res_ll + fixed <= (uint32_t)smem_limit)
                best_sa = sa, best_sb = 1, b_bytes = (uint32_t)res_ll;
    } else {
        for (int sb = kHaloMaxB; sb >= 2 && !best_sa; --sb)
            if (2u * a_stride + (uint32_t)sb * stage_b + fixed <= (uint32_t)smem_limit)
                best_sa = 2, best_sb = sb, b_bytes = (uint32_t)sb * stage_b;
        while (best_sa > 0 && best_sa < kHaloMaxA &&
               (uint32_t)(best_sa + 1) * a_stride + b_bytes + fixed <= (uint32_t)smem_limit)
            ++best_sa;
    }
    if (!best_sa) return false;
    p.halo_sa = best_sa;
    p.halo_sb = best_sb;
    p.halo_b_off = (int)((uint32_t)best_sa * a_stride);
    p.halo_stage_off = p.halo_b_off + (int)b_bytes;
    p.halo_bar_off = p.halo_stage_off + (int)staging;
    p.halo_smem = p.halo_bar_off + (int)bars + 1024;
    p.res_b_bytes = res ? (int)b_bytes : 0;
    return true;
}

size_t halo_smem_bytes(int bn)
{
    switch (bn) {
    case 64: return HaloCfg<64>::smem;
    case 128: return HaloCfg<128>::smem;
    case 256: return HaloCfg<256>::smem;
    default: return 0;
    }
}

cudaError_t launch_halo_conv(int bn, int fmt, const UmmaParams &p, const CUtensorMap &map_a,
                             const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                             cudaStream_t stream)
{
    // outputs written in place with 16-bit operands take a kernel narrowed to
    // their output form: 16-bit with no epilogue op by TMA stores (1) or from
    // registers (2), or fp32 by TMA stores with the op chosen at run time (3)
    if (fmt != 2 && !p.ws && !p.red_add) {
        const int form = p.out_dt != BIGEMM_F32 ? (p.epi == BIGEMM_EPI_NONE ? (p.store_tma ? 1 : 2) : 0)
                                                : (p.store_tma ? 3 : 0);
        if (form == 1) return launch_halo_plain_tma(bn, fmt, p, map_a, map_b, map_c, grid, stream);
        if (form == 2) return launch_halo_plain_reg(bn, fmt, p, map_a, map_b, map_c, grid, stream);
        if (form == 3) return launch_halo_f32_tma(bn, fmt, p, map_a, map_b, map_c, grid, stream);
    }
    switch (fmt) {
    case 0: return dispatch_halo_bn<0>(bn, p, map_a, map_b, map_c, grid, stream);
    case 1: return dispatch_halo_bn<1>(bn, p, map_a, map_b, map_c, grid, stream);
    default: return dispatch_halo_bn<2>(bn, p, map_a, map_b, map_c, grid, stream);
    }
}

}  // namespace bigemm
