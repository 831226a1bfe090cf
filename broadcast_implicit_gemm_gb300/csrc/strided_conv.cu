// strided_conv.cu -- the strided operand mode (a stride-2 1x1 convolution on
// 16-bit NCHW data read in place, strided_main.cuh): its shared-memory layout
// and its launch, every output form decided at run time; strided_plain.cu
// holds the kernels narrowed to 16-bit outputs with no epilogue op.
#include "strided_main.cuh"

namespace bigemm {

// Shared memory of the strided kernel for a tile of bn output channels: at
// least two operand / weight ring slots, then as many 32 KB staging slots as
// fit (two to kStridedMaxSS: the staging copies' latency is what paces the
// kernel), then more ring slots with what is left, beside the epilogue warps'
// 2 KB staging and the barriers.
bool strided_layout(int bn, int smem_limit, UmmaParams &p)
{
    const int slot = kABytes + bn * kRowBytes;
    const int stage_out = kEpiWarps * kStridedEpiStage;
    const int bars = (2 * kStridedMaxSS + 3 * kStridedMaxS + 5) * 8 + 16;
    const int fixed = stage_out + bars + 1024;
    int s = 2, ss = 0;
    for (int k = kStridedMaxSS; k >= 2 && !ss; --k)
        if (s * slot + k * kStridedStage + fixed <= smem_limit) ss = k;
    if (!ss) return false;
    while (s < kStridedMaxS && (s + 1) * slot + ss * kStridedStage + fixed <= smem_limit) ++s;
    p.halo_sa = s;
    p.halo_sb = ss;
    p.halo_b_off = s * kABytes + ss * kStridedStage;
    p.halo_stage_off = p.halo_b_off + s * bn * kRowBytes;
    p.halo_bar_off = p.halo_stage_off + stage_out;
    p.halo_smem = p.halo_bar_off + bars + 1024;
    p.res_b_bytes = 0;
    return true;
}

size_t strided_smem_bytes(int bn)
{
    UmmaParams p{};
    return strided_layout(bn, 1 << 30, p) ? (size_t)p.halo_smem : 0;
}

cudaError_t launch_strided_conv(int bn, int fmt, const UmmaParams &p, const CUtensorMap &map_a,
                                const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                                cudaStream_t stream)
{
    return dispatch_strided<0>(bn, fmt, p, map_a, map_b, map_c, grid, stream);
}

}  // namespace bigemm
