// umma_res.cu -- the per-tap (nhwc) and direct implicit-GEMM kernels with the
// weights of the block's output-channel tile resident in shared memory: they
// are loaded once per block, and only the pixel operand streams through the
// ring.  Worth it when a block runs several units of a small weight tile
// (1x1 convs, short K), where reloading the weights for every unit would move
// more bytes from L2 than the pixels themselves.
#include "umma_main.cuh"

namespace bigemm {

bool main_res_layout(int bn, int k_blocks, int smem_limit, UmmaParams &p)
{
    const long long b_bytes = (long long)k_blocks * bn * kRowBytes;
    const uint32_t staging = (uint32_t)kEpiWarps * 4096u;
    const uint32_t bars = (2 * kResMaxA + 6) * 8 + 16;
    const long long fixed = b_bytes + staging + bars + 1024;
    int sa = 0;
    for (int s = kResMaxA; s >= 2 && !sa; --s)
        if ((long long)s * kABytes + fixed <= smem_limit) sa = s;
    if (!sa) return false;
    p.halo_sa = sa;
    p.halo_sb = 0;
    p.halo_b_off = sa * kABytes;
    p.halo_stage_off = p.halo_b_off + (int)b_bytes;
    p.halo_bar_off = p.halo_stage_off + (int)staging;
    p.halo_smem = p.halo_bar_off + (int)bars + 1024;
    p.res_b_bytes = (int)b_bytes;
    return true;
}

cudaError_t launch_umma_res(int amode, int fmt, int bn, bool epi16, const UmmaParams &p,
                            const CUtensorMap &map_a, const CUtensorMap &map_b,
                            const CUtensorMap &map_c, int grid, cudaStream_t stream)
{
    if (p.split != 1 || grid % p.co_tiles != 0 || p.res_b_bytes <= 0) return cudaErrorInvalidValue;
    if (amode == A_NHWC)
        return dispatch_fmt<A_NHWC, true>(fmt, bn, epi16, p, map_a, map_b, map_c, grid, stream);
    if (amode == A_DIRECT)
        return dispatch_fmt<A_DIRECT, true>(fmt, bn, epi16, p, map_a, map_b, map_c, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace bigemm
