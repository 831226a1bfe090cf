// umma_add.cu -- the per-tap (nhwc) and direct implicit-GEMM kernels whose K
// slices add their partial tiles into an fp32 output (TMA reduce-add boxes, or
// atomic adds where TMA cannot address the rows), the first slice bringing the
// bias.  The kernel is the one of umma_main.cuh with its epilogue narrowed to
// that form (FORM 4); umma_conv.cu routes such launches here.
#include "umma_main.cuh"

namespace bigemm {

cudaError_t launch_umma_add(int amode, int fmt, int bn, bool epi16, const UmmaParams &p,
                            const CUtensorMap &map_a, const CUtensorMap &map_b,
                            const CUtensorMap &map_c, int grid, cudaStream_t stream)
{
    if (amode == A_NHWC)
        return dispatch_fmt<A_NHWC, false, 4>(fmt, bn, epi16, p, map_a, map_b, map_c, grid, stream);
    if (amode == A_DIRECT)
        return dispatch_fmt<A_DIRECT, false, 4>(fmt, bn, epi16, p, map_a, map_b, map_c, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace bigemm
