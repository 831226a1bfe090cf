// umma_plain_reg.cu -- the per-tap (nhwc) and direct implicit-GEMM kernels for
// 16-bit outputs that TMA cannot store (rows of Wo x 2 bytes that are not a
// multiple of 16), written from registers, with no bias or epilogue op.  The
// kernel is the one of umma_main.cuh with its epilogue narrowed to that form
// (FORM 2), so it carries none of the other output paths; umma_conv.cu routes
// such launches here.
#include "umma_main.cuh"

namespace bigemm {

cudaError_t launch_umma_plain_reg(int amode, bool rb, int fmt, int bn, bool epi16,
                                  const UmmaParams &p, const CUtensorMap &map_a,
                                  const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                                  cudaStream_t stream)
{
    if (amode == A_NHWC)
        return rb ? dispatch_fmt<A_NHWC, true, 2>(fmt, bn, epi16, p, map_a, map_b, map_c, grid, stream)
                  : dispatch_fmt<A_NHWC, false, 2>(fmt, bn, epi16, p, map_a, map_b, map_c, grid, stream);
    if (amode == A_DIRECT)
        return rb ? dispatch_fmt<A_DIRECT, true, 2>(fmt, bn, epi16, p, map_a, map_b, map_c, grid, stream)
                  : dispatch_fmt<A_DIRECT, false, 2>(fmt, bn, epi16, p, map_a, map_b, map_c, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace bigemm
