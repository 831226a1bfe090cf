// halo_forms_f32.cu -- the halo-mode kernel (halo_main.cuh) narrowed to fp32
// outputs written in place by TMA stores, the epilogue op chosen at run time
// (FORM 3 of epilogue_warp), for 16-bit operands; halo_conv.cu routes such
// launches here.
#include "halo_main.cuh"

namespace bigemm {

cudaError_t launch_halo_f32_tma(int bn, int fmt, const UmmaParams &p, const CUtensorMap &map_a,
                                const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                                cudaStream_t stream)
{
    if (fmt == 0) return dispatch_halo_bn<0, 3>(bn, p, map_a, map_b, map_c, grid, stream);
    if (fmt == 1) return dispatch_halo_bn<1, 3>(bn, p, map_a, map_b, map_c, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace bigemm
