// halo_pair_plain.cu -- the CTA-pair halo kernel (halo_pair_main.cuh)
// narrowed to 16-bit outputs with no epilogue op: written in place by TMA
// stores where the output rows allow them, else from registers.
#include "halo_pair_main.cuh"

namespace bigemm {

cudaError_t launch_halo_pair_plain(int bn, int fmt, bool tma, const UmmaParams &p,
                                   const CUtensorMap &map_a, const CUtensorMap &map_b,
                                   const CUtensorMap &map_c, int grid, cudaStream_t stream)
{
    if (fmt != 0 && fmt != 1) return cudaErrorInvalidValue;
    return tma ? dispatch_halo_pair<1>(bn, fmt, p, map_a, map_b, map_c, grid, stream)
               : dispatch_halo_pair<2>(bn, fmt, p, map_a, map_b, map_c, grid, stream);
}

}  // namespace bigemm
