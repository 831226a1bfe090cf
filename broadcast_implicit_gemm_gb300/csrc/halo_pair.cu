// halo_pair.cu -- the halo-mode kernel for CTA pairs (halo_pair_main.cuh):
// its launch with the output form decided at run time; halo_pair_plain.cu
// holds the forms narrowed to 16-bit outputs with no epilogue op.
#include "halo_pair_main.cuh"

namespace bigemm {

cudaError_t launch_halo_pair(int bn, int fmt, const UmmaParams &p, const CUtensorMap &map_a,
                             const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                             cudaStream_t stream)
{
    if (fmt != 2 && !p.ws && !p.red_add && p.out_dt != BIGEMM_F32 && p.epi == BIGEMM_EPI_NONE)
        return launch_halo_pair_plain(bn, fmt, p.store_tma != 0, p, map_a, map_b, map_c, grid,
                                      stream);
    return dispatch_halo_pair<0>(bn, fmt, p, map_a, map_b, map_c, grid, stream);
}

}  // namespace bigemm
