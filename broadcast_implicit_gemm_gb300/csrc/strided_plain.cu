// strided_plain.cu -- the strided-mode kernel (strided_main.cuh) narrowed to
// 16-bit outputs with no bias or epilogue op: written in place by TMA stores
// where the output rows allow them, else from registers.
#include "strided_main.cuh"

namespace bigemm {

cudaError_t launch_strided_plain(int bn, int fmt, bool tma, const UmmaParams &p,
                                 const CUtensorMap &map_a, const CUtensorMap &map_b,
                                 const CUtensorMap &map_c, int grid, cudaStream_t stream)
{
    return tma ? dispatch_strided<1>(bn, fmt, p, map_a, map_b, map_c, grid, stream)
               : dispatch_strided<2>(bn, fmt, p, map_a, map_b, map_c, grid, stream);
}

}  // namespace bigemm
