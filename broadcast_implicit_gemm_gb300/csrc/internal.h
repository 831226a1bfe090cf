// internal.h -- types shared by the library's translation units (host side).
#pragma once
#include <cstddef>
#include <cstdint>
#include <string>
#include <utility>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/bigemm.h"
#include "fastdiv.h"

namespace bigemm {

inline size_t dtype_size(int dt) { return dt == BIGEMM_F32 ? 4 : 2; }

inline int out_extent(int in, int k, int s, int p)
{
    const int span = in + 2 * p - k;
    return span < 0 ? 0 : span / s + 1;
}

// Everything a conv kernel needs to know about the problem.
struct ConvShape {
    int N, CI, H, W, CO, KH, KW, stride, pad, groups;
    int Ho, Wo;
    int in_dt, out_dt, epi;
};

// -------------------------------------------------------------- UMMA kernel
// Operand-A (pixel) modes of the implicit GEMM.
enum AMode {
    A_NHWC = 0,     // packed channels-last copy of data, K-major, 4-D box per tap
    A_DIRECT = 1,   // 1x1 / stride 1 / pad 0: data read in place as [CI][H*W], MN-major
    A_HALO = 2,     // stride 1, K x K: one halo box per channel block serves every tap
    A_STRIDED = 3,  // 1x1 / stride 2 / pad 0, 16-bit: data read in place as rows of 2W
                    // elements (an even and an odd input row), the pixels the conv
                    // reads kept by compaction warps into an MN-major operand
};

// How the pack lays the data out for the A_NHWC / A_HALO kernels.
enum PackLayout {
    PACK_PLAIN = 0,   // [N][H][W][Ch]
    PACK_SUB = 1,     // 1x1, pad 0, stride s: [N][Ho][Wo][Ch] of the pixels the conv reads;
                      // the kernel then runs a stride-1 1x1 conv over it
    PACK_STACK = 2,   // stride 1: [N][H+pad][W][Ch], images stacked with pad zero rows
                      // between them, so a halo tile may span several images
    PACK_IM2COL = 3,  // [N][H][W][Ch] read by TMA im2col loads (A_NHWC): a tile is 128
                      // consecutive output pixels of the flattened N x Ho x Wo, across
                      // rows and images, and each tap's load walks their windows
};

struct UmmaTiling {
    int amode;        // AMode
    int pack;         // PackLayout
    int bres;         // weights resident in shared memory (A_HALO: one output-channel
                      // tile; A_NHWC / A_DIRECT: the block's tile, split 1)
    int bn;           // output channels per tile (N of the MMA), multiple of 32
    int stages;       // smem ring depth
    int box_w, box_h; // output pixels per TMA box (A_NHWC); A_DIRECT: box_w = row pixels
    int bpt;          // boxes per 128-pixel tile
    int split;        // K slices
    int epi16;        // A_NHWC / A_DIRECT, bn = 128: 16 epilogue warps (four per TMEM
                      // lane quadrant, 576 threads) instead of 8
    int pair;         // A_HALO with resident weights: clusters of two CTAs share each
                      // MMA (tcgen05 cta_group::2, M = 256), each holding half of B
};

struct UmmaParams {
    int N, CI, H, W, CO, KH, KW, stride, pad, Ho, Wo;
    int box_w, box_h, bpt;          // pixel boxes
    int boxes_x, boxes_y;           // boxes per image row / column (A_NHWC)
    int boxes_per_img;
    int total_boxes;
    int pix_tiles, co_tiles;
    int k_blocks, kb_per_split, split;
    int ci_blocks, bk;              // channels per K block (128 bytes)
    int cip;                        // packed weight channels per tap (A_NHWC)
    int units;
    int epi;
    float eps;
    const float *bias;
    void *out;
    int out_dt;
    float *ws;                      // split-K partial sums or null
    int red_add;                    // split-K into a zeroed fp32 output: each K slice adds
                                    // its partial tile to out (atomic adds; the first slice
                                    // adds the bias of EPI_BIAS), no workspace
    long long out_elems;
    int *err;
    unsigned long long timeout_ns;
    int store_tma;                  // 1: stage tiles in smem, write with TMA stores (map_c)
    int hp;                         // A_HALO over stacked images: rows per image (H + pad)
                                    // in the packed data and in tile row space; 0 otherwise
    int res_b_bytes;                // resident weights: their bytes (0: streamed)
    int im2col;                     // A_NHWC over PACK_IM2COL: tile pt is the flattened output
                                    // pixels 128 pt .. 128 pt + 127 (no boxes)
    // Dynamic shared-memory layout of the halo kernels (halo_layout) and of the
    // resident-weight nhwc / direct kernels (main_res_layout): A stages, streamed
    // weight stages, byte offsets of the weights, the output staging and the
    // barriers, and the total
    int halo_sa, halo_sb, halo_b_off, halo_stage_off, halo_bar_off, halo_smem;
    // divisors of the index arithmetic; launch_umma_conv fills them from the fields above
    FastDiv fd_co, fd_pix, fd_bpi, fd_bx, fd_hp, fd_cib, fd_kw, fd_howo, fd_wo;
};

// Returns a CUDA error code of the launch.
// map_c describes the output (or the split-K workspace) for TMA stores; it is
// read only when p.store_tma is set.
cudaError_t launch_umma_conv(const UmmaTiling &t, int in_dt, const UmmaParams &p,
                             const CUtensorMap &map_a, const CUtensorMap &map_b,
                             const CUtensorMap &map_c, int grid, cudaStream_t stream);
size_t umma_smem_bytes(const UmmaTiling &t);
// The halo kernel's shared-memory layout for a tiling (res: resident weights;
// rows: output rows per tile, 16 or 32), written into p; false when it does
// not fit in smem_limit bytes.
bool halo_layout(int bn, bool res, int rows, int kh, int kk, int ci_blocks, int smem_limit,
                 UmmaParams &p);
// The halo-mode kernels (halo_conv.cu); fmt 0 f16, 1 bf16, 2 tf32.
size_t halo_smem_bytes(int bn);
cudaError_t launch_halo_conv(int bn, int fmt, const UmmaParams &p, const CUtensorMap &map_a,
                             const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                             cudaStream_t stream);
bool umma_tiling_compiled(const UmmaTiling &t, int in_dt);
// The nhwc / direct kernels with resident weights (umma_res.cu): the layout
// (A stages, weights, output staging, barriers) of one output-channel tile's
// k_blocks K blocks, written into p's layout fields; false when it does not fit.
bool main_res_layout(int bn, int k_blocks, int smem_limit, UmmaParams &p);
// Launch; the grid must be a multiple of p.co_tiles and p.split must be 1.
// The halo kernel narrowed to an output form (16-bit operands): 16-bit output
// with no epilogue op by TMA stores or from registers, fp32 output by TMA
// stores (halo_forms_*.cu).
cudaError_t launch_halo_plain_tma(int bn, int fmt, const UmmaParams &p, const CUtensorMap &map_a,
                                  const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                                  cudaStream_t stream);
cudaError_t launch_halo_plain_reg(int bn, int fmt, const UmmaParams &p, const CUtensorMap &map_a,
                                  const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                                  cudaStream_t stream);
cudaError_t launch_halo_f32_tma(int bn, int fmt, const UmmaParams &p, const CUtensorMap &map_a,
                                const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                                cudaStream_t stream);
// The per-tap and direct kernels narrowed to a 16-bit output with no epilogue
// op, written in place by TMA stores (umma_plain_tma.cu) or from registers
// (umma_plain_reg.cu); 16-bit operand formats only.
cudaError_t launch_umma_plain_tma(int amode, bool rb, int fmt, int bn, bool epi16,
                                  const UmmaParams &p, const CUtensorMap &map_a,
                                  const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                                  cudaStream_t stream);
cudaError_t launch_umma_plain_reg(int amode, bool rb, int fmt, int bn, bool epi16,
                                  const UmmaParams &p, const CUtensorMap &map_a,
                                  const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                                  cudaStream_t stream);
// The per-tap and direct kernels narrowed to split-K slices added into an fp32
// output (umma_add.cu), weights streamed.
cudaError_t launch_umma_add(int amode, int fmt, int bn, bool epi16, const UmmaParams &p,
                            const CUtensorMap &map_a, const CUtensorMap &map_b,
                            const CUtensorMap &map_c, int grid, cudaStream_t stream);
cudaError_t launch_umma_res(int amode, int fmt, int bn, bool epi16, const UmmaParams &p,
                            const CUtensorMap &map_a, const CUtensorMap &map_b,
                            const CUtensorMap &map_c, int grid, cudaStream_t stream);

// The CTA-pair halo kernels (halo_pair.cu, halo_pair_plain.cu): resident
// weights, one 16 x 8 tile per CTA, p.units pair units (tiles 2u and 2u + 1),
// an even grid; the second form is narrowed to 16-bit outputs with no
// epilogue op (tma: written by TMA stores, else from registers).
cudaError_t launch_halo_pair(int bn, int fmt, const UmmaParams &p, const CUtensorMap &map_a,
                             const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                             cudaStream_t stream);
cudaError_t launch_halo_pair_plain(int bn, int fmt, bool tma, const UmmaParams &p,
                                   const CUtensorMap &map_a, const CUtensorMap &map_b,
                                   const CUtensorMap &map_c, int grid, cudaStream_t stream);

// The strided-mode kernels (strided_conv.cu, strided_plain.cu): the
// shared-memory layout for a tile of bn output channels, written into p's
// layout fields (false when it does not fit in smem_limit bytes); its size
// without a limit; the launch with every output form, and the one narrowed to
// 16-bit outputs with no epilogue op (tma: written by TMA stores, else from
// registers).  fmt 0 f16, 1 bf16.
bool strided_layout(int bn, int smem_limit, UmmaParams &p);
size_t strided_smem_bytes(int bn);
cudaError_t launch_strided_conv(int bn, int fmt, const UmmaParams &p, const CUtensorMap &map_a,
                                const CUtensorMap &map_b, const CUtensorMap &map_c, int grid,
                                cudaStream_t stream);
cudaError_t launch_strided_plain(int bn, int fmt, bool tma, const UmmaParams &p,
                                 const CUtensorMap &map_a, const CUtensorMap &map_b,
                                 const CUtensorMap &map_c, int grid, cudaStream_t stream);

// -------------------------------------------------------------- other kernels
cudaError_t launch_pack_nhwc(const void *x, void *xh, int N, int C, int HW, int Ch, int dt,
                             cudaStream_t stream);
// Both packs in one launch.  The data goes to a per-image [Hop][Wop][Ch] grid
// whose pixel (yo, xo) is input pixel (s*yo, s*xo), zero outside the image:
// (H, W, 1) is the plain copy, Hop > H adds zero rows below each image, s > 1
// subsamples.  xh must be 16-byte aligned.  zero (16-byte aligned, or null):
// zero_elems floats that the same launch sets to 0 (the output that split-K
// slices then add into).
cudaError_t launch_pack_operands(const void *x, void *xh, int N, int C, int H, int W, int Hop,
                                 int Wop, int s, int Ch, const void *w, void *wp, int CO, int CI,
                                 int KHKW, int cip, int dt, cudaStream_t stream,
                                 float *zero = nullptr, long long zero_elems = 0);
cudaError_t launch_splitk_reduce(const float *ws, int split, long long elems, int CO, int HoWo,
                                 int epi, const float *bias, float eps, void *out, int out_dt,
                                 cudaStream_t stream);
cudaError_t launch_simt_conv(const ConvShape &s, const void *x, const void *w,
                             const float *bias, float eps, void *out, int variant,
                             cudaStream_t stream);
cudaError_t launch_dw_conv(const ConvShape &s, const void *x, const void *w, const float *bias,
                           float eps, void *out, int rows_per_block, cudaStream_t stream);
// Streaming depthwise kernel (square 3/5/7 with pad K/2, stride 1 or 2).
bool dw_stream_ok(const ConvShape &s);
// rows: output rows per thread (2, 4 or 8).
cudaError_t launch_dw_stream(const ConvShape &s, const void *x, const void *w, const float *bias,
                             float eps, void *out, int rows, cudaStream_t stream);
// Whole-plane depthwise kernel for planes up to 32 x 32 (same kernels as the
// streaming one): one or two planes per warp staged in shared memory.
bool dw_plane_ok(const ConvShape &s);
cudaError_t launch_dw_plane(const ConvShape &s, const void *x, const void *w, const float *bias,
                            float eps, void *out, cudaStream_t stream);
// Small-plane depthwise kernel (stride 1, square 3/5/7 with pad K/2, outputs at
// most 16 wide and 32 tall): whole planes per warp in shared memory, ty x 8
// outputs per thread (ty = 2 or 4).
bool dw_small_ok(const ConvShape &s, int ty);
// Band depthwise kernel (square 3/5/7 with pad K/2, stride 1 or 2, input rows
// of whole 16-byte chunks up to 512 bytes): bands of rows per warp in shared
// memory, 4 x 8 outputs per thread.
bool dw_band_ok(const ConvShape &s);
cudaError_t launch_dw_band(const ConvShape &s, const void *x, const void *w, const float *bias,
                           float eps, void *out, cudaStream_t stream);
cudaError_t launch_dw_small(const ConvShape &s, const void *x, const void *w, const float *bias,
                            float eps, void *out, int ty, cudaStream_t stream);
// [1, P, 1] => [B0, P, B1]: the per-channel kernel for long rows, bcast_rows
// for short ones (bcast.cu).
bool bcast_long_rows(long long B1, int out_dt);
cudaError_t launch_bcast_general(int B0, int P, int B1, int op, const float *var, float eps,
                                 void *out, int out_dt, cudaStream_t stream);
cudaError_t launch_bcast(int N, int C, int HW, int op, const float *var, float eps, void *out,
                         int out_dt, int flat, cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(int *err, unsigned long long timeout_ns,
                                      cudaStream_t stream);

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel on the stream finishes; it calls griddepcontrol.wait
// before touching memory the previous kernel uses.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// -------------------------------------------------------------- runtime state
struct DeviceState {
    int device = -1;
    int sm_count = 0;
    int max_smem_optin = 0;
    int *err = nullptr;          // device address of the sticky error word (a file-scope
                                 // __device__ int, not an allocation)
};
// The current device's state; nullptr on failure.  Allocates nothing: the
// first call on a device queries its attributes and looks up the address of
// the error word (cudaGetSymbolAddress), so make it before any stream capture.
DeviceState *device_state();
unsigned long long wait_timeout_ns();

// Profiling hooks: record events around a launch when enabled.
struct ProfScope {
    ProfScope(const char *name, cudaStream_t s);
    ~ProfScope();
    const char *name_;
    cudaStream_t s_;
    int slot_ = -1;
};

// TMA descriptor encoding through the driver entry point.
bool encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                  const uint32_t *estrides, CUtensorMapSwizzle swz);
// An im2col descriptor over a 4-D channels-last tensor {C, W, H, N}: each load
// brings `pixels` consecutive pixels (W fastest, then H, then N) of `channels`
// channels, walking base positions from lower[d] to dims[d] - 1 + upper[d]
// (d = W, H) in steps of estrides[d + 1]; the load's offsets shift every
// pixel's read position, and reads outside the tensor are zeros.
bool encode_im2col(CUtensorMap *map, CUtensorMapDataType dt, const void *base,
                   const uint64_t *dims, const uint64_t *strides_bytes, const int *lower,
                   const int *upper, uint32_t channels, uint32_t pixels, const uint32_t *estrides,
                   CUtensorMapSwizzle swz);

}  // namespace bigemm
