// noalloc.cu -- conv2d_nchw_run_noalloc: the channels-last implicit-GEMM
// convolution for callers that must not allocate device memory (code running
// where cudaMalloc is not allowed, or inside a memory budget fixed by someone
// else).  Its scratch -- the channels-last copy of the data, the re-laid-out
// kernel and the split-K partial sums -- lives in one fixed array in the
// library's own device memory, created when the library is loaded and kept
// until the process exits.  Nothing here calls cudaMalloc, cudaFree or any
// routine that allocates.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "internal.h"

namespace bigemm {

namespace {

// Upper bound of the scratch one call may use (bytes).  Held on every GPU that
// loads the library.
constexpr size_t kScratchBytes = 16u << 20;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[64];     // device address of g_scratch, per device
int g_sm_count[64];

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

template <typename T>
__global__ void na_pack_weights(const T *__restrict__ w, T *__restrict__ wp, int CO, int CI,
                                int KHKW, int cip)
{
    const long long total = (long long)CO * KHKW * cip;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(i % cip);
        const long long r = i / cip;
        const int t = (int)(r % KHKW);
        const int f = (int)(r / KHKW);
        wp[i] = c < CI ? w[((size_t)f * CI + c) * KHKW + t] : T(0);
    }
}

__device__ __forceinline__ float na_epi(int epi, float acc, float b, float eps)
{
    switch (epi) {
    case BIGEMM_EPI_NONE: return acc;
    case BIGEMM_EPI_BIAS: return acc + b;
    case BIGEMM_EPI_BIAS_EXP: return expf(acc + b);
    case BIGEMM_EPI_BIAS_RSQRT: return rsqrtf(acc + b + eps);
    case BIGEMM_EPI_BIAS_RELU: return fmaxf(acc + b, 0.f);
    default: return 1.0f / (acc + b);
    }
}

__global__ void na_splitk_reduce(const float *__restrict__ ws, int split, long long elems, int CO,
                                 int HoWo, int epi, const float *__restrict__ bias, float eps,
                                 void *__restrict__ out, int out_dt)
{
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < elems;
         i += (long long)gridDim.x * blockDim.x) {
        float s = ws[i];
        for (int k = 1; k < split; ++k) s += ws[(long long)k * elems + i];
        const int f = (int)((i / HoWo) % CO);
        const float v = na_epi(epi, s, epi ? bias[f] : 0.f, eps);
        if (out_dt == BIGEMM_F32)
            static_cast<float *>(out)[i] = v;
        else if (out_dt == BIGEMM_F16)
            static_cast<__half *>(out)[i] = __float2half_rn(v);
        else
            static_cast<__nv_bfloat16 *>(out)[i] = __float2bfloat16_rn(v);
    }
}

// Once per device, with that device current: the device address of the
// scratch array (in host code its name is only a host-side stand-in).
bigemm_status setup_device(int dev, void **addr, int *sms)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return BIGEMM_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            return BIGEMM_ERR_CUDA;
        g_sm_count[dev] = n;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    *sms = g_sm_count[dev];
    return BIGEMM_OK;
}

CUtensorMapDataType na_tma_dt(int dt)
{
    return dt == BIGEMM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
           : dt == BIGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

}  // namespace
}  // namespace bigemm

using namespace bigemm;

extern "C" bigemm_status conv2d_nchw_run_noalloc(int N, int H, int W, int CO, int CI, int KH,
                                                 int KW, int stride, int padding,
                                                 bigemm_dtype in_dtype, bigemm_dtype out_dtype,
                                                 bigemm_epilogue epi, const void *data,
                                                 const void *kernel, const float *bias, float eps,
                                                 void *out, int *timeout_flag, void *stream)
{
    if (N < 1 || H < 1 || W < 1 || CO < 1 || CI < 1 || KH < 1 || KW < 1 || stride < 1 || padding < 0)
        return BIGEMM_ERR_INVALID_ARG;
    if (in_dtype < BIGEMM_F32 || in_dtype > BIGEMM_BF16 || out_dtype < BIGEMM_F32 ||
        out_dtype > BIGEMM_BF16 || epi < BIGEMM_EPI_NONE || epi > BIGEMM_EPI_BIAS_RELU)
        return BIGEMM_ERR_INVALID_ARG;
    if (!data || !kernel || !out || (epi != BIGEMM_EPI_NONE && !bias)) return BIGEMM_ERR_INVALID_ARG;
    if (((uintptr_t)data | (uintptr_t)kernel | (uintptr_t)out) & 15) return BIGEMM_ERR_INVALID_ARG;
    if (timeout_flag && ((uintptr_t)timeout_flag & 3)) return BIGEMM_ERR_INVALID_ARG;
    const int Ho = out_extent(H, KH, stride, padding), Wo = out_extent(W, KW, stride, padding);
    if (Ho < 1 || Wo < 1) return BIGEMM_ERR_INVALID_ARG;
    if (stride > 8 || N > 65535 || (long long)H * W > (1ll << 30)) return BIGEMM_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BIGEMM_ERR_CUDA;
    void *scratch = nullptr;
    int sms = 0;
    bigemm_status st = setup_device(dev, &scratch, &sms);
    if (st != BIGEMM_OK) return st;
    // Without a caller's flag the kernels raise the library's sticky error word
    // (itself a file-scope device variable, so this allocates nothing either).
    DeviceState *ds = timeout_flag ? nullptr : device_state();
    if (!timeout_flag && (!ds || !ds->err)) return BIGEMM_ERR_CUDA;

    // Tiling: 128 output pixels per tile as two 8x8 boxes, BN output channels,
    // K blocks of 128 bytes of channels per tap; split K when the tiles alone
    // would leave most SMs idle.
    const int e = (int)dtype_size(in_dtype);
    UmmaTiling t{};
    t.amode = A_NHWC;
    t.bn = CO <= 64 ? 64 : (CO <= 128 || CO % 256) ? 128 : 256;
    t.box_w = 8, t.box_h = 8, t.bpt = 2;
    UmmaParams p{};
    p.N = N, p.CI = CI, p.H = H, p.W = W, p.CO = CO, p.KH = KH, p.KW = KW;
    p.stride = stride, p.pad = padding, p.Ho = Ho, p.Wo = Wo;
    p.bk = 128 / e;
    p.ci_blocks = (int)cdiv(CI, p.bk);
    p.box_w = t.box_w, p.box_h = t.box_h, p.bpt = t.bpt;
    p.boxes_x = (int)cdiv(Wo, t.box_w);
    p.boxes_y = (int)cdiv(Ho, t.box_h);
    const long long bpi = (long long)p.boxes_x * p.boxes_y;
    if ((long long)N * bpi >= (1ll << 30)) return BIGEMM_ERR_UNSUPPORTED;
    p.boxes_per_img = (int)bpi;
    p.k_blocks = KH * KW * p.ci_blocks;
    p.cip = p.ci_blocks * p.bk;
    p.total_boxes = N * p.boxes_per_img;
    p.pix_tiles = (int)cdiv(p.total_boxes, t.bpt);
    p.co_tiles = (int)cdiv(CO, t.bn);
    const long long tiles = (long long)p.pix_tiles * p.co_tiles;
    p.out_elems = (long long)N * CO * Ho * Wo;

    // Scratch layout: [channels-last data | packed kernel | partial sums].
    const int ch = (int)cdiv(CI, 16 / e) * (16 / e);
    const size_t off_x = 0;
    const size_t xh_bytes = (size_t)N * H * W * ch * e;
    const size_t off_w = off_x + round256(xh_bytes);
    const size_t wp_bytes = (size_t)CO * KH * KW * p.cip * e;
    const size_t off_ws = off_w + round256(wp_bytes);
    if (off_ws > kScratchBytes) return BIGEMM_ERR_UNSUPPORTED;
    // K slices: enough to give most SMs a unit when the tiles alone would
    // leave them idle, then fewer until the partial sums fit in what is left
    // of the array (split 1 needs none).
    const long long room = (long long)((kScratchBytes - off_ws) / sizeof(float));
    int split = 1;
    if (tiles * 2 < sms && p.k_blocks >= 4)
        split = (int)std::max(1ll, std::min(cdiv(sms, tiles), (long long)p.k_blocks / 2));
    for (;;) {
        p.kb_per_split = (int)cdiv(p.k_blocks, split);
        p.split = (int)cdiv(p.k_blocks, p.kb_per_split);
        if (p.split == 1 || (long long)p.split * p.out_elems <= room) break;
        split = p.split - 1;
    }
    t.split = p.split;
    if (tiles * p.split >= (1ll << 31)) return BIGEMM_ERR_UNSUPPORTED;
    p.units = (int)(tiles * p.split);
    p.epi = epi, p.eps = eps, p.bias = bias, p.out_dt = out_dtype;
    p.timeout_ns = wait_timeout_ns();
    unsigned char *base = static_cast<unsigned char *>(scratch);
    int *err = timeout_flag ? timeout_flag : ds->err;
    void *xh = base + off_x, *wp = base + off_w;
    float *ws = p.split > 1 ? reinterpret_cast<float *>(base + off_ws) : nullptr;
    p.err = err;
    p.ws = ws;
    p.out = out;

    CUtensorMap map_a, map_b;
    const uint64_t dims[4] = {(uint64_t)ch, (uint64_t)W, (uint64_t)H, (uint64_t)N};
    const uint64_t str[3] = {(uint64_t)ch * e, (uint64_t)W * ch * e, (uint64_t)H * W * ch * e};
    const uint32_t box[4] = {(uint32_t)p.bk, (uint32_t)(t.box_w * stride),
                             (uint32_t)(t.box_h * stride), 1u};
    const uint32_t es[4] = {1u, (uint32_t)stride, (uint32_t)stride, 1u};
    if (!encode_tiled(&map_a, na_tma_dt(in_dtype), 4, xh, dims, str, box, es,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return BIGEMM_ERR_UNSUPPORTED;
    const uint64_t kt = (uint64_t)KH * KW * p.cip;
    const uint64_t bd[2] = {kt, (uint64_t)CO};
    const uint64_t bs[1] = {kt * e};
    const uint32_t bb[2] = {(uint32_t)p.bk, (uint32_t)t.bn};
    const uint32_t bes[2] = {1u, 1u};
    if (!encode_tiled(&map_b, na_tma_dt(in_dtype), 2, wp, bd, bs, bb, bes,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return BIGEMM_ERR_UNSUPPORTED;

    cudaStream_t s = (cudaStream_t)stream;
    if (launch_pack_nhwc(data, xh, N, CI, H * W, ch, in_dtype, s) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    const long long wtotal = (long long)CO * KH * KW * p.cip;
    const int wgrid = (int)std::min<long long>(cdiv(wtotal, 256), (long long)sms * 16);
    if (e == 4)
        na_pack_weights<uint32_t><<<wgrid, 256, 0, s>>>(static_cast<const uint32_t *>(kernel),
                                                        static_cast<uint32_t *>(wp), CO, CI,
                                                        KH * KW, p.cip);
    else
        na_pack_weights<uint16_t><<<wgrid, 256, 0, s>>>(static_cast<const uint16_t *>(kernel),
                                                        static_cast<uint16_t *>(wp), CO, CI,
                                                        KH * KW, p.cip);
    if (cudaGetLastError() != cudaSuccess) return BIGEMM_ERR_CUDA;
    const int grid = (int)std::min<long long>(p.units, sms);
    // p.store_tma = 0: the epilogue stores straight from registers (map_c unread)
    if (launch_umma_conv(t, in_dtype, p, map_a, map_b, map_a, grid, s) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    if (p.split > 1) {
        const int rgrid = (int)std::min<long long>(cdiv(p.out_elems, 256), (long long)sms * 16);
        na_splitk_reduce<<<rgrid, 256, 0, s>>>(ws, p.split, p.out_elems, CO, Ho * Wo, epi, bias,
                                               eps, out, out_dtype);
        if (cudaGetLastError() != cudaSuccess) return BIGEMM_ERR_CUDA;
    }
    return BIGEMM_OK;
}
