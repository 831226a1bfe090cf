// plan.cu -- conv plans: validation, candidate kernels, timed search, cache,
// and the conv entry points of the C ABI.
//
// The search follows the tuning flow of "Tuning High Performance Convolution
// on NVIDIA GPUs" (TVM v0.5 autotvm tutorial), Step 2: a small space of
// tilings (the analogue of its split knobs on f/y/x/rc and unroll options) is
// enumerated; invalid points are rejected on the host before any launch
// (its "invalid gpu kernel" records); each valid point is timed as three
// repeats of runs, each repeat lasting at least a minimum time (its repeat /
// min_repeat_ms measure option); and the best record is kept per workload,
// like its log of best configurations.  The candidates run on seeded non-zero
// inputs, and where the problem's tensors fit in L2 each timed run starts
// after an L2 flush, as in a step that reads its inputs from HBM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <map>
#include <mutex>
#include <sstream>
#include <string>
#include <vector>

#include "internal.h"

namespace bigemm {

size_t dw_smem_bytes(const ConvShape &s, int rows);

namespace {

enum SimtVariant { SV_NAIVE = 0, SV_TILED = 1, SV_DW = 2, SV_DWS = 3, SV_DWP = 4, SV_DWR = 5, SV_DWB = 6 };

struct Cand {
    int kind = BIGEMM_KIND_SIMT;
    int simt_variant = SV_NAIVE;
    int dw_rows = 8;
    UmmaTiling t{};
};

const char *amode_name(int amode)
{
    return amode == A_DIRECT ? "direct" : amode == A_HALO ? "halo" : amode == A_STRIDED ? "strided" : "nhwc";
}

std::string cand_str(const Cand &c)
{
    char b[160];
    if (c.kind == BIGEMM_KIND_UMMA)
        snprintf(b, sizeof b, "umma:%s:bn%d:box%dx%dx%d:split%d%s%s%s%s",
                 amode_name(c.t.amode), c.t.bn,
                 c.t.box_w, c.t.box_h, c.t.bpt, c.t.split,
                 c.t.pack == PACK_SUB     ? ":sub"
                 : c.t.pack == PACK_STACK ? ":stack"
                 : c.t.pack == PACK_IM2COL ? ":im2col"
                                           : "",
                 c.t.bres ? ":bres" : "", c.t.epi16 ? ":e16" : "", c.t.pair ? ":pair" : "");
    else if (c.simt_variant == SV_DW)
        snprintf(b, sizeof b, "simt:depthwise:rows%d", c.dw_rows);
    else if (c.simt_variant == SV_DWS)
        snprintf(b, sizeof b, "simt:depthwise:stream%d", c.dw_rows);
    else if (c.simt_variant == SV_DWP)
        snprintf(b, sizeof b, "simt:depthwise:plane");
    else if (c.simt_variant == SV_DWR)
        snprintf(b, sizeof b, "simt:depthwise:small%d", c.dw_rows);
    else if (c.simt_variant == SV_DWB)
        snprintf(b, sizeof b, "simt:depthwise:band");
    else
        snprintf(b, sizeof b, "simt:%s", c.simt_variant == SV_TILED ? "tiled" : "naive");
    return b;
}

bool parse_cand(const std::string &s, Cand &c)
{
    int a, b, d, e, f, g;
    char mode[16], layout[16] = "", layout2[16] = "", layout3[16] = "";
    const int got = sscanf(s.c_str(),
                           "umma:%15[a-z]:bn%d:box%dx%dx%d:split%d:%15[a-z0-9]:%15[a-z0-9]:%15[a-z0-9]",
                           mode, &a, &b, &d, &e, &f, layout, layout2, layout3);
    if (got >= 6 && got <= 9) {
        c = Cand{};
        c.kind = BIGEMM_KIND_UMMA;
        c.t.amode = strcmp(mode, "direct") == 0    ? A_DIRECT
                    : strcmp(mode, "halo") == 0    ? A_HALO
                    : strcmp(mode, "strided") == 0 ? A_STRIDED
                                                   : A_NHWC;
        c.t.pack = strcmp(layout, "sub") == 0      ? PACK_SUB
                   : strcmp(layout, "stack") == 0  ? PACK_STACK
                   : strcmp(layout, "im2col") == 0 ? PACK_IM2COL
                                                   : PACK_PLAIN;
        c.t.bres = strcmp(layout, "bres") == 0 || strcmp(layout2, "bres") == 0;
        c.t.epi16 = strcmp(layout, "e16") == 0 || strcmp(layout2, "e16") == 0 ||
                    strcmp(layout3, "e16") == 0;
        c.t.pair = strcmp(layout, "pair") == 0 || strcmp(layout2, "pair") == 0 ||
                   strcmp(layout3, "pair") == 0;
        c.t.bn = a, c.t.box_w = b, c.t.box_h = d, c.t.bpt = e, c.t.split = f;
        return true;
    }
    if (sscanf(s.c_str(), "simt:depthwise:rows%d", &g) == 1) {
        c = Cand{};
        c.simt_variant = SV_DW, c.dw_rows = g;
        return true;
    }
    if (sscanf(s.c_str(), "simt:depthwise:stream%d", &g) == 1 && (g == 2 || g == 4 || g == 8)) {
        c = Cand{};
        c.simt_variant = SV_DWS, c.dw_rows = g;
        return true;
    }
    if (s == "simt:depthwise:plane") return c = Cand{}, c.simt_variant = SV_DWP, true;
    if (s == "simt:depthwise:band") return c = Cand{}, c.simt_variant = SV_DWB, true;
    if (sscanf(s.c_str(), "simt:depthwise:small%d", &g) == 1 && (g == 2 || g == 4)) {
        c = Cand{};
        c.simt_variant = SV_DWR, c.dw_rows = g;
        return true;
    }
    if (s == "simt:tiled") return c = Cand{}, c.simt_variant = SV_TILED, true;
    if (s == "simt:naive") return c = Cand{}, c.simt_variant = SV_NAIVE, true;
    return false;
}

CUtensorMapDataType tma_dt(int dt)
{
    return dt == BIGEMM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
           : dt == BIGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

bool is_depthwise(const ConvShape &s) { return s.groups > 1 && s.groups == s.CI && s.CO == s.CI; }

// The conv the UMMA kernel computes: with the subsampling pack, a strided 1x1
// conv becomes a stride-1 1x1 conv over the [Ho][Wo] grid of pixels it reads.
ConvShape kernel_shape(const ConvShape &s, const UmmaTiling &t)
{
    if (t.pack != PACK_SUB) return s;
    ConvShape k = s;
    k.H = s.Ho, k.W = s.Wo, k.stride = 1;
    return k;
}

bool sub_ok(const ConvShape &s)
{
    return s.groups == 1 && s.KH == 1 && s.KW == 1 && s.pad == 0 && s.stride > 1;
}

// Rows per image in the stacked layout: at least pad zero rows below each
// image, which serve as the bottom padding of that image and the top padding
// of the next.  When the output rows can take TMA stores, the pitch is rounded
// up to 4 rows so that an epilogue warp's 4 x 8 pixels lie in one image.
int stack_pitch(const ConvShape &s, const UmmaTiling &t)
{
    const int ec = t.split > 1 ? 4 : (int)dtype_size(s.out_dt);
    const int rows = s.H + s.pad;
    return (s.Wo * ec) % 16 == 0 ? (rows + 3) / 4 * 4 : rows;
}

struct Box {
    int w, h, bpt;
    double eff;
};

// Pixel boxes for the NHWC mode, best coverage first.
std::vector<Box> box_options(const ConvShape &s)
{
    std::vector<Box> v;
    for (int w = 1; w <= 128; w *= 2)
        for (int h = 1; w * h <= 128; h *= 2) {
            if ((w * h) % 8) continue;
            const int bpt = 128 / (w * h);
            if (w * s.stride > 256 || h * s.stride > 256) continue;
            const double cover = (double)ceil_div(s.Ho, h) * h * ceil_div(s.Wo, w) * w;
            const double eff = (double)s.Ho * s.Wo / cover;
            v.push_back({w, h, bpt, eff});
        }
    // also boxes that match the image width exactly (w*h multiple of 8, < 128 rows),
    // unless the power-of-two sizes above already hold the same box
    for (int h = 1; h <= 128; ++h) {
        const int w = s.Wo;
        if (w > 128 || w * h > 128 || (w * h) % 8) continue;
        if (w * s.stride > 256 || h * s.stride > 256) continue;
        if (std::any_of(v.begin(), v.end(), [&](const Box &b) { return b.w == w && b.h == h; })) continue;
        const int bpt = 128 / (w * h);
        const double cover = (double)ceil_div(s.Ho, h) * h * w;
        const double eff = (double)s.Ho * s.Wo / cover * (double)(bpt * w * h) / 128.0;
        v.push_back({w, h, bpt, eff});
    }
    std::stable_sort(v.begin(), v.end(), [](const Box &a, const Box &b) {
        if (std::fabs(a.eff - b.eff) > 1e-9) return a.eff > b.eff;
        return a.bpt < b.bpt;
    });
    return v;
}

struct UmmaGeom {
    UmmaParams p;
    int grid;
    int ch, cip;
    bool fits;      // box and unit counts fit the kernel's 32-bit indexing
};

UmmaGeom umma_geometry(const ConvShape &s0, const UmmaTiling &t, int sm_count)
{
    UmmaGeom g{};
    UmmaParams &p = g.p;
    const ConvShape s = kernel_shape(s0, t);
    const int e = (int)dtype_size(s.in_dt);
    p.N = s.N, p.CI = s.CI, p.H = s.H, p.W = s.W, p.CO = s.CO, p.KH = s.KH, p.KW = s.KW;
    p.stride = s.stride, p.pad = s.pad, p.Ho = s.Ho, p.Wo = s.Wo;
    p.bk = 128 / e;
    p.ci_blocks = (int)ceil_div(s.CI, p.bk);
    p.box_w = t.box_w, p.box_h = t.box_h, p.bpt = t.bpt;
    long long bpi;
    if (t.pack == PACK_IM2COL) {
        // 128-pixel tiles of the flattened N x Ho x Wo output, one im2col load per tap
        p.boxes_x = 1, p.boxes_y = 1;
        bpi = ceil_div((long long)s.N * s.Ho * s.Wo, 128);
        p.k_blocks = s.KH * s.KW * p.ci_blocks;
        g.cip = p.ci_blocks * p.bk;
        g.ch = (int)ceil_div(s.CI, 16 / e) * (16 / e);
        p.im2col = 1;
    } else if (t.amode == A_NHWC || t.amode == A_HALO) {
        p.boxes_x = (int)ceil_div(s.Wo, t.box_w);
        p.boxes_y = (int)ceil_div(s.Ho, t.box_h);
        if (t.pack == PACK_STACK) {
            // one tall image of N * hp rows
            p.hp = stack_pitch(s, t);
            p.boxes_y = (int)std::min<long long>(ceil_div((long long)s.N * p.hp, t.box_h), INT32_MAX);
        }
        bpi = (long long)p.boxes_x * p.boxes_y;
        // halo: one K block is a channel block with every tap inside it
        p.k_blocks = (t.amode == A_HALO ? 1 : s.KH * s.KW) * p.ci_blocks;
        g.cip = p.ci_blocks * p.bk;
        g.ch = (int)ceil_div(s.CI, 16 / e) * (16 / e);
    } else if (t.amode == A_STRIDED) {
        // boxes of box_w x box_h output pixels over the [Ho][Wo] output
        p.boxes_x = (int)ceil_div(s.Wo, t.box_w);
        p.boxes_y = (int)ceil_div(s.Ho, t.box_h);
        bpi = (long long)p.boxes_x * p.boxes_y;
        p.k_blocks = p.ci_blocks;
        g.cip = s.CI;
        g.ch = s.CI;
    } else {
        p.boxes_x = 1, p.boxes_y = 1;
        bpi = ceil_div((long long)s.H * s.W, t.box_w);
        p.k_blocks = p.ci_blocks;
        g.cip = s.CI;
        g.ch = s.CI;
    }
    p.cip = g.cip;
    const long long total = (t.pack == PACK_STACK || t.pack == PACK_IM2COL ? 1 : (long long)s.N) * bpi;
    // CTA pairs: a unit is two tiles, one per block of the pair
    const long long ptiles = ceil_div(ceil_div(total, t.bpt), t.pair ? 2 : 1);
    p.co_tiles = (int)ceil_div(s.CO, t.bn);
    p.kb_per_split = (int)ceil_div(p.k_blocks, t.split);
    p.split = (int)ceil_div(p.k_blocks, p.kb_per_split);
    const long long units = ptiles * p.co_tiles * p.split;
    g.fits = total < (1ll << 31) && units < (1ll << 31);
    p.boxes_per_img = (int)std::min<long long>(bpi, INT32_MAX);
    p.total_boxes = (int)std::min<long long>(total, INT32_MAX);
    p.pix_tiles = (int)std::min<long long>(ptiles, INT32_MAX);
    p.units = (int)std::min<long long>(units, INT32_MAX);
    p.epi = s.epi;
    p.out_dt = s.out_dt;
    p.out_elems = (long long)s.N * s.CO * s.Ho * s.Wo;
    DeviceState *ds = device_state();
    const int limit = ds ? ds->max_smem_optin : 232448;
    if (t.amode == A_HALO) {
        // shared-memory layout: streamed or resident weights (a CTA pair's
        // blocks hold half of the weights each)
        g.fits = g.fits && halo_layout(t.pair ? t.bn / 2 : t.bn, t.bres != 0, t.box_h, s.KH,
                                       s.KH * s.KW, p.ci_blocks, limit, p);
    } else if (t.amode == A_STRIDED) {
        g.fits = g.fits && strided_layout(t.bn, limit, p);
    } else if (t.bres) {
        // resident weights of one output-channel tile, every K block
        g.fits = g.fits && main_res_layout(t.bn, p.k_blocks, limit, p);
    }
    g.grid = (int)std::min<long long>(p.units, sm_count);
    if (t.pair) g.grid = (int)std::min<long long>(2 * p.units, sm_count & ~1);
    if (t.bres && t.amode != A_HALO && p.co_tiles > 0) {
        // each block keeps one output-channel tile: a grid of whole tile groups
        g.grid = std::max(p.co_tiles, g.grid / p.co_tiles * p.co_tiles);
    }
    return g;
}

// Host-side validity of a UMMA tiling for a shape; reason on failure.
bool umma_valid(const ConvShape &s0, const UmmaTiling &t, int sm_count, std::string *why)
{
    auto bad = [&](const char *m) {
        if (why) *why = m;
        return false;
    };
    if (t.pack == PACK_SUB) {
        if (t.amode != A_NHWC) return bad("the subsampling pack feeds the nhwc mode");
        if (!sub_ok(s0)) return bad("the subsampling pack needs a strided 1x1 conv without padding");
    } else if (t.pack == PACK_STACK) {
        if (t.amode != A_HALO) return bad("stacked images feed the halo mode");
        if (s0.Ho > s0.H + s0.pad) return bad("stacking needs pad <= KH - 1");
        if ((long long)s0.N * stack_pitch(s0, t) + 16 >= (1ll << 31)) return bad("stacked rows exceed 2^31");
    } else if (t.pack == PACK_IM2COL) {
        if (t.amode != A_NHWC) return bad("im2col loads feed the nhwc mode");
        if (s0.KH * s0.KW < 2) return bad("im2col tiles are for kernels larger than 1x1");
        if (s0.stride > 2) return bad("im2col tiles take stride 1 or 2");
        if (s0.KH > 8 || s0.KW > 8 || s0.pad > 7) return bad("im2col offsets and corners are small");
        if (t.box_w != 128 || t.box_h != 1 || t.bpt != 1) return bad("an im2col tile is 128 pixels");
        if ((long long)s0.N * s0.Ho * s0.Wo >= (1ll << 31)) return bad("more than 2^31 output pixels");
    } else if (t.pack != PACK_PLAIN) {
        return bad("unknown pack layout");
    }
    const ConvShape s = kernel_shape(s0, t);
    const size_t e = dtype_size(s.in_dt);
    if (s.groups != 1) return bad("grouped conv");
    if (t.bn != 64 && t.bn != 128 && t.bn != 256) return bad("tile_n not 64/128/256");
    if (t.split < 1) return bad("split < 1");
    if (t.bpt < 1) return bad("boxes per tile < 1");
    if (t.amode == A_DIRECT) {
        if (s.KH != 1 || s.KW != 1 || s.stride != 1 || s.pad != 0) return bad("direct mode needs 1x1/s1/p0");
        // The direct mode reads data as an MN-major operand; tf32 MMAs take
        // K-major operands only (measured: an MN-major tf32 A reads as zeros).
        if (s.in_dt == BIGEMM_F32) return bad("direct mode needs 16-bit operands");
        if (((long long)s.H * s.W * e) % 16) return bad("H*W row not 16-byte multiple");
        if ((s.CI * e) % 16) return bad("CI row not 16-byte multiple");
        if (t.box_w != (int)(128 / e) || t.box_h != 1 || t.bpt * t.box_w != 128)
            return bad("direct box must be one 128-byte row of pixels");
    } else if (t.amode == A_STRIDED) {
        if (s.KH != 1 || s.KW != 1 || s.stride != 2 || s.pad != 0)
            return bad("strided mode needs 1x1 / stride 2 / pad 0");
        // MN-major operand (tf32 MMAs take K-major operands only)
        if (s.in_dt == BIGEMM_F32) return bad("strided mode needs 16-bit operands");
        // rows of 2W elements (an even input row and the odd one below it) are
        // the TMA rows: 16-byte multiples, and H a whole number of such pairs
        if (s.H % 2 || (2LL * s.W * e) % 16) return bad("strided mode needs even H and 2W*e a 16-byte multiple");
        if ((s.CI * e) % 16) return bad("CI row not 16-byte multiple");
        if (t.box_w != 16 || t.box_h != 4 || t.bpt != 2) return bad("strided boxes are 16 x 4 pixels, two per tile");
        if (t.bres || t.epi16) return bad("strided mode streams its weights with 8 epilogue warps");
        if (!umma_geometry(s0, t, 1).fits) return bad("strided buffers exceed shared memory");
    } else if (t.amode == A_HALO) {
        if (t.bres && s.CO > t.bn) return bad("resident weights need one output-channel tile");
        if (!umma_geometry(s0, t, 1).fits) return bad("halo buffers exceed shared memory");
        if (s.stride != 1) return bad("halo mode needs stride 1");
        if (s.KH * s.KW < 2) return bad("halo mode is for kernels larger than 1x1");
        if (s.KH > 7 || s.KW > 8) return bad("halo mode holds up to 7 rows x 8 columns of taps");
        if (t.box_w != 8 || (t.box_h != 16 && t.box_h != 32) || t.bpt != 1)
            return bad("halo tile is 8 x 16 pixels, or two of them stacked (8 x 32)");
        if (t.box_h == 32 && (t.bn > 128 || t.bres))
            return bad("two-tile halo units need BN <= 128 and streamed weights");
    } else {
        if (s.stride > 8) return bad("stride > 8");
        if (t.box_w < 1 || t.box_h < 1) return bad("empty box");
        if ((t.box_w * t.box_h) % 8) return bad("box pixels not a multiple of 8");
        if (t.box_w * t.box_h * t.bpt > 128) return bad("boxes exceed 128 rows");
        if (t.box_w * s.stride > 256 || t.box_h * s.stride > 256) return bad("box > 256");
    }
    if (t.bres && t.amode != A_HALO && t.split != 1) return bad("resident weights need split 1");
    if (t.pair) {
        if (t.amode != A_HALO || !t.bres || t.box_h != 16)
            return bad("CTA pairs run the halo mode with resident weights and 16-row tiles");
        if (t.bn != 64 && t.bn != 128) return bad("CTA pairs take tile_n 64 or 128");
        if (t.split != 1) return bad("CTA pairs need split 1");
        if (sm_count < 2) return bad("CTA pairs need two SMs");
    }
    if (t.epi16 && (t.amode == A_HALO || t.amode == A_STRIDED || (t.bn != 128 && t.bn != 64)))
        return bad("16 epilogue warps need the nhwc or direct mode and BN = 64 or 128");
    if (t.bpt > 16) return bad("more than 16 boxes per tile");
    if (umma_smem_bytes(t) == 0) return bad("no compiled kernel");
    if (!umma_geometry(s0, t, 1).fits) return bad("more than 2^31 boxes or work units");
    DeviceState *ds = device_state();
    if (ds && !t.bres && t.amode != A_STRIDED && (int)umma_smem_bytes(t) > ds->max_smem_optin)
        return bad("smem exceeds opt-in limit");
    if (t.bres && t.amode != A_HALO && !umma_geometry(s0, t, 1).fits)
        return bad("resident weights exceed shared memory");
    (void)sm_count;
    return true;
}

}  // namespace

}  // namespace bigemm

using namespace bigemm;

struct bigemm_plan_s {
    ConvShape s{};
    int device = 0;
    int sm_count = 0;
    Cand c;
    UmmaGeom g{};
    void *xh = nullptr;
    size_t xh_bytes = 0;
    void *wp = nullptr;
    size_t wp_bytes = 0;
    float *ws = nullptr;
    size_t ws_bytes = 0;
    CUtensorMap map_a{}, map_b{}, map_c{};
    const void *map_a_src = nullptr, *map_b_src = nullptr;   // DIRECT: pointers encoded
    const void *map_c_src = nullptr;                         // output pointer encoded in map_c
    bool store_tma = false;
    bool maps_ready = false;
    bool raw_b = false;        // 1x1 nhwc mode: map_b reads the caller's kernel [CO][CI] as is
    bool red_add = false;      // split K into the zeroed fp32 output by atomic adds (no workspace)
    std::string search_log;
    std::string chosen_by = "heuristic";
};

namespace bigemm {
namespace {

bigemm_status validate(const ConvShape &s)
{
    if (s.N < 1 || s.H < 1 || s.W < 1 || s.CO < 1 || s.CI < 1 || s.KH < 1 || s.KW < 1)
        return BIGEMM_ERR_INVALID_ARG;
    if (s.stride < 1 || s.pad < 0 || s.groups < 1) return BIGEMM_ERR_INVALID_ARG;
    if (s.CI % s.groups || s.CO % s.groups) return BIGEMM_ERR_INVALID_ARG;
    if (s.in_dt < BIGEMM_F32 || s.in_dt > BIGEMM_BF16) return BIGEMM_ERR_INVALID_ARG;
    if (s.out_dt < BIGEMM_F32 || s.out_dt > BIGEMM_BF16) return BIGEMM_ERR_INVALID_ARG;
    if (s.epi < BIGEMM_EPI_NONE || s.epi > BIGEMM_EPI_BIAS_RELU) return BIGEMM_ERR_INVALID_ARG;
    if (s.Ho < 1 || s.Wo < 1) return BIGEMM_ERR_INVALID_ARG;
    if ((long long)s.H * s.W > (1ll << 30) || (long long)s.Ho * s.Wo > (1ll << 30))
        return BIGEMM_ERR_UNSUPPORTED;
    if (s.N > 65535 || s.CO > 65535) return BIGEMM_ERR_UNSUPPORTED;
    return BIGEMM_OK;
}

bool simt_valid(const ConvShape &s, const Cand &c, std::string *why)
{
    if (c.simt_variant == SV_TILED && s.groups != 1) {
        if (why) *why = "tiled SIMT needs groups = 1";
        return false;
    }
    if (c.simt_variant == SV_DWP && !dw_plane_ok(s))
        return why && (*why = "plane depthwise needs a streaming-kernel shape with H, W <= 32", true),
               false;
    if (c.simt_variant == SV_DWR && !dw_small_ok(s, c.dw_rows))
        return why && (*why = "small-plane depthwise needs a square 3/5/7 kernel, pad K/2, stride 1 "
                              "and outputs at most 16 wide, 32 tall",
                       true),
               false;
    if (c.simt_variant == SV_DWB && !dw_band_ok(s))
        return why && (*why = "band depthwise needs a square 3/5/7 kernel, pad K/2, stride 1-2 and "
                              "input rows of 16-byte chunks, at most 512 bytes",
                       true),
               false;
    if (c.simt_variant == SV_DWS && !dw_stream_ok(s))
        return why && (*why = "streaming depthwise needs a square 3/5/7 kernel, pad K/2, stride 1-2",
                       true),
               false;
    if (c.simt_variant == SV_DW) {
        if (!is_depthwise(s)) return why && (*why = "not depthwise", true), false;
        if (s.KH * s.KW > 49) return why && (*why = "depthwise kernel > 7x7", true), false;
        DeviceState *ds = device_state();
        const size_t smem = dw_smem_bytes(s, c.dw_rows);
        if (c.dw_rows < 1 || (ds && smem > (size_t)ds->max_smem_optin))
            return why && (*why = "depthwise band exceeds shared memory", true), false;
    }
    return true;
}

bool cand_valid(const ConvShape &s, const Cand &c, int sms, std::string *why)
{
    if (c.kind == BIGEMM_KIND_UMMA) return umma_valid(s, c.t, sms, why);
    return simt_valid(s, c, why);
}

int heuristic_split(const ConvShape &s, UmmaTiling t, int sms)
{
    t.split = 1;
    const UmmaGeom g = umma_geometry(s, t, sms);
    const long long tiles = (long long)g.p.pix_tiles * g.p.co_tiles;
    if (tiles * 2 >= sms || g.p.k_blocks < 4) return 1;
    long long want = (sms + tiles - 1) / tiles;
    want = std::min<long long>(want, g.p.k_blocks / 2);
    return (int)std::max<long long>(1, want);
}

UmmaTiling default_tiling(const ConvShape &s, int amode, int bn, int sms, int pack = PACK_PLAIN)
{
    UmmaTiling t{};
    t.amode = amode;
    t.pack = pack;
    t.bn = bn;
    t.stages = 0;
    if (amode == A_DIRECT) {
        t.box_w = (int)(128 / dtype_size(s.in_dt));
        t.box_h = 1;
        t.bpt = 128 / t.box_w;
    } else if (amode == A_HALO) {
        t.box_w = 8, t.box_h = 16, t.bpt = 1;
    } else if (amode == A_STRIDED) {
        t.box_w = 16, t.box_h = 4, t.bpt = 2;
    } else if (pack == PACK_IM2COL) {
        t.box_w = 128, t.box_h = 1, t.bpt = 1;
    } else {
        const Box b = box_options(kernel_shape(s, t)).front();
        t.box_w = b.w, t.box_h = b.h, t.bpt = b.bpt;
    }
    t.split = 1;
    t.split = heuristic_split(s, t, sms);
    return t;
}

int default_bn(const ConvShape &s)
{
    if (s.CO <= 64) return 64;
    if (s.CO <= 128) return 128;
    return (s.CO % 256 == 0) ? 256 : 128;
}

// Fraction of the halo tiles' 16 x 8 output pixels that lie inside the
// output, per image or with the images stacked; 0 when the layout does not
// apply.
double halo_cover(const ConvShape &s, int pack)
{
    UmmaTiling t{};
    t.amode = A_HALO;
    t.pack = pack;
    t.bn = 64;
    t.box_w = 8, t.box_h = 16, t.bpt = 1;
    t.split = 1;
    if (!umma_valid(s, t, 1, nullptr)) return 0.0;
    const double rows = pack == PACK_STACK ? (double)ceil_div((long long)s.N * stack_pitch(s, t), 16) * 16
                                           : (double)s.N * ceil_div(s.Ho, 16) * 16;
    return (double)s.N * s.Ho * s.Wo / (rows * ceil_div(s.Wo, 8) * 8);
}

// Keep the weights resident when one output-channel tile covers CO and they fit.
void prefer_resident(const ConvShape &s, UmmaTiling &t)
{
    if (t.amode != A_HALO || s.CO > t.bn) return;
    UmmaTiling r = t;
    r.bres = 1;
    if (umma_valid(s, r, 1, nullptr)) t.bres = 1;
}

// Sixteen epilogue warps for 128-channel tiles over whole K ranges: the
// epilogue, not the MMA, paces such tiles (measured on the 1x1 64->256 layer
// at 56x56, N = 256: 110 -> 90 us).
void prefer_epi16(const ConvShape &s, UmmaTiling &t)
{
    if (t.amode == A_HALO || t.bn != 128 || t.split != 1) return;
    UmmaTiling r = t;
    r.epi16 = 1;
    if (umma_valid(s, r, 1, nullptr)) t.epi16 = 1;
}

// Halo tiles are worth it when they are mostly inside the output.
bool halo_ok(const ConvShape &s)
{
    return std::max(halo_cover(s, PACK_PLAIN), halo_cover(s, PACK_STACK)) >= 0.7;
}

// The halo layout for a shape: stacked images when they cover clearly more of
// the tiles, else the plain packed copy.
int halo_pack(const ConvShape &s)
{
    const double cp = halo_cover(s, PACK_PLAIN), cs = halo_cover(s, PACK_STACK);
    return cs > cp + 0.02 ? PACK_STACK : PACK_PLAIN;
}

bool strided_ok(const ConvShape &s)
{
    UmmaTiling t{};
    t.amode = A_STRIDED;
    t.bn = 64;
    t.box_w = 16, t.box_h = 4, t.bpt = 2;
    t.split = 1;
    return umma_valid(s, t, 1, nullptr);
}

bool direct_ok(const ConvShape &s)
{
    UmmaTiling t{};
    t.amode = A_DIRECT;
    t.bn = 64;
    t.box_w = (int)(128 / dtype_size(s.in_dt));
    t.box_h = 1;
    t.bpt = 128 / t.box_w;
    t.split = 1;
    return umma_valid(s, t, 1, nullptr);
}

Cand heuristic(const ConvShape &s, int sms)
{
    Cand c;
    // small planes: whole planes per warp (4-row blocks above 8 rows)
    for (int ty : {s.Ho > 8 ? 4 : 2, 2})
        if (dw_small_ok(s, ty)) {
            c.simt_variant = SV_DWR;
            c.dw_rows = ty;
            return c;
        }
    if (dw_stream_ok(s)) {
        c.simt_variant = SV_DWS;
        c.dw_rows = 2;
        return c;
    }
    if (is_depthwise(s) && s.KH * s.KW <= 49) {
        c.simt_variant = SV_DW;
        c.dw_rows = std::max(1, std::min(s.Ho, 2048 / std::max(1, s.Wo)));
        while (c.dw_rows > 1 && !simt_valid(s, c, nullptr)) c.dw_rows /= 2;
        return c;
    }
    if (s.groups != 1) return c;   // naive
    const long long kdim = (long long)s.CI * s.KH * s.KW;
    if (kdim >= 32) {
        Cand u;
        u.kind = BIGEMM_KIND_UMMA;
        if (direct_ok(s))
            u.t = default_tiling(s, A_DIRECT, default_bn(s), sms);
        else if (strided_ok(s))
            u.t = default_tiling(s, A_STRIDED, default_bn(s), sms);
        else if (sub_ok(s))
            u.t = default_tiling(s, A_NHWC, default_bn(s), sms, PACK_SUB);
        else if (halo_ok(s)) {
            u.t = default_tiling(s, A_HALO, default_bn(s), sms, halo_pack(s));
            prefer_resident(s, u.t);
        } else
            u.t = default_tiling(s, A_NHWC, default_bn(s), sms);
        prefer_epi16(s, u.t);
        if (umma_valid(s, u.t, sms, nullptr)) return u;
    }
    c.simt_variant = SV_TILED;
    return c;
}

std::vector<Cand> candidates(const ConvShape &s, int sms)
{
    std::vector<Cand> v;
    if (is_depthwise(s)) {
        for (int ty : {4, 2})
            if (dw_small_ok(s, ty)) {
                Cand c;
                c.simt_variant = SV_DWR;
                c.dw_rows = ty;
                v.push_back(c);
            }
        if (dw_band_ok(s)) {
            Cand c;
            c.simt_variant = SV_DWB;
            v.push_back(c);
        }
        if (dw_plane_ok(s)) {
            Cand c;
            c.simt_variant = SV_DWP;
            v.push_back(c);
        }
        if (dw_stream_ok(s))
            for (int rows : {2, 4, 8}) {
                if (rows == 8 && !(s.stride == 1 && s.KH <= 5)) continue;
                Cand c;
                c.simt_variant = SV_DWS;
                c.dw_rows = rows;
                v.push_back(c);
            }
        for (int rows : {1, 2, 4, 8, 16, 32}) {
            Cand c;
            c.simt_variant = SV_DW;
            c.dw_rows = rows;
            if (rows <= s.Ho && simt_valid(s, c, nullptr)) v.push_back(c);
        }
        if (v.empty()) v.push_back(Cand{});
        return v;
    }
    if (s.groups != 1) {
        v.push_back(Cand{});
        return v;
    }
    std::vector<std::pair<int, int>> modes;   // (A mode, pack layout)
    if (direct_ok(s)) modes.push_back({A_DIRECT, PACK_PLAIN});
    const double hc_plain = halo_cover(s, PACK_PLAIN), hc_stack = halo_cover(s, PACK_STACK);
    if (hc_plain >= 0.7) modes.push_back({A_HALO, PACK_PLAIN});
    if (hc_stack >= 0.7 && hc_stack > hc_plain + 0.02) modes.push_back({A_HALO, PACK_STACK});
    if (strided_ok(s)) modes.push_back({A_STRIDED, PACK_PLAIN});
    if (sub_ok(s)) modes.push_back({A_NHWC, PACK_SUB});
    modes.push_back({A_NHWC, PACK_PLAIN});
    if (s.KH * s.KW > 1 && s.stride <= 2) modes.push_back({A_NHWC, PACK_IM2COL});
    for (const auto &mp : modes) {
        const int amode = mp.first, pack = mp.second;
        UmmaTiling probe{};
        probe.pack = pack;
        const std::vector<Box> boxes = box_options(kernel_shape(s, probe));
        std::vector<std::pair<int, int>> bx;   // (w,h) with bpt
        std::vector<int> bpts;
        if (amode == A_DIRECT) {
            const int w = (int)(128 / dtype_size(s.in_dt));
            bx.push_back({w, 1});
            bpts.push_back(128 / w);
        } else if (amode == A_HALO) {
            bx.push_back({8, 16});
            bpts.push_back(1);
            bx.push_back({8, 32});   // two tiles sharing each weight tile
            bpts.push_back(1);
        } else if (amode == A_STRIDED) {
            bx.push_back({16, 4});
            bpts.push_back(2);
        } else if (pack == PACK_IM2COL) {
            bx.push_back({128, 1});
            bpts.push_back(1);
        } else {
            for (size_t i = 0; i < boxes.size() && bx.size() < 2; ++i) {
                if (i > 0 && boxes[i].eff < boxes[0].eff - 0.05) break;
                bx.push_back({boxes[i].w, boxes[i].h});
                bpts.push_back(boxes[i].bpt);
            }
            // Output rows that TMA cannot store are written by the lanes
            // directly; boxes spanning whole output rows keep a warp's 32
            // pixels contiguous in each channel plane.
            const ConvShape ks = kernel_shape(s, probe);
            if ((ks.Wo * (long long)dtype_size(s.out_dt)) % 16 != 0) {
                for (const Box &b : boxes)
                    if (b.w == ks.Wo &&
                        std::find(bx.begin(), bx.end(), std::make_pair(b.w, b.h)) == bx.end()) {
                        bx.push_back({b.w, b.h});
                        bpts.push_back(b.bpt);
                        break;
                    }
            }
        }
        for (size_t bi = 0; bi < bx.size(); ++bi)
            for (int bn : {64, 128, 256}) {
                if (bn > 64 && bn / 2 >= s.CO) continue;   // a smaller tile covers CO
                UmmaTiling t{};
                t.amode = amode, t.pack = pack, t.bn = bn, t.box_w = bx[bi].first,
                t.box_h = bx[bi].second;
                t.bpt = bpts[bi];
                t.split = 1;
                const UmmaGeom g = umma_geometry(s, t, sms);
                const long long tiles = (long long)g.p.pix_tiles * g.p.co_tiles;
                for (int split : {1, 2, 4, 8, 16, 32}) {
                    if (split > 1 && (tiles * split > 4LL * sms || g.p.k_blocks / split < 2)) continue;
                    t.split = split;
                    Cand c;
                    c.kind = BIGEMM_KIND_UMMA;
                    c.t = t;
                    if (umma_valid(s, t, sms, nullptr)) v.push_back(c);
                    if ((amode == A_HALO && s.CO <= bn) || (amode != A_HALO && split == 1)) {
                        c.t.bres = 1;   // the resident-weights form too
                        if (umma_valid(s, c.t, sms, nullptr)) v.push_back(c);
                        if (amode == A_HALO && split == 1) {
                            Cand pc = c;   // and its CTA-pair form
                            pc.t.pair = 1;
                            if (umma_valid(s, pc.t, sms, nullptr)) v.push_back(pc);
                        }
                    }
                    if (amode != A_HALO && amode != A_STRIDED && (bn == 128 || bn == 64)) {
                        // both forms again with 16 epilogue warps
                        for (int br : {0, 1}) {
                            if (br && split != 1) continue;
                            Cand e = c;
                            e.t.bres = br, e.t.epi16 = 1;
                            if (umma_valid(s, e.t, sms, nullptr)) v.push_back(e);
                        }
                    }
                }
            }
    }
    Cand tiled;
    tiled.simt_variant = SV_TILED;
    v.push_back(tiled);
    return v;
}

// ------------------------------------------------------------ scratch + run
// Output tiles can be written by TMA stores when the output's (or the split-K
// workspace's) innermost extent and every box start are 16-byte aligned.
bool store_tma_ok(const ConvShape &s, const UmmaTiling &t, int split)
{
    const long long ec = split > 1 ? 4 : (long long)dtype_size(s.out_dt);
    // im2col tiles run across rows and images: stores from registers
    if (t.pack == PACK_IM2COL) return false;
    if ((t.box_w * ec) % 16) return false;
    // each epilogue warp stores its 32 pixels as one box: 32 of a row, or whole rows
    const bool wide = t.box_w % 32 == 0;
    if (!wide && !(32 % t.box_w == 0 && (t.box_w * t.box_h) % 32 == 0)) return false;
    if (t.amode == A_DIRECT) return ((long long)s.Ho * s.Wo * ec) % 16 == 0;
    // stacked images: a warp's rows (32 / box_w of them) must not straddle two images
    if (t.pack == PACK_STACK && (wide || stack_pitch(s, t) % (32 / t.box_w))) return false;
    return ((long long)s.Wo * ec) % 16 == 0;
}

bool encode_store_map(bigemm_plan_s *p, void *dst, bool is_ws)
{
    const ConvShape &s = p->s;
    const UmmaTiling &t = p->c.t;
    const int split = p->g.p.split;
    const uint64_t ec = is_ws ? 4 : dtype_size(s.out_dt);
    const CUtensorMapDataType dt = is_ws ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : tma_dt(s.out_dt);
    const uint64_t nn = (uint64_t)s.N * (is_ws ? split : 1);
    if (t.amode == A_DIRECT) {
        const uint64_t hw = (uint64_t)s.Ho * s.Wo;
        const uint64_t dims[3] = {hw, (uint64_t)s.CO, nn};
        const uint64_t str[2] = {hw * ec, hw * s.CO * ec};
        // 2 KB boxes: 32 channels of 16-bit output, 16 of fp32
        const uint32_t box[3] = {32u, ec == 4 ? 16u : 32u, 1u};
        const uint32_t es[3] = {1u, 1u, 1u};
        return encode_tiled(&p->map_c, dt, 3, dst, dims, str, box, es, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    const uint64_t dims[4] = {(uint64_t)s.Wo, (uint64_t)s.Ho, (uint64_t)s.CO, nn};
    const uint64_t str[3] = {(uint64_t)s.Wo * ec, (uint64_t)s.Ho * s.Wo * ec,
                             (uint64_t)s.CO * s.Ho * s.Wo * ec};
    const uint32_t sw = t.box_w >= 32 ? 32u : (uint32_t)t.box_w;
    // 2 KB boxes: 32 channels of 16-bit output, 16 of fp32
    const uint32_t co_box = ec == 4 ? 16u : 32u;
    const uint32_t box[4] = {sw, 32u / sw, co_box, 1u};
    const uint32_t es[4] = {1u, 1u, 1u, 1u};
    return encode_tiled(&p->map_c, dt, 4, dst, dims, str, box, es, CU_TENSOR_MAP_SWIZZLE_NONE);
}

void free_scratch(bigemm_plan_s *p)
{
    if (p->xh) cudaFree(p->xh);
    if (p->wp) cudaFree(p->wp);
    if (p->ws) cudaFree(p->ws);
    p->xh = p->wp = nullptr;
    p->ws = nullptr;
    p->xh_bytes = p->wp_bytes = p->ws_bytes = 0;
    p->maps_ready = false;
}

bigemm_status setup_plan(bigemm_plan_s *p)
{
    const ConvShape &s = p->s;
    if (p->c.kind != BIGEMM_KIND_UMMA) return BIGEMM_OK;
    const UmmaTiling &t = p->c.t;
    p->g = umma_geometry(s, t, p->sm_count);
    const size_t e = dtype_size(s.in_dt);
    if (t.amode == A_HALO) {
        // channels-last data read as one halo box per channel block: 16 pixels
        // wide (the 2 KB smem row pitch), 16 + KH - 1 rows high.  Stacked: one
        // image of N * (H + pad) rows.
        const bool stack = t.pack == PACK_STACK;
        const uint64_t rows = stack ? (uint64_t)s.N * p->g.p.hp : (uint64_t)s.H;
        const uint64_t imgs = stack ? 1u : (uint64_t)s.N;
        p->xh_bytes = (size_t)(imgs * rows) * s.W * p->g.ch * e;
        p->wp_bytes = (size_t)s.CO * s.KH * s.KW * p->g.cip * e;
        if (cudaMalloc(&p->xh, p->xh_bytes) != cudaSuccess) return BIGEMM_ERR_CUDA;
        if (cudaMalloc(&p->wp, p->wp_bytes) != cudaSuccess) return BIGEMM_ERR_CUDA;
        const uint64_t dims[4] = {(uint64_t)p->g.ch, (uint64_t)s.W, rows, imgs};
        const uint64_t str[3] = {p->g.ch * e, (uint64_t)s.W * p->g.ch * e,
                                 rows * s.W * p->g.ch * e};
        const uint32_t box[4] = {(uint32_t)p->g.p.bk, 16u, (uint32_t)(t.box_h + s.KH - 1), 1u};
        const uint32_t es[4] = {1u, 1u, 1u, 1u};
        if (!encode_tiled(&p->map_a, tma_dt(s.in_dt), 4, p->xh, dims, str, box, es,
                          CU_TENSOR_MAP_SWIZZLE_128B))
            return BIGEMM_ERR_UNSUPPORTED;
        // packed weights [CO][tap][cip] viewed as (channel, output channel, tap):
        // one box brings TB taps, each a [BN][128 B] K-major tile
        // (CTA pairs: each block loads half of the tile's output channels)
        const int tb = (t.bres || t.box_h == 32) ? 1 : 32768 / (t.bn * 128);
        const uint64_t kk = (uint64_t)s.KH * s.KW;
        const uint64_t bd[3] = {(uint64_t)p->g.cip, (uint64_t)s.CO, kk};
        const uint64_t bs[2] = {kk * p->g.cip * e, (uint64_t)p->g.cip * e};
        const uint32_t bb[3] = {(uint32_t)p->g.p.bk, (uint32_t)(t.pair ? t.bn / 2 : t.bn),
                                (uint32_t)tb};
        const uint32_t bes[3] = {1u, 1u, 1u};
        if (!encode_tiled(&p->map_b, tma_dt(s.in_dt), 3, p->wp, bd, bs, bb, bes,
                          CU_TENSOR_MAP_SWIZZLE_128B))
            return BIGEMM_ERR_UNSUPPORTED;
        p->maps_ready = true;
    } else if (t.amode == A_NHWC) {
        // the subsampling pack hands the kernel a stride-1 1x1 conv over [Ho][Wo]
        const ConvShape k = kernel_shape(s, t);
        // a 1x1 kernel [CO][CI] is already the K-major B operand
        p->raw_b = k.KH * k.KW == 1 && (k.CI * e) % 16 == 0;
        p->xh_bytes = (size_t)k.N * k.H * k.W * p->g.ch * e;
        p->wp_bytes = p->raw_b ? 0 : (size_t)k.CO * k.KH * k.KW * p->g.cip * e;
        if (cudaMalloc(&p->xh, p->xh_bytes) != cudaSuccess) return BIGEMM_ERR_CUDA;
        if (!p->raw_b && cudaMalloc(&p->wp, p->wp_bytes) != cudaSuccess) return BIGEMM_ERR_CUDA;
        const uint64_t dims[4] = {(uint64_t)p->g.ch, (uint64_t)k.W, (uint64_t)k.H, (uint64_t)k.N};
        const uint64_t str[3] = {p->g.ch * e, (uint64_t)k.W * p->g.ch * e,
                                 (uint64_t)k.H * k.W * p->g.ch * e};
        const uint32_t box[4] = {(uint32_t)p->g.p.bk, (uint32_t)(t.box_w * k.stride),
                                 (uint32_t)(t.box_h * k.stride), 1u};
        const uint32_t es[4] = {1u, (uint32_t)k.stride, (uint32_t)k.stride, 1u};
        if (t.pack == PACK_IM2COL) {
            // window base positions x * stride - pad for the Wo (Ho) outputs: from
            // -pad to W - 1 + (pad - (KW - 1)), in steps of the stride
            const int lower[2] = {-k.pad, -k.pad};
            const int upper[2] = {k.pad - (k.KW - 1), k.pad - (k.KH - 1)};
            if (!encode_im2col(&p->map_a, tma_dt(s.in_dt), p->xh, dims, str, lower, upper,
                               (uint32_t)p->g.p.bk, 128u, es, CU_TENSOR_MAP_SWIZZLE_128B))
                return BIGEMM_ERR_UNSUPPORTED;
        } else if (!encode_tiled(&p->map_a, tma_dt(s.in_dt), 4, p->xh, dims, str, box, es,
                                 CU_TENSOR_MAP_SWIZZLE_128B)) {
            return BIGEMM_ERR_UNSUPPORTED;
        }
        if (!p->raw_b) {
            const uint64_t kt = (uint64_t)k.KH * k.KW * p->g.cip;
            const uint64_t bd[2] = {kt, (uint64_t)k.CO};
            const uint64_t bs[1] = {kt * e};
            const uint32_t bb[2] = {(uint32_t)p->g.p.bk, (uint32_t)t.bn};
            const uint32_t bes[2] = {1u, 1u};
            if (!encode_tiled(&p->map_b, tma_dt(s.in_dt), 2, p->wp, bd, bs, bb, bes,
                              CU_TENSOR_MAP_SWIZZLE_128B))
                return BIGEMM_ERR_UNSUPPORTED;
        }
        p->maps_ready = true;
    }
    // fp32 outputs whose epilogue is linear take the K slices' partial tiles as
    // atomic adds (TMA reduce-add) into the output, zeroed first; the others go
    // through a workspace and a reduction pass
    p->red_add = p->g.p.split > 1 && s.out_dt == BIGEMM_F32 &&
                 (s.epi == BIGEMM_EPI_NONE || s.epi == BIGEMM_EPI_BIAS);
    if (p->g.p.split > 1 && !p->red_add) {
        p->ws_bytes = (size_t)p->g.p.split * p->g.p.out_elems * sizeof(float);
        if (cudaMalloc(&p->ws, p->ws_bytes) != cudaSuccess) return BIGEMM_ERR_CUDA;
    }
    p->store_tma = store_tma_ok(s, t, p->g.p.split) && !getenv("BIGEMM_NO_TMA_STORE");
    if (p->store_tma && p->g.p.split > 1 && !p->red_add) {
        if (!encode_store_map(p, p->ws, true)) p->store_tma = false;
        p->map_c_src = p->ws;
    }
    return BIGEMM_OK;
}

bigemm_status encode_direct_maps(bigemm_plan_s *p, const void *data, const void *kernel)
{
    if (p->maps_ready && p->map_a_src == data && p->map_b_src == kernel) return BIGEMM_OK;
    const ConvShape &s = p->s;
    const UmmaTiling &t = p->c.t;
    const size_t e = dtype_size(s.in_dt);
    const uint64_t hw = (uint64_t)s.H * s.W;
    const uint64_t dims[3] = {hw, (uint64_t)s.CI, (uint64_t)s.N};
    const uint64_t str[2] = {hw * e, hw * s.CI * e};
    const uint32_t box[3] = {(uint32_t)t.box_w, (uint32_t)p->g.p.bk, 1u};
    const uint32_t es[3] = {1u, 1u, 1u};
    if (!encode_tiled(&p->map_a, tma_dt(s.in_dt), 3, data, dims, str, box, es,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return BIGEMM_ERR_INVALID_ARG;
    const uint64_t bd[2] = {(uint64_t)s.CI, (uint64_t)s.CO};
    const uint64_t bs[1] = {(uint64_t)s.CI * e};
    const uint32_t bb[2] = {(uint32_t)p->g.p.bk, (uint32_t)t.bn};
    const uint32_t bes[2] = {1u, 1u};
    if (!encode_tiled(&p->map_b, tma_dt(s.in_dt), 2, kernel, bd, bs, bb, bes,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return BIGEMM_ERR_INVALID_ARG;
    p->map_a_src = data;
    p->map_b_src = kernel;
    p->maps_ready = true;
    return BIGEMM_OK;
}

// The strided mode's maps, re-encoded when a pointer changes: the data as
// rows of 2W elements (an even input row and the odd one below it) x H/2 row
// pairs x CI x N, read by 32-element x 4-row x 64-channel staging boxes
// without swizzle; the kernel [CO][CI] as the K-major B operand.
bigemm_status encode_strided_maps(bigemm_plan_s *p, const void *data, const void *kernel)
{
    if (p->maps_ready && p->map_a_src == data && p->map_b_src == kernel) return BIGEMM_OK;
    const ConvShape &s = p->s;
    const UmmaTiling &t = p->c.t;
    const size_t e = dtype_size(s.in_dt);
    const uint64_t dims[4] = {2ull * s.W, (uint64_t)s.H / 2, (uint64_t)s.CI, (uint64_t)s.N};
    const uint64_t str[3] = {2ull * s.W * e, (uint64_t)s.H * s.W * e, (uint64_t)s.CI * s.H * s.W * e};
    const uint32_t box[4] = {2u * (uint32_t)t.box_w, (uint32_t)t.box_h, (uint32_t)p->g.p.bk, 1u};
    const uint32_t es[4] = {1u, 1u, 1u, 1u};
    if (!encode_tiled(&p->map_a, tma_dt(s.in_dt), 4, data, dims, str, box, es,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
        return BIGEMM_ERR_INVALID_ARG;
    const uint64_t bd[2] = {(uint64_t)s.CI, (uint64_t)s.CO};
    const uint64_t bs[1] = {(uint64_t)s.CI * e};
    const uint32_t bb[2] = {(uint32_t)p->g.p.bk, (uint32_t)t.bn};
    const uint32_t bes[2] = {1u, 1u};
    if (!encode_tiled(&p->map_b, tma_dt(s.in_dt), 2, kernel, bd, bs, bb, bes,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return BIGEMM_ERR_INVALID_ARG;
    p->map_a_src = data;
    p->map_b_src = kernel;
    p->maps_ready = true;
    return BIGEMM_OK;
}

// The raw-kernel B map of a 1x1 nhwc plan, re-encoded when the kernel pointer
// changes: [CO][CI] with channel blocks past CI zero-filled by the copy.
bigemm_status encode_raw_b(bigemm_plan_s *p, const void *kernel)
{
    if (p->map_b_src == kernel) return BIGEMM_OK;
    const ConvShape &s = p->s;
    const size_t e = dtype_size(s.in_dt);
    const uint64_t bd[2] = {(uint64_t)s.CI, (uint64_t)s.CO};
    const uint64_t bs[1] = {(uint64_t)s.CI * e};
    const uint32_t bb[2] = {(uint32_t)p->g.p.bk, (uint32_t)p->c.t.bn};
    const uint32_t bes[2] = {1u, 1u};
    if (!encode_tiled(&p->map_b, tma_dt(s.in_dt), 2, kernel, bd, bs, bb, bes,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return BIGEMM_ERR_INVALID_ARG;
    p->map_b_src = kernel;
    return BIGEMM_OK;
}

int launches_per_run(const bigemm_plan_s *p)
{
    if (p->c.kind != BIGEMM_KIND_UMMA) return 1;
    int n = 1;
    if (p->c.t.amode != A_DIRECT && p->c.t.amode != A_STRIDED) n += 1;   // the pack
    if (p->g.p.split > 1 && !p->red_add) n += 1;
    return n;
}

bigemm_status run_plan(bigemm_plan_s *p, const void *data, const void *kernel, const float *bias,
                       float eps, void *out, cudaStream_t st)
{
    const ConvShape &s = p->s;
    if (!data || !kernel || !out) return BIGEMM_ERR_INVALID_ARG;
    if (!aligned16(data) || !aligned16(kernel) || !aligned16(out)) return BIGEMM_ERR_INVALID_ARG;
    if (s.epi != BIGEMM_EPI_NONE && !bias) return BIGEMM_ERR_INVALID_ARG;
    DeviceState *ds = device_state();
    if (!ds) return BIGEMM_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (p->c.kind != BIGEMM_KIND_UMMA) {
        if (p->c.simt_variant == SV_DWR)
            e = launch_dw_small(s, data, kernel, bias, eps, out, p->c.dw_rows, st);
        else if (p->c.simt_variant == SV_DWB)
            e = launch_dw_band(s, data, kernel, bias, eps, out, st);
        else if (p->c.simt_variant == SV_DWP)
            e = launch_dw_plane(s, data, kernel, bias, eps, out, st);
        else if (p->c.simt_variant == SV_DWS)
            e = launch_dw_stream(s, data, kernel, bias, eps, out, p->c.dw_rows, st);
        else if (p->c.simt_variant == SV_DW)
            e = launch_dw_conv(s, data, kernel, bias, eps, out, p->c.dw_rows, st);
        else
            e = launch_simt_conv(s, data, kernel, bias, eps, out, p->c.simt_variant, st);
        return e == cudaSuccess ? BIGEMM_OK : BIGEMM_ERR_CUDA;
    }
    UmmaParams up = p->g.p;
    up.eps = eps;
    up.bias = bias;
    up.out = out;
    up.ws = p->red_add ? nullptr : p->ws;
    up.red_add = p->red_add ? 1 : 0;
    up.err = ds->err;
    up.timeout_ns = wait_timeout_ns();
    if (p->c.t.amode != A_DIRECT && p->c.t.amode != A_STRIDED) {
        const int pk = p->c.t.pack;
        const int hop = pk == PACK_SUB ? s.Ho : pk == PACK_STACK ? up.hp : s.H;
        const int wop = pk == PACK_SUB ? s.Wo : s.W;
        if (p->raw_b) {
            bigemm_status r = encode_raw_b(p, kernel);
            if (r != BIGEMM_OK) return r;
        }
        e = launch_pack_operands(data, p->xh, s.N, s.CI, s.H, s.W, hop, wop,
                                 pk == PACK_SUB ? s.stride : 1, p->g.ch, p->raw_b ? nullptr : kernel,
                                 p->wp, s.CO, s.CI, s.KH * s.KW, p->g.cip, s.in_dt, st,
                                 p->red_add ? static_cast<float *>(out) : nullptr, up.out_elems);
        if (e != cudaSuccess) return BIGEMM_ERR_CUDA;
    } else {
        bigemm_status r = p->c.t.amode == A_STRIDED ? encode_strided_maps(p, data, kernel)
                                                    : encode_direct_maps(p, data, kernel);
        if (r != BIGEMM_OK) return r;
        if (p->red_add &&
            cudaMemsetAsync(out, 0, (size_t)up.out_elems * sizeof(float), st) != cudaSuccess)
            return BIGEMM_ERR_CUDA;
    }
    up.store_tma = 0;
    if (p->store_tma) {
        if ((up.split == 1 || p->red_add) && p->map_c_src != out) {
            if (encode_store_map(p, out, false))
                p->map_c_src = out;
            else
                p->map_c_src = nullptr;
        }
        up.store_tma = p->map_c_src != nullptr ? 1 : 0;
    }
    e = launch_umma_conv(p->c.t, s.in_dt, up, p->map_a, p->map_b, p->map_c, p->g.grid, st);
    if (e != cudaSuccess) return BIGEMM_ERR_CUDA;
    if (up.split > 1 && !p->red_add) {
        e = launch_splitk_reduce(p->ws, up.split, up.out_elems, s.CO, s.Ho * s.Wo, s.epi, bias, eps,
                                 out, s.out_dt, st);
        if (e != cudaSuccess) return BIGEMM_ERR_CUDA;
    }
    return BIGEMM_OK;
}

bigemm_status make_plan(const ConvShape &s, const Cand &c, int sms, bigemm_plan_s **out)
{
    bigemm_plan_s *p = new bigemm_plan_s;
    p->s = s;
    cudaGetDevice(&p->device);
    p->sm_count = sms;
    p->c = c;
    bigemm_status r = setup_plan(p);
    if (r != BIGEMM_OK) {
        free_scratch(p);
        delete p;
        return r;
    }
    *out = p;
    return BIGEMM_OK;
}

// ------------------------------------------------------------- plan cache
std::mutex g_cache_mu;
std::map<std::string, std::pair<std::string, double>> g_cache;   // key -> (cand, ms)
bool g_cache_loaded = false;

std::string cache_key(const ConvShape &s)
{
    char name[256] = "gpu";
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess) snprintf(name, sizeof name, "%s", prop.name);
    char b[512];
    snprintf(b, sizeof b, "%s|N%d|H%d|W%d|CO%d|CI%d|K%dx%d|s%d|p%d|g%d|in%d|out%d|epi%d", name, s.N,
             s.H, s.W, s.CO, s.CI, s.KH, s.KW, s.stride, s.pad, s.groups, s.in_dt, s.out_dt, s.epi);
    return b;
}

void load_cache_file()
{
    if (g_cache_loaded) return;
    g_cache_loaded = true;
    const char *path = getenv("BIGEMM_PLAN_CACHE");
    if (!path || !*path) return;
    std::ifstream f(path);
    std::string line;
    while (std::getline(f, line)) {
        // {"key": "...", "cand": "...", "ms": x}
        auto get = [&](const char *k) -> std::string {
            std::string pat = std::string("\"") + k + "\": \"";
            size_t a = line.find(pat);
            if (a == std::string::npos) return "";
            a += pat.size();
            size_t b = line.find('"', a);
            return b == std::string::npos ? "" : line.substr(a, b - a);
        };
        std::string key = get("key"), cand = get("cand");
        double ms = 0;
        size_t m = line.find("\"ms\": ");
        if (m != std::string::npos) ms = atof(line.c_str() + m + 6);
        Cand c;
        if (!key.empty() && parse_cand(cand, c)) g_cache[key] = {cand, ms};
    }
}

void append_cache_file(const std::string &key, const std::string &cand, double ms)
{
    const char *path = getenv("BIGEMM_PLAN_CACHE");
    if (!path || !*path) return;
    std::ofstream f(path, std::ios::app);
    f << "{\"key\": \"" << key << "\", \"cand\": \"" << cand << "\", \"ms\": " << ms << "}\n";
}

// ------------------------------------------------------------ timed search
struct SearchBuffers {
    void *x = nullptr, *w = nullptr, *o = nullptr;
    float *b = nullptr;
    void *flush = nullptr;          // L2 flush buffer (null: the tensors exceed L2)
    size_t flush_bytes = 0;
    ~SearchBuffers()
    {
        if (x) cudaFree(x);
        if (w) cudaFree(w);
        if (o) cudaFree(o);
        if (b) cudaFree(b);
        if (flush) cudaFree(flush);
    }
};

// Search inputs: element i is a counter-based hash of (i, seed) -- the
// splitmix64 output function (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators", 2014) -- mapped to [-amp, amp] and stored
// in the operand type.  Non-zero operands keep the tensor cores' power draw
// (and so their clocks) as in real use; zeros would flatter every candidate.
__global__ void search_fill(void *p, long long n, int dt, float amp, unsigned long long seed)
{
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        unsigned long long z = (unsigned long long)i + (seed + 1) * 0x9E3779B97F4A7C15ull;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z ^= z >> 31;
        const float v = ((float)(z >> 40) * (2.0f / 16777216.0f) - 1.0f) * amp;
        if (dt == BIGEMM_F32)
            static_cast<float *>(p)[i] = v;
        else if (dt == BIGEMM_F16)
            static_cast<__half *>(p)[i] = __float2half_rn(v);
        else
            static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    }
}

cudaError_t fill_search_input(void *p, long long n, int dt, float amp, unsigned long long seed,
                              int sms, cudaStream_t st)
{
    const int grid = (int)std::max(1ll, std::min(ceil_div(n, 256), (long long)sms * 8));
    search_fill<<<grid, 256, 0, st>>>(p, n, dt, amp, seed);
    return cudaGetLastError();
}

double min_repeat_ms()
{
    const char *v = getenv("BIGEMM_MIN_REPEAT_MS");
    double ms = v ? atof(v) : 2.0;
    return ms > 0 ? ms : 2.0;
}

// Time one candidate: three repeats, each of `number` runs lasting at least
// min_repeat_ms; cost = median of the repeat means.  Without an L2 flush the
// runs of a repeat go back to back between two events; with one, every run
// is timed on its own between events, after a flush that lies outside them.
// status as in the tutorial's measure records: 0 ok, 1 invalid (host check),
// 4 run error, 6 device wait timed out.
int time_candidate(const ConvShape &s, const Cand &c, int sms, SearchBuffers &sb,
                   cudaStream_t st, double *ms_out, std::string *why)
{
    if (!cand_valid(s, c, sms, why)) return 1;
    bigemm_plan_s *p = nullptr;
    if (make_plan(s, c, sms, &p) != BIGEMM_OK) {
        if (why) *why = "scratch allocation or descriptor encoding failed";
        return 4;
    }
    int status = 0;
    cudaEvent_t a = nullptr, b = nullptr;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    auto once = [&]() { return run_plan(p, sb.x, sb.w, sb.b, 1e-5f, sb.o, st); };
    auto flush = [&]() {
        return sb.flush ? cudaMemsetAsync(sb.flush, 0, sb.flush_bytes, st) : cudaSuccess;
    };
    // one run between events (after a flush when there is one); its time in ms, < 0 on failure
    auto timed_once = [&]() -> float {
        if (flush() != cudaSuccess) return -1.f;
        cudaEventRecord(a, st);
        if (once() != BIGEMM_OK) return -1.f;
        cudaEventRecord(b, st);
        if (cudaEventSynchronize(b) != cudaSuccess) return -1.f;
        float t = 0;
        cudaEventElapsedTime(&t, a, b);
        return t;
    };
    do {
        if (once() != BIGEMM_OK || cudaStreamSynchronize(st) != cudaSuccess) {
            status = 4;
            break;
        }
        const float one = timed_once();
        if (one < 0) { status = 4; break; }
        const double target = min_repeat_ms();
        const int cap = sb.flush ? 64 : 10000;
        const int number =
            (int)std::min((double)cap, std::max(1.0, std::ceil(target / std::max(one, 1e-4f))));
        double rep[3];
        for (int r = 0; r < 3 && status == 0; ++r) {
            double tot = 0;
            if (sb.flush) {
                for (int i = 0; i < number; ++i) {
                    const float t = timed_once();
                    if (t < 0) { status = 4; break; }
                    tot += t;
                }
            } else {
                cudaEventRecord(a, st);
                for (int i = 0; i < number; ++i)
                    if (once() != BIGEMM_OK) { status = 4; break; }
                cudaEventRecord(b, st);
                if (cudaEventSynchronize(b) != cudaSuccess) { status = 4; break; }
                float t = 0;
                cudaEventElapsedTime(&t, a, b);
                tot = t;
            }
            rep[r] = tot / number;
        }
        if (status) break;
        std::sort(rep, rep + 3);
        *ms_out = rep[1];
    } while (0);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (status == 0 && bigemm_last_device_error() == BIGEMM_ERR_TIMEOUT) {
        status = 6;
        bigemm_clear_device_error();
    }
    if (status == 4 && why) *why = cudaGetErrorString(cudaGetLastError());
    free_scratch(p);
    delete p;
    return status;
}

bigemm_status search(const ConvShape &s, int sms, cudaStream_t st, Cand *best, std::string *log,
                     const std::vector<Cand> &cands)
{
    SearchBuffers sb;
    const size_t e = dtype_size(s.in_dt);
    const long long xn = (long long)s.N * s.CI * s.H * s.W;
    const long long wn = (long long)s.CO * (s.CI / s.groups) * s.KH * s.KW;
    const size_t xb = (size_t)xn * e, wb = (size_t)wn * e;
    const size_t ob = (size_t)s.N * s.CO * s.Ho * s.Wo * dtype_size(s.out_dt);
    if (cudaMalloc(&sb.x, xb) != cudaSuccess || cudaMalloc(&sb.w, wb) != cudaSuccess ||
        cudaMalloc(&sb.o, ob) != cudaSuccess || cudaMalloc(&sb.b, s.CO * sizeof(float)) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    // inputs like the ones a layer sees: data in [-1, 1], kernel of variance
    // about 2/fan_in, bias in [-1, 1]
    const float fan = (float)((s.CI / s.groups) * s.KH * s.KW);
    if (fill_search_input(sb.x, xn, s.in_dt, 1.0f, 1, sms, st) != cudaSuccess ||
        fill_search_input(sb.w, wn, s.in_dt, sqrtf(6.0f / fan), 2, sms, st) != cudaSuccess ||
        fill_search_input(sb.b, s.CO, BIGEMM_F32, 1.0f, 3, sms, st) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    // An L2 flush before every timed run when the tensors would otherwise stay
    // in L2 between runs: twice the L2 size, written with a memset.
    int dev = 0, l2 = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) == cudaSuccess && l2 > 0 &&
        xb + wb + ob < 2 * (size_t)l2) {
        sb.flush_bytes = 2 * (size_t)l2;
        if (cudaMalloc(&sb.flush, sb.flush_bytes) != cudaSuccess) {
            sb.flush = nullptr;
            return BIGEMM_ERR_CUDA;
        }
    }
    if (cudaStreamSynchronize(st) != cudaSuccess) return BIGEMM_ERR_CUDA;
    double best_ms = 1e30;
    int best_i = -1;
    std::ostringstream os;
    os.precision(9);   // enough digits that the log orders the records as the choice did
    os << "[";
    for (size_t i = 0; i < cands.size(); ++i) {
        double ms = 0;
        std::string why;
        const int status = time_candidate(s, cands[i], sms, sb, st, &ms, &why);
        if (getenv("BIGEMM_LOG"))
            fprintf(stderr, "[bigemm] %-44s status=%d ms=%.5f %s\n", cand_str(cands[i]).c_str(),
                    status, status ? 0.0 : ms, why.c_str());
        os << (i ? ", " : "") << "{\"cand\": \"" << cand_str(cands[i]) << "\", \"status\": " << status;
        if (status == 0) os << ", \"ms\": " << ms;
        os << "}";
        if (status == 0 && ms < best_ms) best_ms = ms, best_i = (int)i;   // ties: lowest index
        if (status == 4 && cudaDeviceSynchronize() != cudaSuccess) break;  // context lost
    }
    os << "]";
    *log = os.str();
    if (best_i < 0) return BIGEMM_ERR_NO_CANDIDATE;
    *best = cands[best_i];
    return BIGEMM_OK;
}

bigemm_status plan_impl(int N, int H, int W, int CO, int CI, int KH, int KW, int stride,
                        int padding, int groups, bigemm_dtype in_dt, bigemm_dtype out_dt,
                        bigemm_epilogue epi, int do_search, const bigemm_plan_options *opts,
                        void *stream, bigemm_plan *out_plan)
{
    if (!out_plan) return BIGEMM_ERR_INVALID_ARG;
    *out_plan = nullptr;
    ConvShape s{N, CI, H, W, CO, KH, KW, stride, padding, groups, 0, 0, (int)in_dt, (int)out_dt, (int)epi};
    if (stride >= 1 && padding >= 0 && KH >= 1 && KW >= 1) {
        s.Ho = out_extent(H, KH, stride, padding);
        s.Wo = out_extent(W, KW, stride, padding);
    }
    bigemm_status r = validate(s);
    if (r != BIGEMM_OK) return r;
    DeviceState *ds = device_state();
    if (!ds) return BIGEMM_ERR_CUDA;
    const int sms = ds->sm_count;
    cudaStream_t st = (cudaStream_t)stream;

    const bool forced = opts && (opts->kind || opts->tile_n || opts->split_k || opts->box_w ||
                                 opts->box_h || opts->stages || opts->mode || opts->resident_b ||
                                 opts->epi_warps || opts->cta_pair);
    Cand c;
    std::string log, chosen = "heuristic";
    if (forced) {
        if (opts->kind == BIGEMM_KIND_SIMT || (opts->kind == 0 && !opts->tile_n && !opts->split_k &&
                                               !opts->box_w && !opts->box_h && !opts->stages &&
                                               !opts->mode && !opts->resident_b && !opts->cta_pair)) {
            c = heuristic(s, sms);
            if (opts->epi_warps != 0 && opts->epi_warps != 8 && opts->epi_warps != 16)
                return BIGEMM_ERR_INVALID_ARG;
            if (c.kind == BIGEMM_KIND_UMMA && opts->epi_warps)
                c.t.epi16 = opts->epi_warps == 16 ? 1 : 0;
            if (opts->kind == BIGEMM_KIND_SIMT && opts->mode != 0) {
                // an explicit SIMT kernel: 1 tiled (groups = 1) or naive, 2 depthwise staged
                // band (box_h rows per block), 3 depthwise streaming (box_h rows per thread),
                // 4 depthwise whole planes (H, W <= 32), 5 depthwise small planes (stride 1,
                // outputs at most 16 x 32; box_h = 2 or 4 output rows per thread), 6
                // depthwise bands of rows (input rows of 16-byte chunks, at most 512 bytes)
                if (opts->mode < 1 || opts->mode > 6) return BIGEMM_ERR_INVALID_ARG;
                c = Cand{};
                if (opts->mode == 1) {
                    c.simt_variant = groups == 1 ? SV_TILED : SV_NAIVE;
                } else if (opts->mode == 2) {
                    c.simt_variant = SV_DW;
                    c.dw_rows = opts->box_h > 0 ? opts->box_h : 8;
                } else if (opts->mode == 4) {
                    c.simt_variant = SV_DWP;
                } else if (opts->mode == 6) {
                    c.simt_variant = SV_DWB;
                } else if (opts->mode == 5) {
                    c.simt_variant = SV_DWR;
                    c.dw_rows = opts->box_h > 0 ? opts->box_h : 4;
                    if (c.dw_rows != 2 && c.dw_rows != 4) return BIGEMM_ERR_INVALID_ARG;
                } else {
                    c.simt_variant = SV_DWS;
                    c.dw_rows = opts->box_h > 0 ? opts->box_h : 2;
                    if (c.dw_rows != 2 && c.dw_rows != 4 && c.dw_rows != 8) return BIGEMM_ERR_INVALID_ARG;
                }
            } else if (opts->kind == BIGEMM_KIND_SIMT && is_depthwise(s) && opts->box_h > 0) {
                // the staged-band depthwise kernel with box_h output rows per block
                c = Cand{};
                c.simt_variant = SV_DW;
                c.dw_rows = opts->box_h;
            } else if (c.kind == BIGEMM_KIND_UMMA) {
                c = Cand{};
                c.simt_variant = is_depthwise(s) ? SV_DW : (groups == 1 ? SV_TILED : SV_NAIVE);
                if (c.simt_variant == SV_DW) {
                    c.dw_rows = std::max(1, std::min(s.Ho, 2048 / std::max(1, s.Wo)));
                    while (c.dw_rows > 1 && !simt_valid(s, c, nullptr)) c.dw_rows /= 2;
                }
            }
        } else {
            c.kind = BIGEMM_KIND_UMMA;
            if (opts->mode < 0 || opts->mode > 7) return BIGEMM_ERR_INVALID_ARG;
            const int amode = (opts->mode == 1 || opts->mode == 4 || opts->mode == 7) ? A_NHWC
                              : opts->mode == 2                    ? A_DIRECT
                              : (opts->mode == 3 || opts->mode == 5) ? A_HALO
                              : opts->mode == 6                    ? A_STRIDED
                              : (opts->box_w && opts->box_h)         ? A_NHWC
                              : direct_ok(s)                         ? A_DIRECT
                              : strided_ok(s)                        ? A_STRIDED
                              : sub_ok(s)                            ? A_NHWC
                              : halo_ok(s)                           ? A_HALO
                                                                     : A_NHWC;
            const int pack = opts->mode == 4   ? PACK_SUB
                             : opts->mode == 5 ? PACK_STACK
                             : opts->mode == 7 ? PACK_IM2COL
                             : opts->mode != 0 ? PACK_PLAIN
                             : amode == A_NHWC && sub_ok(s) && !(opts->box_w && opts->box_h) ? PACK_SUB
                             : amode == A_HALO ? halo_pack(s)
                                               : PACK_PLAIN;
            c.t = default_tiling(s, amode, opts->tile_n ? opts->tile_n : default_bn(s), sms, pack);
            if (opts->box_w && opts->box_h && pack != PACK_IM2COL) {
                c.t.box_w = opts->box_w, c.t.box_h = opts->box_h;
                c.t.bpt = std::max(1, 128 / (opts->box_w * opts->box_h));
                c.t.split = heuristic_split(s, c.t, sms);
            }
            if (opts->split_k) c.t.split = opts->split_k;
            if (opts->stages) c.t.stages = opts->stages;
            if (opts->resident_b < -1 || opts->resident_b > 1) return BIGEMM_ERR_INVALID_ARG;
            if (opts->resident_b == 1) {
                c.t.bres = 1;
                // resident weights outside the halo modes run whole K ranges
                if (c.t.amode != A_HALO && !opts->split_k) c.t.split = 1;
            } else if (opts->resident_b == 0) {
                prefer_resident(s, c.t);
            }
            if (opts->epi_warps != 0 && opts->epi_warps != 8 && opts->epi_warps != 16)
                return BIGEMM_ERR_INVALID_ARG;
            if (opts->epi_warps == 16)
                c.t.epi16 = 1;
            else if (opts->epi_warps == 0)
                prefer_epi16(s, c.t);
            if (opts->cta_pair < -1 || opts->cta_pair > 1) return BIGEMM_ERR_INVALID_ARG;
            if (opts->cta_pair == 1) c.t.pair = 1;
        }
        std::string why;
        if (!cand_valid(s, c, sms, &why)) return BIGEMM_ERR_UNSUPPORTED;
        chosen = "forced";
    } else if (do_search) {
        const std::string key = cache_key(s);
        bool hit = false;
        {
            std::lock_guard<std::mutex> lk(g_cache_mu);
            load_cache_file();
            auto it = g_cache.find(key);
            if (it != g_cache.end() && parse_cand(it->second.first, c) && cand_valid(s, c, sms, nullptr)) {
                hit = true;
                chosen = "cache";
            }
        }
        if (!hit) {
            r = search(s, sms, st, &c, &log, candidates(s, sms));
            if (r != BIGEMM_OK) return r;
            chosen = "search";
            double ms = 0;
            size_t at = log.find("\"cand\": \"" + cand_str(c) + "\"");
            if (at != std::string::npos) {
                size_t m = log.find("\"ms\": ", at);
                if (m != std::string::npos) ms = atof(log.c_str() + m + 6);
            }
            std::lock_guard<std::mutex> lk(g_cache_mu);
            g_cache[key] = {cand_str(c), ms};
            append_cache_file(key, cand_str(c), ms);
        }
    } else {
        c = heuristic(s, sms);
    }
    bigemm_plan_s *p = nullptr;
    r = make_plan(s, c, sms, &p);
    if (r != BIGEMM_OK) return r;
    p->search_log = log;
    p->chosen_by = chosen;
    *out_plan = p;
    return BIGEMM_OK;
}

}  // namespace
}  // namespace bigemm

extern "C" {

bigemm_status conv2d_nchw_plan(int N, int H, int W, int CO, int CI, int KH, int KW, int stride,
                               int padding, int groups, bigemm_dtype in_dtype,
                               bigemm_dtype out_dtype, bigemm_epilogue epi, int search,
                               void *stream, bigemm_plan *out_plan)
{
    return plan_impl(N, H, W, CO, CI, KH, KW, stride, padding, groups, in_dtype, out_dtype, epi,
                     search, nullptr, stream, out_plan);
}

bigemm_status conv2d_nchw_plan_ex(int N, int H, int W, int CO, int CI, int KH, int KW,
                                  int stride, int padding, int groups, bigemm_dtype in_dtype,
                                  bigemm_dtype out_dtype, bigemm_epilogue epi, int search,
                                  const bigemm_plan_options *opts, void *stream,
                                  bigemm_plan *out_plan)
{
    return plan_impl(N, H, W, CO, CI, KH, KW, stride, padding, groups, in_dtype, out_dtype, epi,
                     search, opts, stream, out_plan);
}

bigemm_status conv2d_nchw_run(bigemm_plan plan, const void *data, const void *kernel,
                              const float *bias, float eps, void *out, void *stream)
{
    if (!plan) return BIGEMM_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BIGEMM_ERR_CUDA;
    if (dev != plan->device) return BIGEMM_ERR_INVALID_ARG;
    return run_plan(plan, data, kernel, bias, eps, out, (cudaStream_t)stream);
}

bigemm_status conv2d_nchw_plan_destroy(bigemm_plan plan)
{
    if (!plan) return BIGEMM_ERR_INVALID_ARG;
    cudaDeviceSynchronize();
    free_scratch(plan);
    delete plan;
    return BIGEMM_OK;
}

bigemm_status conv2d_nchw_plan_describe(bigemm_plan plan, char *buf, size_t len)
{
    if (!plan || !buf || len == 0) return BIGEMM_ERR_INVALID_ARG;
    std::ostringstream os;
    const Cand &c = plan->c;
    os << "{\"cand\": \"" << cand_str(c) << "\", \"kind\": \""
       << (c.kind == BIGEMM_KIND_UMMA ? "umma" : "simt") << "\"";
    if (c.kind == BIGEMM_KIND_UMMA) {
        const UmmaParams &p = plan->g.p;
        os << ", \"amode\": \"" << amode_name(c.t.amode)
           << "\", \"pack\": \""
           << (c.t.pack == PACK_SUB      ? "sub"
               : c.t.pack == PACK_STACK  ? "stack"
               : c.t.pack == PACK_IM2COL ? "im2col"
                                         : "plain")
           << "\", \"resident_b\": " << (c.t.bres ? "true" : "false")
           << ", \"epi_warps\": " << (c.t.epi16 ? 16 : 8)
           << ", \"cta_pair\": " << (c.t.pair ? "true" : "false")
           << ", \"bn\": " << c.t.bn
           << ", \"box\": [" << c.t.box_w << ", " << c.t.box_h << ", " << c.t.bpt << "]"
           << ", \"split\": " << p.split << ", \"k_blocks\": " << p.k_blocks
           << ", \"split_sum\": \"" << (p.split == 1 ? "none" : plan->red_add ? "add" : "reduce") << "\""
           << ", \"pix_tiles\": " << p.pix_tiles << ", \"co_tiles\": " << p.co_tiles
           << ", \"units\": " << p.units << ", \"grid\": " << plan->g.grid
           << ", \"smem\": " << ((c.t.amode == A_HALO || c.t.amode == A_STRIDED || c.t.bres)
                                   ? (size_t)p.halo_smem : umma_smem_bytes(c.t))
           << ", \"halo_stages\": " << p.halo_sa << ", \"weight_stages\": " << p.halo_sb
           << ", \"store\": \"" << (plan->store_tma ? "tma" : "direct") << "\"";
    }
    os << ", \"launches\": " << launches_per_run(plan)
       << ", \"scratch_bytes\": " << (plan->xh_bytes + plan->wp_bytes + plan->ws_bytes)
       << ", \"chosen_by\": \"" << plan->chosen_by << "\"";
    if (!plan->search_log.empty()) os << ", \"search\": " << plan->search_log;
    os << "}";
    const std::string s = os.str();
    const size_t n = std::min(len - 1, s.size());
    memcpy(buf, s.data(), n);
    buf[n] = 0;
    return BIGEMM_OK;
}

}  // extern "C"
