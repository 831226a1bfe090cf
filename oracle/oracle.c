/*
 * oracle.c -- plain CPU reference for NCHW 2-D convolution and the per-channel
 * NCHW broadcast.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, loads or calls this
 * file.  It is used by the tests, by the smoke check and by the benchmark's
 * CPU-baseline leg, and by nothing else.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * It is the plain definition written out, in double precision, with one
 * output element computed at a time:
 *
 *   conv2d  -- "Tuning High Performance Convolution on NVIDIA GPUs" (TVM v0.5
 *              autotvm tutorial), Step 1: the compute is
 *              topi.nn.conv2d_nchw(data[N,CI,H,W], kernel[CO,CI,KH,KW], stride,
 *              padding, dilation=1), with the zero-padding stage inlined
 *              ("inline padding").  Output axes n,f,y,x; reduce axes rc,ry,rx:
 *                out[n,f,y,x] = sum_{rc,ry,rx} pad(data)[n,rc,y*s+ry,x*s+rx]
 *                                            * kernel[f,rc,ry,rx]
 *              where pad() adds `padding` zeros on every side of H and W.
 *              Grouped convolution (groups = CI = CO, i.e. depthwise, which
 *              the tutorial names as a variant of the same template) reads
 *              input channel g*(CI/groups)+rc for output channel f in group g.
 *   broadcast -- "[CINN] Add the TileBroadcastTactic for NCHW broadcast"
 *              (PaddlePaddle PR 70092), Introduction and Example: a
 *              per-channel value [1,C,1,1] => [N,C,H,W], e.g.
 *              out[n,c,h,w] = exp(var[c]).
 *
 * Precision: inputs arrive as doubles that hold the exact values the device
 * kernels read (fp16/bf16/fp32 values widen exactly); products and sums are
 * formed in fp64 in the fixed order rc -> ry -> rx.  Each conv output also
 * returns S = sum |a*w| over the same terms, the scale of the tolerance.
 *
 * Parity is pinned by the tests (hand-worked cases, identity / all-ones /
 * spike closed forms, the output-size rule, the FLOP count against the
 * tutorial's tuning log, and a float64 library convolution on small shapes).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Output extent of one spatial axis: floor((in + 2*pad - k) / stride) + 1.
 * Returns 0 when the window does not fit and -1 for a non-positive stride. */
int oracle_out_size(int in, int k, int stride, int pad)
{
    if (stride <= 0 || k <= 0 || in < 0 || pad < 0) return -1;
    int span = in + 2 * pad - k;
    if (span < 0) return 0;
    return span / stride + 1;
}

/* 2 * N * CO * Ho * Wo * (CI/groups) * KH * KW : one multiply and one add per
 * reduction term, the count the tutorial's tuner divides by the run time. */
double oracle_conv_flops(int N, int CI, int H, int W, int CO, int KH, int KW,
                         int stride, int pad, int groups)
{
    int Ho = oracle_out_size(H, KH, stride, pad);
    int Wo = oracle_out_size(W, KW, stride, pad);
    if (Ho <= 0 || Wo <= 0 || groups <= 0) return 0.0;
    return 2.0 * N * CO * (double)Ho * Wo * (CI / groups) * KH * KW;
}

/* Epilogue codes (the fused per-channel broadcast applied to the conv sum):
 * the complex ops the CINN broadcast page names -- div, exp, rsqrt -- each
 * after the per-channel bias, and add + ReLU: max(acc + bias[f], 0). */
enum { ORC_EPI_NONE = 0, ORC_EPI_BIAS = 1, ORC_EPI_BIAS_EXP = 2, ORC_EPI_BIAS_RSQRT = 3,
       ORC_EPI_BIAS_RECIP = 4, ORC_EPI_BIAS_RELU = 5 };

typedef struct {
    int N, CI, H, W, CO, KH, KW, stride, pad, groups, Ho, Wo;
} conv_shape;

static int make_shape(conv_shape *s, int N, int CI, int H, int W, int CO, int KH,
                      int KW, int stride, int pad, int groups)
{
    s->N = N; s->CI = CI; s->H = H; s->W = W; s->CO = CO; s->KH = KH; s->KW = KW;
    s->stride = stride; s->pad = pad; s->groups = groups;
    if (N < 0 || CI <= 0 || CO <= 0 || H <= 0 || W <= 0 || KH <= 0 || KW <= 0) return -1;
    if (groups <= 0 || CI % groups != 0 || CO % groups != 0) return -1;
    s->Ho = oracle_out_size(H, KH, stride, pad);
    s->Wo = oracle_out_size(W, KW, stride, pad);
    if (s->Ho <= 0 || s->Wo <= 0) return -1;
    return 0;
}

/* One output element, straight from the definition. */
static void conv_point(const conv_shape *s, const double *data, const double *kernel,
                       int n, int f, int y, int x, double *acc_out, double *abs_out)
{
    const int cig = s->CI / s->groups;          /* input channels per group  */
    const int cog = s->CO / s->groups;          /* output channels per group */
    const int g = f / cog;                      /* group of output channel f */
    double acc = 0.0, sabs = 0.0;
    for (int rc = 0; rc < cig; ++rc) {
        const int ci = g * cig + rc;
        for (int ry = 0; ry < s->KH; ++ry) {
            const int iy = y * s->stride + ry - s->pad;
            for (int rx = 0; rx < s->KW; ++rx) {
                const int ix = x * s->stride + rx - s->pad;
                double a = 0.0;                 /* zero padding outside [0,H)x[0,W) */
                if (iy >= 0 && iy < s->H && ix >= 0 && ix < s->W)
                    a = data[(((size_t)n * s->CI + ci) * s->H + iy) * s->W + ix];
                const double w = kernel[(((size_t)f * cig + rc) * s->KH + ry) * s->KW + rx];
                acc += a * w;
                sabs += fabs(a * w);
            }
        }
    }
    *acc_out = acc;
    *abs_out = sabs;
}

static double apply_epilogue(int epi, double acc, const double *bias, int f, double eps)
{
    switch (epi) {
    case ORC_EPI_NONE:       return acc;
    case ORC_EPI_BIAS:       return acc + bias[f];
    case ORC_EPI_BIAS_EXP:   return exp(acc + bias[f]);
    case ORC_EPI_BIAS_RSQRT: return 1.0 / sqrt(acc + bias[f] + eps);
    case ORC_EPI_BIAS_RECIP: return 1.0 / (acc + bias[f]);
    case ORC_EPI_BIAS_RELU:  return acc + bias[f] > 0.0 ? acc + bias[f] : 0.0;
    default:                 return NAN;
    }
}

/* Full convolution.  out and absum are [N, CO, Ho, Wo]; absum may be NULL.
 * bias is [CO] (read only when epi != NONE).  nthreads > 1 splits the
 * (n, f) planes over OpenMP threads; each element is computed the same way.
 * Returns 0, or -1 for an invalid shape / epilogue. */
int oracle_conv2d_nchw(int N, int CI, int H, int W, int CO, int KH, int KW,
                       int stride, int pad, int groups,
                       const double *data, const double *kernel, const double *bias,
                       int epi, double eps, double *out, double *absum, int nthreads)
{
    conv_shape s;
    if (make_shape(&s, N, CI, H, W, CO, KH, KW, stride, pad, groups) != 0) return -1;
    if (epi < ORC_EPI_NONE || epi > ORC_EPI_BIAS_RELU) return -1;
    if (epi != ORC_EPI_NONE && bias == NULL) return -1;
    const long planes = (long)N * CO;
    (void)nthreads;
#ifdef _OPENMP
    #pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (long pl = 0; pl < planes; ++pl) {
        const int n = (int)(pl / CO), f = (int)(pl % CO);
        for (int y = 0; y < s.Ho; ++y)
            for (int x = 0; x < s.Wo; ++x) {
                double acc, sabs;
                conv_point(&s, data, kernel, n, f, y, x, &acc, &sabs);
                const size_t o = (((size_t)n * CO + f) * s.Ho + y) * s.Wo + x;
                out[o] = apply_epilogue(epi, acc, bias, f, eps);
                if (absum) absum[o] = sabs;
            }
    }
    return 0;
}

/* The same definition at chosen outputs only: idx[i] is a flat index into
 * [N, CO, Ho, Wo].  Used for parity at sizes where a full CPU pass is too
 * slow.  Returns 0, or -1 for an invalid shape or an index out of range. */
int oracle_conv2d_nchw_points(int N, int CI, int H, int W, int CO, int KH, int KW,
                              int stride, int pad, int groups,
                              const double *data, const double *kernel, const double *bias,
                              int epi, double eps, long npts, const int64_t *idx,
                              double *out, double *absum)
{
    conv_shape s;
    if (make_shape(&s, N, CI, H, W, CO, KH, KW, stride, pad, groups) != 0) return -1;
    if (epi < ORC_EPI_NONE || epi > ORC_EPI_BIAS_RELU) return -1;
    if (epi != ORC_EPI_NONE && bias == NULL) return -1;
    const int64_t total = (int64_t)N * CO * s.Ho * s.Wo;
    for (long i = 0; i < npts; ++i) {
        int64_t t = idx[i];
        if (t < 0 || t >= total) return -1;
        const int x = (int)(t % s.Wo); t /= s.Wo;
        const int y = (int)(t % s.Ho); t /= s.Ho;
        const int f = (int)(t % CO);   t /= CO;
        const int n = (int)t;
        double acc, sabs;
        conv_point(&s, data, kernel, n, f, y, x, &acc, &sabs);
        out[i] = apply_epilogue(epi, acc, bias, f, eps);
        if (absum) absum[i] = sabs;
    }
    return 0;
}

/* Broadcast op codes. */
enum { ORC_BC_COPY = 0, ORC_BC_EXP = 1, ORC_BC_RSQRT = 2, ORC_BC_RECIP = 3 };

/* The per-channel value, in fp64.  For rsqrt the +eps is a float add, as the
 * device computes it; the square root and reciprocal are then exact-ish fp64. */
double oracle_bcast_value(int op, float v, float eps)
{
    switch (op) {
    case ORC_BC_COPY:  return (double)v;
    case ORC_BC_EXP:   return exp((double)v);
    case ORC_BC_RSQRT: {
        volatile float t = v + eps;             /* one fp32 rounding */
        return 1.0 / sqrt((double)t);
    }
    case ORC_BC_RECIP: return 1.0 / (double)v;
    default:           return NAN;
    }
}

/* out[n,c,h,w] = op(var[c]) for every n,h,w; out is [N,C,H,W] doubles. */
int oracle_bcast_nchw(int N, int C, int H, int W, int op, const float *var, float eps,
                      double *out)
{
    if (N < 0 || C <= 0 || H <= 0 || W <= 0) return -1;
    if (op < ORC_BC_COPY || op > ORC_BC_RECIP) return -1;
    const size_t hw = (size_t)H * W;
    for (int n = 0; n < N; ++n)
        for (int c = 0; c < C; ++c) {
            const double v = oracle_bcast_value(op, var[c], eps);
            double *plane = out + ((size_t)n * C + c) * hw;
            for (size_t i = 0; i < hw; ++i) plane[i] = v;
        }
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
