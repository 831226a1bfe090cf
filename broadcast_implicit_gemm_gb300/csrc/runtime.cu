// runtime.cu -- per-device state, the sticky device error word, the bound on
// device-side waits, per-kernel event timing, and TMA descriptor encoding.
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace bigemm {

namespace {

std::mutex g_mu;
DeviceState g_dev[64];
// The sticky error word, one per device (every GPU that loads the library
// holds its own copy, zero at load).  A file-scope device variable rather than
// an allocation, so that the allocation-free entry point can raise it too.
static __device__ int g_err_word;
std::atomic<unsigned long long> g_timeout_ns{2000000000ull};

struct ProfRec {
    const char *name;
    cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event()
{
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// One block, one thread: a barrier nothing arrives on, waited on with the
// same bounded wait the conv kernels use.
__global__ void wait_timeout_probe_kernel(int *err, unsigned long long timeout_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, timeout_ns, (volatile int *)&abort_flag, err);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

typedef CUresult (*EncodeIm2colFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const int *, const int *,
                                   cuuint32_t, cuuint32_t, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeIm2colFn encode_im2col_fn()
{
    static EncodeIm2colFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeIm2colFn>(p);
    });
    return fn;
}

}  // namespace

DeviceState *device_state()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (d.device == dev) return &d;
    int sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return nullptr;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return nullptr;
    // the device address of g_err_word on this device (its name in host code
    // is a host-side stand-in, not a device address)
    int *err = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&err), g_err_word) != cudaSuccess || !err)
        return nullptr;
    d.sm_count = sms;
    d.max_smem_optin = smem;
    d.err = err;
    d.device = dev;
    return &d;
}

unsigned long long wait_timeout_ns() { return g_timeout_ns.load(); }

ProfScope::ProfScope(const char *name, cudaStream_t s) : name_(name), s_(s)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return;
    ProfRec r{name, take_event(), take_event()};
    if (!r.a || !r.b) return;
    cudaEventRecord(r.a, s);
    slot_ = (int)g_prof.size();
    g_prof.push_back(r);
}

ProfScope::~ProfScope()
{
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (slot_ < (int)g_prof.size()) cudaEventRecord(g_prof[slot_].b, s_);
}

bool encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                  const uint32_t *estrides, CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = estrides[i];
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    CUresult r = fn(map, dt, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_im2col(CUtensorMap *map, CUtensorMapDataType dt, const void *base,
                   const uint64_t *dims, const uint64_t *strides_bytes, const int *lower,
                   const int *upper, uint32_t channels, uint32_t pixels, const uint32_t *estrides,
                   CUtensorMapSwizzle swz)
{
    EncodeIm2colFn fn = encode_im2col_fn();
    if (!fn) return false;
    cuuint64_t d[4], st[3];
    cuuint32_t es[4];
    for (int i = 0; i < 4; ++i) {
        d[i] = dims[i];
        es[i] = estrides[i];
        if (i < 3) st[i] = strides_bytes[i];
    }
    int lo[2] = {lower[0], lower[1]}, up[2] = {upper[0], upper[1]};
    CUresult r = fn(map, dt, 4u, const_cast<void *>(base), d, st, lo, up, channels, pixels, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaError_t launch_wait_timeout_probe(int *err, unsigned long long timeout_ns,
                                      cudaStream_t stream)
{
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace bigemm

using namespace bigemm;

extern "C" {

bigemm_status bigemm_set_wait_timeout_ns(uint64_t ns)
{
    g_timeout_ns.store(ns < 1000 ? 1000 : ns);
    return BIGEMM_OK;
}

bigemm_status bigemm_last_device_error(void)
{
    DeviceState *ds = device_state();
    if (!ds) return BIGEMM_ERR_CUDA;
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return BIGEMM_ERR_CUDA;
    if (cudaMemcpy(&v, ds->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    return v ? BIGEMM_ERR_TIMEOUT : BIGEMM_OK;
}

bigemm_status bigemm_clear_device_error(void)
{
    DeviceState *ds = device_state();
    if (!ds) return BIGEMM_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return BIGEMM_ERR_CUDA;
    if (cudaMemset(ds->err, 0, sizeof(int)) != cudaSuccess) return BIGEMM_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return BIGEMM_ERR_CUDA;
    return BIGEMM_OK;
}

bigemm_status bigemm_debug_wait_timeout(uint64_t timeout_ns, void *stream)
{
    DeviceState *ds = device_state();
    if (!ds) return BIGEMM_ERR_CUDA;
    if (timeout_ns < 1000) timeout_ns = 1000;
    if (timeout_ns > 5000000000ull) return BIGEMM_ERR_INVALID_ARG;
    if (launch_wait_timeout_probe(ds->err, timeout_ns, (cudaStream_t)stream) != cudaSuccess)
        return BIGEMM_ERR_CUDA;
    return BIGEMM_OK;
}

bigemm_status bigemm_profile_enable(int on)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (on) {
        cudaDeviceSynchronize();
        for (auto &r : g_prof) {
            g_event_pool.push_back(r.a);
            g_event_pool.push_back(r.b);
        }
        g_prof.clear();
    }
    g_prof_on = on != 0;
    return BIGEMM_OK;
}

bigemm_status bigemm_profile_read(bigemm_kernel_time *out, int max, int *count)
{
    if (!count || (max > 0 && !out)) return BIGEMM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (cudaDeviceSynchronize() != cudaSuccess) return BIGEMM_ERR_CUDA;
    std::vector<std::pair<std::string, std::pair<int, double>>> agg;
    for (auto &r : g_prof) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) continue;
        bool found = false;
        for (auto &e : agg)
            if (e.first == r.name) {
                e.second.first += 1;
                e.second.second += ms;
                found = true;
                break;
            }
        if (!found) agg.push_back({r.name, {1, (double)ms}});
    }
    *count = (int)agg.size();
    for (int i = 0; i < (int)agg.size() && i < max; ++i) {
        std::memset(out[i].name, 0, sizeof(out[i].name));
        std::strncpy(out[i].name, agg[i].first.c_str(), sizeof(out[i].name) - 1);
        out[i].launches = agg[i].second.first;
        out[i].total_ms = agg[i].second.second;
    }
    return BIGEMM_OK;
}

}  // extern "C"
