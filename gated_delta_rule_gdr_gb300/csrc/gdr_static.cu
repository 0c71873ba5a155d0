// gdr_static.cu -- chunked prefill that allocates nothing: the staged kernels
// (decay, WY/UT, state pass, output) run on a fixed scratch area that the
// library owns, instead of on scratch that the caller (or an allocator) provides.
//
// Who needs it: callers that must not allocate device memory while they run.
// Examples are a plugin inside a host framework that owns every byte of
// device memory through its own pool and forbids side allocations, and a
// latency-critical or certified deployment that allows no allocation after
// start-up, because an allocation can stall or fail with out-of-memory in
// mid-stream.  Such callers still pass their own input and output buffers;
// only the intermediates move to this static area.

#include "gdr.h"
#include "gdr_internal.h"

#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

namespace {

// Fixed scratch: 32 MiB of device memory, held by every GPU that loads the
// library until the process exits.  Host code must never pass the symbol
// itself to a kernel (on the host it is only a stand-in, not a device
// address); it resolves the device address below.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The array's device address is a property of the CUDA context the library's
// module is loaded in: another context on the same device, or the primary
// context re-created after cudaDeviceReset, loads the module again and may
// place the array elsewhere.  So the address is cached per context, keyed by
// the context's unique ID (cuCtxGetId: IDs are never reused within a process,
// unlike context handles), and looked up once in each context.
constexpr int kMaxContexts = 64;
struct CtxAddr {
    unsigned long long id;
    void *addr;
};
CtxAddr g_cache[kMaxContexts];
int g_cache_n = 0;
std::mutex g_cache_mu;

PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
    static PFN_cuCtxGetCurrent_v4000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                                 &q) == cudaSuccess &&
                q == cudaDriverEntryPointSuccess)
                   ? reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p)
                   : nullptr;
    }();
    return fn;
}
PFN_cuCtxGetId_v12000 ctx_get_id() {
    static PFN_cuCtxGetId_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault,
                                                 &q) == cudaSuccess &&
                q == cudaDriverEntryPointSuccess)
                   ? reinterpret_cast<PFN_cuCtxGetId_v12000>(p)
                   : nullptr;
    }();
    return fn;
}

// Unique ID of the calling thread's current context (making the device's
// primary context current first if the thread has none yet).
bool current_context_id(unsigned long long *id) {
    auto get = ctx_get_current();
    auto getid = ctx_get_id();
    if (!get || !getid) return false;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return false;
    if (ctx == nullptr) {
        int dev = 0;   // no context yet: bind the current device's primary context
        if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return false;
        if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    }
    return getid(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the calling thread's current context.
cudaError_t scratch_in_current_context(void **addr) {
    unsigned long long id = 0;
    if (!current_context_id(&id)) return cudaErrorDeviceUninitialized;
    std::lock_guard<std::mutex> lock(g_cache_mu);
    for (int i = 0; i < g_cache_n; ++i)
        if (g_cache[i].id == id) {
            *addr = g_cache[i].addr;
            return cudaSuccess;
        }
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    if (g_cache_n < kMaxContexts) g_cache[g_cache_n++] = {id, p};   // else look up every call
    *addr = p;
    return cudaSuccess;
}

bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool chunk_ok(int c) { return c == 16 || c == 32 || c == 64; }

}  // namespace

extern "C" gdr_status_t gdr_chunk_fwd_static(const void *q, const void *k, const void *v,
                                             const float *g, const float *beta, float a_min,
                                             const float *init_state, void *out,
                                             float *final_state, int B, int H, int T, int dk,
                                             int dv, int chunk, gdr_dtype_t dtype,
                                             void *stream) {
    if (B < 0 || H < 0 || T < 0) return GDR_ERR_INVALID_ARG;
    if (dtype != GDR_DTYPE_F32 && dtype != GDR_DTYPE_BF16) return GDR_ERR_UNSUPPORTED;
    if (!(a_min > 0.0f && a_min <= 1.0f)) return GDR_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv) || !chunk_ok(chunk)) return GDR_ERR_UNSUPPORTED;
    if ((double)chunk * -std::log((double)a_min) > 80.0) return GDR_ERR_RANGE;
    const int64_t BH = (int64_t)B * H;
    // Every token-head needs at least one fp32 value of scratch, so work with more
    // token-heads than the array has floats cannot fit; rejecting it first also keeps
    // the size formula below far from int64 overflow.
    if (BH > 0x7fffffff || BH * (int64_t)T > (int64_t)(kStaticScratchBytes / sizeof(float)))
        return GDR_ERR_UNSUPPORTED;
    if (gdr::staged_scratch_bytes(BH, T, dk, dv, chunk) > kStaticScratchBytes)
        return GDR_ERR_UNSUPPORTED;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *scratch = nullptr;
    if (scratch_in_current_context(&scratch) != cudaSuccess) return GDR_ERR_CUDA;
    if (BH == 0) return GDR_OK;
    if (T == 0) {
        if (final_state == nullptr) return GDR_OK;
        return gdr::launch_copy_state(init_state, final_state, BH * dk * dv, s) == cudaSuccess
                   ? GDR_OK
                   : GDR_ERR_CUDA;
    }
    if (!q || !k || !v || !g || !beta || !out) return GDR_ERR_INVALID_ARG;

    // Every intermediate is written before it is read, so nothing left over
    // from an earlier call needs clearing.
    const gdr::Elem e = dtype == GDR_DTYPE_F32 ? gdr::Elem::F32 : gdr::Elem::BF16;
    return gdr::launch_staged(q, k, v, g, beta, a_min, init_state, out, final_state, scratch,
                              (int)BH, T, dk, dv, chunk, e, s) == cudaSuccess
               ? GDR_OK
               : GDR_ERR_CUDA;
}
