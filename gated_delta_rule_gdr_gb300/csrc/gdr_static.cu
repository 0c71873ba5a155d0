// gdr_static.cu -- chunked prefill that allocates nothing: the staged kernels
// (decay, WY/UT, state pass, output) run on a fixed scratch area that the
// library owns, instead of on stream-ordered scratch from cudaMallocAsync.
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

#include <cmath>
#include <cstdint>
#include <mutex>

namespace {

// Fixed scratch: 32 MiB of device memory, held by every GPU that loads the
// library until the process exits.  Host code must never pass the symbol
// itself to a kernel (on the host it is only a stand-in, not a device
// address); it resolves the device address once per device below.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the calling thread's current device,
// looked up with that device current the first time and cached afterwards.
cudaError_t scratch_on_current_device(void **addr) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
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
    if (BH > 0x7fffffff) return GDR_ERR_UNSUPPORTED;
    const int64_t NC = ((int64_t)T + chunk - 1) / chunk;
    const int64_t n_tok = BH * (int64_t)T;
    // gamma, U, Wk, W per token-head and one state per chunk start, all fp32
    const int64_t need = (int64_t)sizeof(float) *
                         (n_tok * (1 + (int64_t)dv + dk + dv) + BH * NC * (int64_t)dk * dv);
    if (need > (int64_t)kStaticScratchBytes) return GDR_ERR_UNSUPPORTED;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *scratch = nullptr;
    if (scratch_on_current_device(&scratch) != cudaSuccess) return GDR_ERR_CUDA;
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
    float *gamma = static_cast<float *>(scratch);
    float *U = gamma + n_tok;
    float *Wk = U + n_tok * dv;
    float *W = Wk + n_tok * dk;
    float *Mn = W + n_tok * dv;
    const int bh = (int)BH;
    cudaError_t err = gdr::launch_decay(g, a_min, gamma, bh, T, chunk, s);
    if (err == cudaSuccess)
        err = gdr::launch_wy(k, v, beta, gamma, U, Wk, bh, T, dk, dv, chunk, e, s);
    if (err == cudaSuccess)
        err = gdr::launch_state(k, gamma, U, Wk, init_state, W, Mn, final_state, bh, T, dk, dv,
                                chunk, e, s);
    if (err == cudaSuccess)
        err = gdr::launch_output(q, k, gamma, Mn, W, out, bh, T, dk, dv, chunk, e, s);
    return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}
