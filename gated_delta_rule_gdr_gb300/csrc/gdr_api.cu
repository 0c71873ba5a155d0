// gdr_api.cu -- the extern "C" boundary of libgdr.so (declared in
// include/gdr.h): argument validation, dispatch to the kernels, status codes.
// No C++ exception crosses this file's functions.

#include "gdr.h"
#include "gdr_internal.h"

#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>

namespace {

using gdr::Elem;

bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool chunk_ok(int c) { return c == 16 || c == 32 || c == 64; }

// a_min in (0, 1]; NaN fails every comparison.
bool a_min_ok(float a_min) { return a_min > 0.0f && a_min <= 1.0f; }

// The pages' range argument allows a worst in-tile cumulative log-decay of
// -80 (e^-80 ~ 1.8e-35 stays a normal fp32 number, its reciprocal ~5.5e34
// stays finite).  With alpha >= a_min the worst is chunk * ln(a_min); with
// log alpha >= g_min it is chunk * g_min.  The kernels take one decay parameter
// d: d = a_min > 0 for the linear-domain form, d = g_min <= 0 for the log form.
bool range_ok(float d, int chunk) {
    const double worst = d > 0.0f ? std::log((double)d) : (double)d;
    return (double)chunk * -worst <= 80.0;
}
// The two-kernel path applies the bound over the pages' 16-token tile: its
// preparation splits each chunk's position-pair decay at 16-row reference
// points and its chain takes only factors at most 1, so the decay over a whole
// chunk may fall below fp32's range.
constexpr int kTile = 16;

gdr_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA; }

Elem elem_of(gdr_dtype_t d) { return d == GDR_DTYPE_F32 ? Elem::F32 : Elem::BF16; }

bool dtype_ok(gdr_dtype_t d) { return d == GDR_DTYPE_F32 || d == GDR_DTYPE_BF16; }

// Common checks of the staged-step entry points.
gdr_status_t check_staged(int BH, int T, int dk, int dv, int chunk) {
    if (BH < 0 || T < 0) return GDR_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv) || !chunk_ok(chunk)) return GDR_ERR_UNSUPPORTED;
    return GDR_OK;
}

// Process-wide options (gdr_set_option).  Relaxed atomics: a value set before a
// call is seen by that call's launches on any thread.
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_fused_variant{0};
std::atomic<int> g_chain_split{0};
std::atomic<int> g_segments{0};
std::atomic<int> g_bwd_variant{0};

}  // namespace

namespace gdr {
uint64_t opt_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
int opt_fused_variant() { return g_fused_variant.load(std::memory_order_relaxed); }
int opt_chain_split() { return g_chain_split.load(std::memory_order_relaxed); }
int opt_segments() { return g_segments.load(std::memory_order_relaxed); }
int opt_bwd_variant() { return g_bwd_variant.load(std::memory_order_relaxed); }
}  // namespace gdr

extern "C" {

gdr_status_t gdr_set_option(gdr_option_t option, int64_t value) {
    switch (option) {
        case GDR_OPT_WAIT_LIMIT_NS:
            if (value < 0) return GDR_ERR_INVALID_ARG;
            g_wait_limit_ns.store((uint64_t)value, std::memory_order_relaxed);
            return GDR_OK;
        case GDR_OPT_FUSED_VARIANT:
            if (value < 0 || value > 2) return GDR_ERR_INVALID_ARG;
            g_fused_variant.store((int)value, std::memory_order_relaxed);
            return GDR_OK;
        case GDR_OPT_CHAIN_SPLIT:
            if (value < 0 || value > 2) return GDR_ERR_INVALID_ARG;
            g_chain_split.store((int)value, std::memory_order_relaxed);
            return GDR_OK;
        case GDR_OPT_SEGMENTS:
            if (value < 0 || value > 4096) return GDR_ERR_INVALID_ARG;
            g_segments.store((int)value, std::memory_order_relaxed);
            return GDR_OK;
        case GDR_OPT_BWD_VARIANT:
            if (value < 0 || value > 2) return GDR_ERR_INVALID_ARG;
            g_bwd_variant.store((int)value, std::memory_order_relaxed);
            return GDR_OK;
    }
    return GDR_ERR_INVALID_ARG;
}

int64_t gdr_get_option(gdr_option_t option) {
    switch (option) {
        case GDR_OPT_WAIT_LIMIT_NS: return (int64_t)gdr::opt_wait_limit_ns();
        case GDR_OPT_FUSED_VARIANT: return gdr::opt_fused_variant();
        case GDR_OPT_CHAIN_SPLIT: return gdr::opt_chain_split();
        case GDR_OPT_SEGMENTS: return gdr::opt_segments();
        case GDR_OPT_BWD_VARIANT: return gdr::opt_bwd_variant();
    }
    return -1;
}

}  // extern "C"

namespace {

// The decay parameter of the kernels for an ABI decay mode and bound, or false.
bool decay_param(gdr_decay_t decay, float bound, float *d) {
    if (decay == GDR_DECAY_AFFINE && a_min_ok(bound)) { *d = bound; return true; }
    if (decay == GDR_DECAY_LOG && bound <= 0.0f && bound >= -1e30f) { *d = bound; return true; }
    return false;   // unknown mode, a bound out of its range, or NaN
}

gdr_status_t chunk_fwd_impl(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float a_min, const float *init_state, void *out,
                            float *final_state, int B, int H, int T, int dk, int dv, int chunk,
                            gdr_dtype_t dtype, void *stream) {
    if (B < 0 || H < 0 || T < 0) return GDR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return GDR_ERR_UNSUPPORTED;
    if (!dim_ok(dk) || !dim_ok(dv) || !chunk_ok(chunk)) return GDR_ERR_UNSUPPORTED;
    if (!range_ok(a_min, chunk)) return GDR_ERR_RANGE;
    const int64_t BH = (int64_t)B * H;
    if (BH > 0x7fffffff || (int64_t)T * BH > ((int64_t)1 << 40)) return GDR_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (BH == 0) return GDR_OK;
    if (T == 0) {
        if (final_state == nullptr) return GDR_OK;
        return from_cuda(gdr::launch_copy_state(init_state, final_state, BH * dk * dv, s));
    }
    if (!q || !k || !v || !g || !beta || !out) return GDR_ERR_INVALID_ARG;
    const Elem e = elem_of(dtype);

    if (gdr::fused_supported(dk, dv, chunk, e))
        return from_cuda(gdr::launch_fused(q, k, v, g, beta, a_min, init_state, out,
                                           final_state, B, H, T, dk, dv, chunk, s));
    // every other shape and fp32: one CUDA-core launch, no scratch
    return from_cuda(gdr::launch_onepass(q, k, v, g, beta, a_min, init_state, out, final_state,
                                         (int)BH, T, dk, dv, chunk, e, s));
}

gdr_status_t decode_impl(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, float a_min, float *state, void *out, int N, int H,
                         int dk, int dv, gdr_dtype_t dtype, void *stream) {
    if (N < 0 || H < 0) return GDR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return GDR_ERR_UNSUPPORTED;
    if (!dim_ok(dk) || !dim_ok(dv)) return GDR_ERR_UNSUPPORTED;
    if ((int64_t)N * H == 0) return GDR_OK;
    if (!q || !k || !v || !g || !beta || !state || !out) return GDR_ERR_INVALID_ARG;
    if ((int64_t)N * H > 0x7fffffff) return GDR_ERR_UNSUPPORTED;
    return from_cuda(gdr::launch_decode(q, k, v, g, beta, a_min, state, out, N, H, dk, dv,
                                        elem_of(dtype), static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

gdr_status_t gdr_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float a_min, const float *init_state, void *out,
                           float *final_state, int B, int H, int T, int dk, int dv, int chunk,
                           gdr_dtype_t dtype, void *stream) {
    if (B < 0 || H < 0 || T < 0) return GDR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return GDR_ERR_UNSUPPORTED;
    if (!a_min_ok(a_min)) return GDR_ERR_INVALID_ARG;
    return chunk_fwd_impl(q, k, v, g, beta, a_min, init_state, out, final_state, B, H, T, dk, dv,
                          chunk, dtype, stream);
}

gdr_status_t gdr_decode_step(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, float a_min, float *state, void *out, int N,
                             int H, int dk, int dv, gdr_dtype_t dtype, void *stream) {
    if (N < 0 || H < 0) return GDR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return GDR_ERR_UNSUPPORTED;
    if (!a_min_ok(a_min)) return GDR_ERR_INVALID_ARG;
    return decode_impl(q, k, v, g, beta, a_min, state, out, N, H, dk, dv, dtype, stream);
}

gdr_status_t gdr_decode_step_ex(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, gdr_decay_t decay, float bound, float *state,
                                void *out,
                                int N, int H, int dk, int dv, gdr_dtype_t dtype, void *stream) {
    float d = 0.0f;
    if (N < 0 || H < 0) return GDR_ERR_INVALID_ARG;
    if (!decay_param(decay, bound, &d)) return GDR_ERR_INVALID_ARG;
    return decode_impl(q, k, v, g, beta, d, state, out, N, H, dk, dv, dtype, stream);
}

gdr_status_t gdr_chunk_decay(const float *g, float a_min, float *gamma, int BH, int T,
                             int chunk, void *stream) {
    if (BH < 0 || T < 0) return GDR_ERR_INVALID_ARG;
    if (!a_min_ok(a_min)) return GDR_ERR_INVALID_ARG;
    if (!chunk_ok(chunk)) return GDR_ERR_UNSUPPORTED;
    if (!range_ok(a_min, chunk)) return GDR_ERR_RANGE;
    if ((int64_t)BH * T == 0) return GDR_OK;
    if (!g || !gamma) return GDR_ERR_INVALID_ARG;
    return from_cuda(gdr::launch_decay(g, a_min, gamma, BH, T, chunk,
                                       static_cast<cudaStream_t>(stream)));
}

gdr_status_t gdr_chunk_wy(const void *k, const void *v, const float *beta, const float *gamma,
                          float *U, float *Wk, int BH, int T, int dk, int dv, int chunk,
                          gdr_dtype_t dtype, void *stream) {
    if (!dtype_ok(dtype)) return GDR_ERR_UNSUPPORTED;
    gdr_status_t st = check_staged(BH, T, dk, dv, chunk);
    if (st != GDR_OK) return st;
    if ((int64_t)BH * T == 0) return GDR_OK;
    if (!k || !v || !beta || !gamma || !U || !Wk) return GDR_ERR_INVALID_ARG;
    return from_cuda(gdr::launch_wy(k, v, beta, gamma, U, Wk, BH, T, dk, dv, chunk,
                                    elem_of(dtype), static_cast<cudaStream_t>(stream)));
}

gdr_status_t gdr_chunk_state(const void *k, const float *gamma, const float *U,
                             const float *Wk, const float *init_state, float *W, float *Mn,
                             float *final_state, int BH, int T, int dk, int dv, int chunk,
                             gdr_dtype_t dtype, void *stream) {
    if (!dtype_ok(dtype)) return GDR_ERR_UNSUPPORTED;
    gdr_status_t st = check_staged(BH, T, dk, dv, chunk);
    if (st != GDR_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (BH == 0) return GDR_OK;
    if (T == 0) return from_cuda(gdr::launch_copy_state(init_state, final_state,
                                                        (int64_t)BH * dk * dv, s));
    if (!k || !gamma || !U || !Wk || !W) return GDR_ERR_INVALID_ARG;
    return from_cuda(gdr::launch_state(k, gamma, U, Wk, init_state, W, Mn, final_state, BH, T,
                                       dk, dv, chunk, elem_of(dtype), s));
}

gdr_status_t gdr_chunk_output(const void *q, const void *k, const float *gamma, const float *Mn,
                              const float *W, void *out, int BH, int T, int dk, int dv,
                              int chunk, gdr_dtype_t dtype, void *stream) {
    if (!dtype_ok(dtype)) return GDR_ERR_UNSUPPORTED;
    gdr_status_t st = check_staged(BH, T, dk, dv, chunk);
    if (st != GDR_OK) return st;
    if ((int64_t)BH * T == 0) return GDR_OK;
    if (!q || !k || !gamma || !Mn || !W || !out) return GDR_ERR_INVALID_ARG;
    return from_cuda(gdr::launch_output(q, k, gamma, Mn, W, out, BH, T, dk, dv, chunk,
                                        elem_of(dtype), static_cast<cudaStream_t>(stream)));
}

gdr_status_t gdr_chunk_fwd_varlen(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, float a_min, const float *init_state,
                                  void *out, float *final_state, const int *cu_seqlens, int S,
                                  int H, int total_T, int dk, int dv, int chunk,
                                  gdr_dtype_t dtype, void *stream) {
    if (S < 0 || H < 0 || total_T < 0) return GDR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return GDR_ERR_UNSUPPORTED;
    if (!a_min_ok(a_min)) return GDR_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv) || !chunk_ok(chunk)) return GDR_ERR_UNSUPPORTED;
    if (!range_ok(a_min, chunk)) return GDR_ERR_RANGE;
    const int64_t SH = (int64_t)S * H;
    if (SH > 0x7fffffff || (int64_t)total_T * H > ((int64_t)1 << 40)) return GDR_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (SH == 0) return GDR_OK;
    if (!cu_seqlens) return GDR_ERR_INVALID_ARG;
    if (total_T == 0) {   // every sequence is empty
        if (final_state == nullptr) return GDR_OK;
        return from_cuda(gdr::launch_copy_state(init_state, final_state, SH * dk * dv, s));
    }
    if (!q || !k || !v || !g || !beta || !out) return GDR_ERR_INVALID_ARG;
    if (!gdr::fused_supported(dk, dv, chunk, elem_of(dtype)))   // fp32 and the other shapes
        return from_cuda(gdr::launch_onepass(q, k, v, g, beta, a_min, init_state, out, final_state,
                                             (int)SH, 0, dk, dv, chunk, elem_of(dtype), s,
                                             cu_seqlens, H, total_T));
    return from_cuda(gdr::launch_fused_varlen(q, k, v, g, beta, a_min, init_state, out,
                                              final_state, cu_seqlens, S, H, total_T, s));
}

// ---- two-kernel path with a caller-owned workspace ----

size_t gdr_chunk_fwd_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                    gdr_dtype_t dtype) {
    if (B < 0 || H < 0 || T < 0 || !dtype_ok(dtype)) return 0;
    if (!dim_ok(dk) || !dim_ok(dv) || !chunk_ok(chunk)) return 0;
    const int64_t BH = (int64_t)B * H;
    if (BH == 0 || BH > 0x7fffffff || T == 0 || (int64_t)T * BH > ((int64_t)1 << 40)) return 0;
    if (gdr::fused_supported(dk, dv, chunk, elem_of(dtype)))   // tiles, then segment maps
        return gdr::prep_workspace_bytes((int)BH, T, nullptr, 0, 0) +
               gdr::segment_workspace_bytes((int)BH, gdr::segment_count((int)BH, T));
    return gdr::staged_scratch_bytes(BH, T, dk, dv, chunk);   // the staged kernels' scratch
}

size_t gdr_chunk_fwd_varlen_workspace_size(int S, int H, int total_T, int dk, int dv, int chunk,
                                           gdr_dtype_t dtype) {
    if (S < 0 || H < 0 || total_T < 0 || !dtype_ok(dtype)) return 0;
    if (!gdr::fused_supported(dk, dv, chunk, elem_of(dtype))) return 0;
    const int64_t SH = (int64_t)S * H;
    if (SH == 0 || SH > 0x7fffffff || total_T == 0) return 0;
    // only the sizes matter here; a non-null marker selects the packed layout
    static const int marker = 0;
    return gdr::prep_workspace_bytes((int)SH, 0, &marker, H, total_T);
}

}  // extern "C"

namespace {

gdr_status_t two_kernel_fwd(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float a_min, const float *init_state, void *out,
                            float *final_state, int BH, int T, void *workspace, void *saved,
                            cudaStream_t s, bool states_only = false);

gdr_status_t chunk_fwd_ws_impl(const void *q, const void *k, const void *v, const float *g,
                               const float *beta, float a_min, const float *init_state, void *out,
                               float *final_state, int B, int H, int T, int dk, int dv, int chunk,
                               gdr_dtype_t dtype, void *workspace, size_t workspace_bytes,
                               void *stream) {
    const size_t need = gdr_chunk_fwd_workspace_size(B, H, T, dk, dv, chunk, dtype);
    if (need == 0 || workspace == nullptr || workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(workspace) & 15))
        return chunk_fwd_impl(q, k, v, g, beta, a_min, init_state, out, final_state, B, H, T, dk,
                              dv, chunk, dtype, stream);
    if (!gdr::fused_supported(dk, dv, chunk, elem_of(dtype))) {
        // the four staged kernels (parallel WY/UT and output steps) on the workspace
        if (!range_ok(a_min, chunk)) return GDR_ERR_RANGE;
        if (!q || !k || !v || !g || !beta || !out) return GDR_ERR_INVALID_ARG;
        return from_cuda(gdr::launch_staged(q, k, v, g, beta, a_min, init_state, out, final_state,
                                            workspace, B * H, T, dk, dv, chunk, elem_of(dtype),
                                            static_cast<cudaStream_t>(stream)));
    }
    if (!range_ok(a_min, kTile)) return GDR_ERR_RANGE;
    if ((int64_t)T * B * H > ((int64_t)1 << 40)) return GDR_ERR_UNSUPPORTED;
    return two_kernel_fwd(q, k, v, g, beta, a_min, init_state, out, final_state, B * H, T,
                          workspace, nullptr, static_cast<cudaStream_t>(stream));
}

// The two-kernel path (dense, arguments checked): the preparation, the segment states when
// the sequence is cut into segments, the chain; saved != nullptr also writes the states and
// W tiles the saved-state backward reads.
gdr_status_t two_kernel_fwd(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float a_min, const float *init_state, void *out,
                            float *final_state, int BH, int T, void *workspace, void *saved,
                            cudaStream_t s, bool states_only) {
    if (!q || !k || !v || !g || !beta || !out) return GDR_ERR_INVALID_ARG;
    const int S = gdr::segment_count(BH, T);
    // training: the preparation also leaves T, P and the row scalars in the saved buffer
    uint8_t *sv = static_cast<uint8_t *>(saved);
    cudaError_t e = gdr::launch_prep(q, k, g, beta, a_min, workspace, BH, T, nullptr, 0, 0, s,
                                     sv ? sv + gdr::saved_tp_offset(BH, T) : nullptr,
                                     sv ? reinterpret_cast<float *>(sv + gdr::saved_sc_offset(BH, T))
                                        : nullptr);
    if (S <= 1) {
        if (e == cudaSuccess)
            e = gdr::launch_chain(q, k, v, g, beta, a_min, init_state, out, final_state, workspace,
                                  BH, T, nullptr, 0, 0, s, 1, nullptr, saved, states_only);
        return from_cuda(e);
    }
    // sequence segments: their maps and the scan, then every segment's chain at once
    float *seg_ws = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                              gdr::prep_workspace_bytes(BH, T, nullptr, 0, 0));
    if (e == cudaSuccess)
        e = gdr::launch_segment_states(k, v, g, beta, a_min, init_state, workspace, seg_ws, BH, T,
                                       S, s);
    if (e == cudaSuccess)
        e = gdr::launch_chain(q, k, v, g, beta, a_min, init_state, out, final_state, workspace, BH,
                              T, nullptr, 0, 0, s, S, gdr::segment_states(seg_ws, BH, S), saved,
                              states_only);
    return from_cuda(e);
}

}  // namespace

extern "C" {

gdr_status_t gdr_chunk_fwd_ws(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, float a_min, const float *init_state, void *out,
                              float *final_state, int B, int H, int T, int dk, int dv, int chunk,
                              gdr_dtype_t dtype, void *workspace, size_t workspace_bytes,
                              void *stream) {
    if (!a_min_ok(a_min)) return GDR_ERR_INVALID_ARG;
    return chunk_fwd_ws_impl(q, k, v, g, beta, a_min, init_state, out, final_state, B, H, T, dk,
                             dv, chunk, dtype, workspace, workspace_bytes, stream);
}

gdr_status_t gdr_chunk_fwd_ex(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, gdr_decay_t decay, float bound,
                              const float *init_state,
                              void *out, float *final_state, int B, int H, int T, int dk, int dv,
                              int chunk, gdr_dtype_t dtype, void *workspace, size_t workspace_bytes,
                              void *stream) {
    float d = 0.0f;
    if (!decay_param(decay, bound, &d)) return GDR_ERR_INVALID_ARG;
    return chunk_fwd_ws_impl(q, k, v, g, beta, d, init_state, out, final_state, B, H, T, dk, dv,
                             chunk, dtype, workspace, workspace_bytes, stream);
}

gdr_status_t gdr_chunk_fwd_varlen_ws(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, float a_min, const float *init_state,
                                     void *out, float *final_state, const int *cu_seqlens, int S,
                                     int H, int total_T, int dk, int dv, int chunk,
                                     gdr_dtype_t dtype, void *workspace, size_t workspace_bytes,
                                     void *stream) {
    const size_t need = gdr_chunk_fwd_varlen_workspace_size(S, H, total_T, dk, dv, chunk, dtype);
    if (need == 0 || workspace == nullptr || workspace_bytes < need)
        return gdr_chunk_fwd_varlen(q, k, v, g, beta, a_min, init_state, out, final_state,
                                    cu_seqlens, S, H, total_T, dk, dv, chunk, dtype, stream);
    if (!a_min_ok(a_min)) return GDR_ERR_INVALID_ARG;
    if (!range_ok(a_min, kTile)) return GDR_ERR_RANGE;
    if ((int64_t)total_T * H > ((int64_t)1 << 40)) return GDR_ERR_UNSUPPORTED;
    if (!cu_seqlens || !q || !k || !v || !g || !beta || !out) return GDR_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int SH = S * H;
    cudaError_t e = gdr::launch_prep(q, k, g, beta, a_min, workspace, SH, 0, cu_seqlens, H,
                                     total_T, s);
    if (e == cudaSuccess)
        e = gdr::launch_chain(q, k, v, g, beta, a_min, init_state, out, final_state, workspace, SH,
                              0, cu_seqlens, H, total_T, s);
    return from_cuda(e);
}

int gdr_chunk_fwd_ws_path(int B, int H, int T, int dk, int dv, int chunk, float a_min,
                          gdr_dtype_t dtype) {
    if (gdr_chunk_fwd_workspace_size(B, H, T, dk, dv, chunk, dtype) > 0 && a_min_ok(a_min)) {
        if (!gdr::fused_supported(dk, dv, chunk, elem_of(dtype)))
            return range_ok(a_min, chunk) ? 1 : -1;
        if (range_ok(a_min, kTile)) {
            const int S = gdr::segment_count(B * H, T);
            if (S > 1) return 7;
            return gdr::chain_split(B * H) == 2 ? 4 : 5;
        }
    }
    return gdr_chunk_fwd_path(B, H, T, dk, dv, chunk, a_min, dtype);
}

int gdr_chunk_fwd_kernels(int B, int H, int T, int dk, int dv, int chunk, float a_min,
                          gdr_dtype_t dtype) {
    if (B < 0 || H < 0 || T < 0 || !dtype_ok(dtype) || !a_min_ok(a_min)) return -1;
    if (!dim_ok(dk) || !dim_ok(dv) || !chunk_ok(chunk) || !range_ok(a_min, chunk)) return -1;
    if ((int64_t)B * H == 0) return 0;
    if (T == 0) return 0;  // a copy or memset, no kernel
    return 1;              // the fused tensor-core kernel or the one-pass CUDA-core kernel
}

int gdr_chunk_fwd_path(int B, int H, int T, int dk, int dv, int chunk, float a_min,
                       gdr_dtype_t dtype) {
    const int n = gdr_chunk_fwd_kernels(B, H, T, dk, dv, chunk, a_min, dtype);
    if (n <= 0) return n;
    const int64_t BH = (int64_t)B * H;
    if (BH > 0x7fffffff) return -1;
    if (!gdr::fused_supported(dk, dv, chunk, elem_of(dtype))) return 6;
    return gdr::fused_uses_pair((int)BH) ? 3 : 2;
}

// ---- host buffers in and out ----

namespace {
size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

// Byte offsets of the pieces of the device buffer of gdr_chunk_fwd_host: q, k, v,
// g, beta, init, out, final, workspace (each 256-byte aligned); returns the total.
size_t host_layout(int B, int H, int T, int dk, int dv, int chunk, gdr_dtype_t dtype,
                   size_t off[9]) {
    const size_t es = dtype == GDR_DTYPE_F32 ? 4 : 2;
    const size_t bht = (size_t)B * H * T, bh = (size_t)B * H;
    const size_t sizes[9] = {bht * dk * es, bht * dk * es, bht * dv * es, bht * 4, bht * 4,
                             bh * dk * dv * 4, bht * dv * es, bh * dk * dv * 4,
                             gdr_chunk_fwd_workspace_size(B, H, T, dk, dv, chunk, dtype)};
    size_t at = 0;
    for (int i = 0; i < 9; ++i) {
        off[i] = at;
        at += align256(sizes[i]);
    }
    return at;
}
}  // namespace

size_t gdr_chunk_fwd_host_buffer_size(int B, int H, int T, int dk, int dv, int chunk,
                                      gdr_dtype_t dtype) {
    if (B < 0 || H < 0 || T < 0 || !dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv) || !chunk_ok(chunk))
        return 0;
    if ((int64_t)B * H > 0x7fffffff || (int64_t)T * B * H > ((int64_t)1 << 40)) return 0;
    size_t off[9];
    return host_layout(B, H, T, dk, dv, chunk, dtype, off);
}

gdr_status_t gdr_chunk_fwd_host(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float a_min, const float *init_state,
                                void *out, float *final_state, int B, int H, int T, int dk, int dv,
                                int chunk, gdr_dtype_t dtype, void *device_buffer,
                                size_t device_bytes, void *stream) {
    if (B < 0 || H < 0 || T < 0) return GDR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return GDR_ERR_UNSUPPORTED;
    if (!a_min_ok(a_min)) return GDR_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv) || !chunk_ok(chunk)) return GDR_ERR_UNSUPPORTED;
    const size_t need = gdr_chunk_fwd_host_buffer_size(B, H, T, dk, dv, chunk, dtype);
    if (need == 0 && (int64_t)B * H * T > 0) return GDR_ERR_UNSUPPORTED;
    if ((int64_t)B * H == 0) return GDR_OK;
    if (!device_buffer || device_bytes < need || (reinterpret_cast<uintptr_t>(device_buffer) & 255))
        return GDR_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDR_ERR_INVALID_ARG;
    // the chunk's range rule of whichever path the call takes, before anything is enqueued
    const bool two = gdr::fused_supported(dk, dv, chunk, elem_of(dtype));
    if (!range_ok(a_min, two ? kTile : chunk)) return GDR_ERR_RANGE;
    size_t off[9];
    host_layout(B, H, T, dk, dv, chunk, dtype, off);
    uint8_t *base = static_cast<uint8_t *>(device_buffer);
    const size_t es = dtype == GDR_DTYPE_F32 ? 4 : 2;
    const size_t bht = (size_t)B * H * T, st = (size_t)B * H * dk * dv * 4;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const void *src[6] = {q, k, v, g, beta, init_state};
    const size_t bytes[6] = {bht * dk * es, bht * dk * es, bht * dv * es, bht * 4, bht * 4, st};
    for (int i = 0; i < 6; ++i) {
        if (!src[i] || bytes[i] == 0) continue;
        if (cudaMemcpyAsync(base + off[i], src[i], bytes[i], cudaMemcpyHostToDevice, s) != cudaSuccess)
            return GDR_ERR_CUDA;
    }
    gdr_status_t rc = chunk_fwd_ws_impl(
        base + off[0], base + off[1], base + off[2], reinterpret_cast<float *>(base + off[3]),
        reinterpret_cast<float *>(base + off[4]),
        a_min, init_state ? reinterpret_cast<float *>(base + off[5]) : nullptr, base + off[6],
        final_state ? reinterpret_cast<float *>(base + off[7]) : nullptr, B, H, T, dk, dv, chunk,
        dtype, base + off[8], off[8] < need ? need - off[8] : 0, stream);
    if (rc != GDR_OK) return rc;
    if (T > 0 && cudaMemcpyAsync(out, base + off[6], bht * dv * es, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GDR_ERR_CUDA;
    if (final_state &&
        cudaMemcpyAsync(final_state, base + off[7], st, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GDR_ERR_CUDA;
    return GDR_OK;
}

// ---- backward ----

size_t gdr_chunk_bwd_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                    gdr_dtype_t dtype) {
    if (B < 0 || H < 0 || T < 0 || !dtype_ok(dtype) || !gdr::bwd_supported(dk, dv, chunk)) return 0;
    const int64_t BH = (int64_t)B * H;
    if (BH == 0 || BH > 0x7fffffff || T == 0) return 0;
    return gdr::bwd_workspace_bytes((int)BH, T, dk, dv, chunk);
}

gdr_status_t gdr_chunk_bwd(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, gdr_decay_t decay, float bound,
                           const float *init_state, const void *d_out, const float *d_final,
                           void *d_q, void *d_k, void *d_v, float *d_g, float *d_beta,
                           float *d_init, int B, int H, int T, int dk, int dv, int chunk,
                           gdr_dtype_t dtype, void *workspace, size_t workspace_bytes,
                           void *stream) {
    float d = 0.0f;
    if (B < 0 || H < 0 || T < 0) return GDR_ERR_INVALID_ARG;
    if (!decay_param(decay, bound, &d)) return GDR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return GDR_ERR_UNSUPPORTED;
    if (!gdr::bwd_supported(dk, dv, chunk)) return GDR_ERR_UNSUPPORTED;
    if (!range_ok(d, chunk)) return GDR_ERR_RANGE;
    const int64_t BH = (int64_t)B * H;
    if (BH > 0x7fffffff || (int64_t)T * BH > ((int64_t)1 << 40)) return GDR_ERR_UNSUPPORTED;
    if (BH == 0) return GDR_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > 0) {
        if (!q || !k || !v || !g || !beta || !d_out || !d_q || !d_k || !d_v || !d_g || !d_beta)
            return GDR_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
             reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(d_out)) & 15)
            return GDR_ERR_INVALID_ARG;   // the kernels read them in 16-byte pieces
        if (!workspace ||
            workspace_bytes < gdr::bwd_workspace_bytes((int)BH, T, dk, dv, chunk) ||
            (reinterpret_cast<uintptr_t>(workspace) & 15))
            return GDR_ERR_INVALID_ARG;
    }
    // bf16, d = 128, chunk 64 (the default per-chunk kernel): the forward's intermediates come
    // from the training forward's kernels, run into the part of the workspace the saved-state
    // backward leaves free (its chain, without the output products, keeps every chunk's state
    // and W tile, its preparation T, P and the row scalars), then the saved-state backward.  The forward's chain recomputes the
    // states faster than the tiles kernel and the forward-state pass of the other path.
    if (T > 0 && gdr::opt_bwd_variant() == 0 && range_ok(d, kTile) &&
        gdr::bwd_saved_shape(dk, dv, chunk, elem_of(dtype), d_q, d_k, d_v)) {
        size_t off = 0, room = 0;
        gdr::bwd_free_region((int)BH, T, dk, dv, chunk, &off, &room);
        auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
        const size_t sv = up(gdr::saved_bytes(BH, T)), ob = up((size_t)BH * T * dv * 2);
        const size_t fw = gdr_chunk_fwd_workspace_size(B, H, T, dk, dv, chunk, dtype);
        if (fw > 0 && sv + ob + fw <= room) {
            uint8_t *base = static_cast<uint8_t *>(workspace) + off;
            // (the forward's chain without its output products: only the states and W tiles)
            const gdr_status_t st = two_kernel_fwd(q, k, v, g, beta, d, init_state, base + sv, nullptr,
                                                   (int)BH, T, base + sv + ob, base, s, true);
            if (st != GDR_OK) return st;
            return from_cuda(gdr::launch_bwd(q, k, v, g, beta, d, init_state, d_out, d_final, d_q, d_k,
                                             d_v, d_g, d_beta, d_init, (int)BH, T, dk, dv, chunk,
                                             workspace, elem_of(dtype), s, base));
        }
    }
    return from_cuda(gdr::launch_bwd(q, k, v, g, beta, d, init_state, d_out, d_final, d_q, d_k,
                                     d_v, d_g, d_beta, d_init, (int)BH, T, dk, dv, chunk,
                                     workspace, elem_of(dtype), s));
}

// ---- training: the forward saves its chunk states, the backward reads them ----

size_t gdr_chunk_saved_size(int B, int H, int T, int dk, int dv, int chunk, gdr_dtype_t dtype) {
    if (B < 0 || H < 0 || T <= 0 || !dtype_ok(dtype)) return 0;
    if (!gdr::fused_supported(dk, dv, chunk, elem_of(dtype))) return 0;
    const int64_t BH = (int64_t)B * H;
    if (BH == 0 || BH > 0x7fffffff || (int64_t)T * BH > ((int64_t)1 << 40)) return 0;
    return gdr::saved_bytes(BH, T);
}

gdr_status_t gdr_chunk_fwd_train(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, gdr_decay_t decay, float bound,
                                 const float *init_state, void *out, float *final_state, int B,
                                 int H, int T, int dk, int dv, int chunk, gdr_dtype_t dtype,
                                 void *workspace, size_t workspace_bytes, void *saved,
                                 size_t saved_bytes, void *stream) {
    float d = 0.0f;
    if (B < 0 || H < 0 || T < 0) return GDR_ERR_INVALID_ARG;
    if (!decay_param(decay, bound, &d)) return GDR_ERR_INVALID_ARG;
    if (!dtype_ok(dtype) || !gdr::fused_supported(dk, dv, chunk, elem_of(dtype)))
        return GDR_ERR_UNSUPPORTED;
    const int64_t BH = (int64_t)B * H;
    if (BH > 0x7fffffff || (int64_t)T * BH > ((int64_t)1 << 40)) return GDR_ERR_UNSUPPORTED;
    if (BH == 0 || T == 0)   // nothing to save: the final state is the initial one
        return chunk_fwd_impl(q, k, v, g, beta, d, init_state, out, final_state, B, H, T, dk, dv,
                              chunk, dtype, stream);
    if (!range_ok(d, kTile)) return GDR_ERR_RANGE;
    const size_t need = gdr_chunk_fwd_workspace_size(B, H, T, dk, dv, chunk, dtype);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15))
        return GDR_ERR_INVALID_ARG;
    if (!saved || saved_bytes < gdr::saved_bytes(BH, T) ||
        (reinterpret_cast<uintptr_t>(saved) & 15))
        return GDR_ERR_INVALID_ARG;
    return two_kernel_fwd(q, k, v, g, beta, d, init_state, out, final_state, (int)BH, T,
                          workspace, saved, static_cast<cudaStream_t>(stream));
}

gdr_status_t gdr_chunk_bwd_saved(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, gdr_decay_t decay, float bound,
                                 const float *init_state, const void *d_out, const float *d_final,
                                 void *d_q, void *d_k, void *d_v, float *d_g, float *d_beta,
                                 float *d_init, int B, int H, int T, int dk, int dv, int chunk,
                                 gdr_dtype_t dtype, const void *saved, size_t saved_bytes,
                                 void *workspace, size_t workspace_bytes, void *stream) {
    if (!dtype_ok(dtype) || !gdr::fused_supported(dk, dv, chunk, elem_of(dtype)))
        return GDR_ERR_UNSUPPORTED;
    const int64_t BH = (int64_t)B * H;
    if (B < 0 || H < 0 || T < 0 || BH == 0 || T == 0)   // no chunk: nothing was saved
        return gdr_chunk_bwd(q, k, v, g, beta, decay, bound, init_state, d_out, d_final, d_q, d_k,
                             d_v, d_g, d_beta, d_init, B, H, T, dk, dv, chunk, dtype, workspace,
                             workspace_bytes, stream);
    float d = 0.0f;
    if (!decay_param(decay, bound, &d)) return GDR_ERR_INVALID_ARG;
    if (!range_ok(d, chunk)) return GDR_ERR_RANGE;
    if (BH > 0x7fffffff || (int64_t)T * BH > ((int64_t)1 << 40)) return GDR_ERR_UNSUPPORTED;
    if (!q || !k || !v || !g || !beta || !d_out || !d_q || !d_k || !d_v || !d_g || !d_beta)
        return GDR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(d_out) |
         reinterpret_cast<uintptr_t>(d_q) | reinterpret_cast<uintptr_t>(d_k) |
         reinterpret_cast<uintptr_t>(d_v) | reinterpret_cast<uintptr_t>(saved)) & 15)
        return GDR_ERR_INVALID_ARG;
    if (!saved || saved_bytes < gdr::saved_bytes(BH, T)) return GDR_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < gdr::bwd_workspace_bytes((int)BH, T, dk, dv, chunk) ||
        (reinterpret_cast<uintptr_t>(workspace) & 15))
        return GDR_ERR_INVALID_ARG;
    return from_cuda(gdr::launch_bwd(q, k, v, g, beta, d, init_state, d_out, d_final, d_q, d_k,
                                     d_v, d_g, d_beta, d_init, (int)BH, T, dk, dv, chunk,
                                     workspace, elem_of(dtype), static_cast<cudaStream_t>(stream),
                                     saved));
}

// ---- gated multi-head latent attention, one decode step ----

size_t gdr_mla_decode_workspace_size(int N, int H, int Lmax, int dc, int dh) {
    if (N <= 0 || H <= 0 || Lmax <= 0 || !gdr::mla_supported(H, dc, dh)) return 0;
    if ((int64_t)N * H > 0x7fffffff || (int64_t)N * Lmax > ((int64_t)1 << 40)) return 0;
    return gdr::mla_workspace_bytes(N, H, Lmax);
}

gdr_status_t gdr_mla_decode(const void *q_abs, const void *ckv, const int *seqlens,
                            const void *w_uv, const float *gate, float scale, void *out, int N,
                            int H, int Lmax, int dc, int dh, void *workspace,
                            size_t workspace_bytes, void *stream) {
    if (N < 0 || H < 0 || Lmax < 0 || dc < 0 || dh < 0) return GDR_ERR_INVALID_ARG;
    if (!(scale > 0.0f) || !std::isfinite(scale)) return GDR_ERR_INVALID_ARG;
    if ((int64_t)N * H == 0) return GDR_OK;
    if (Lmax == 0 || !gdr::mla_supported(H, dc, dh)) return GDR_ERR_UNSUPPORTED;
    if ((int64_t)N * H > 0x7fffffff || (int64_t)N * Lmax > ((int64_t)1 << 40))
        return GDR_ERR_UNSUPPORTED;
    if (!q_abs || !ckv || !seqlens || !w_uv || !gate || !out) return GDR_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q_abs) | reinterpret_cast<uintptr_t>(ckv) |
         reinterpret_cast<uintptr_t>(w_uv)) & 15)
        return GDR_ERR_INVALID_ARG;   // TMA and 16-byte loads
    const size_t need = gdr::mla_workspace_bytes(N, H, Lmax);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15))
        return GDR_ERR_INVALID_ARG;
    return from_cuda(gdr::launch_mla_decode(q_abs, ckv, seqlens, w_uv, gate, scale, out, N, H, Lmax,
                                            dh, workspace, static_cast<cudaStream_t>(stream)));
}

gdr_status_t gdr_last_device_error(void *stream) {
    unsigned word = 0;
    cudaError_t e = gdr::read_and_clear_device_error(static_cast<cudaStream_t>(stream), &word);
    if (e != cudaSuccess) return GDR_ERR_CUDA;
    if (word & gdr::kDevErrTimeout) return GDR_ERR_TIMEOUT;
    return GDR_OK;
}

const char *gdr_status_string(gdr_status_t status) {
    switch (status) {
        case GDR_OK: return "ok";
        case GDR_ERR_INVALID_ARG: return "invalid argument";
        case GDR_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case GDR_ERR_RANGE:
            return "the decay over a chunk (a 16-token tile on the workspace path) falls below e^-80";
        case GDR_ERR_CUDA: return "CUDA runtime error";
        case GDR_ERR_TIMEOUT: return "device-side bounded wait timed out";
    }
    return "unknown status";
}

const char *gdr_version(void) { return "gdr 0.1.0 sm_103a"; }

}  // extern "C"
