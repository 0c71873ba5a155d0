// gdr_decode.cu -- single-token decode of the gated delta rule.
//
// Each (sequence, head) carries a fixed-size fp32 state M = S^T [dk][dv];
// one step reads it once and writes it once, which is the whole point of the
// recurrent form at inference time: the cost per token does not depend on
// how long the context already is ("Trillion-Parameter MoE Multimodal LLMs:
// How to Evaluate the New Generation", section 2.1; "How to Think About
// Trillion-Parameter Sparse Multimodal LLMs", section 2.2).
//
// Per (n, h), with alpha = a_min + (1 - a_min) sigmoid(g):
//   p = S k, r = S q          (one pass over the state, two reductions)
//   u = v - alpha p
//   o = alpha r + beta (q . k) u          (= S_new q)
//   M <- alpha M + k (beta u)^T           (in place)
//
// The kernel is a pure HBM stream: 64 KB of state per (n, h) at d = 128,
// read with evict-first 16-byte loads, held in registers across the two
// reductions, and written back with streaming stores.

#include "gdr_internal.h"
#include "gdr_math.cuh"

#include <cuda_bf16.h>

#include <cstdint>

namespace gdr {
namespace {

__device__ __forceinline__ float ld_elem(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_elem(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_elem(__nv_bfloat16 *p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}


// dk = dv = 128: 256 threads; warp w owns state rows 16w..16w+15, lane l owns
// columns 4l..4l+3 (one float4 per row), so every warp load is one fully
// coalesced 512-byte row.
template <typename TE>
__global__ void __launch_bounds__(256, 2)
decode128_kernel(const TE *__restrict__ q, const TE *__restrict__ k, const TE *__restrict__ v,
                 const float *__restrict__ g, const float *__restrict__ beta, float a_min,
                 float *__restrict__ state, TE *__restrict__ out) {
    constexpr int D = 128, RW = 16;
    __shared__ float qs[D], ks[D];
    __shared__ __align__(16) float red_p[8][D];
    __shared__ __align__(16) float red_r[8][D];
    __shared__ __align__(16) float bu[D];
    __shared__ float qk_s;
    const int64_t nh = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    float4 *M = reinterpret_cast<float4 *>(state + nh * D * D);

    float4 m[RW];
#pragma unroll
    for (int e = 0; e < RW; ++e) m[e] = __ldcs(M + (w * RW + e) * (D / 4) + lane);

    if (tid < D) {
        qs[tid] = ld_elem(q, nh * D + tid);
        ks[tid] = ld_elem(k, nh * D + tid);
    }
    const float a = decay_alpha(g[nh], a_min);
    const float b = beta[nh];
    __syncthreads();

    float4 p = make_float4(0.f, 0.f, 0.f, 0.f), r = p;
#pragma unroll
    for (int e = 0; e < RW; ++e) {
        const float ki = ks[w * RW + e], qi = qs[w * RW + e];
        p.x = fmaf(m[e].x, ki, p.x); p.y = fmaf(m[e].y, ki, p.y);
        p.z = fmaf(m[e].z, ki, p.z); p.w = fmaf(m[e].w, ki, p.w);
        r.x = fmaf(m[e].x, qi, r.x); r.y = fmaf(m[e].y, qi, r.y);
        r.z = fmaf(m[e].z, qi, r.z); r.w = fmaf(m[e].w, qi, r.w);
    }
    reinterpret_cast<float4 *>(red_p[w])[lane] = p;
    reinterpret_cast<float4 *>(red_r[w])[lane] = r;
    if (w == 0) {
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < D / 32; ++e) d = fmaf(qs[lane + 32 * e], ks[lane + 32 * e], d);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        if (lane == 0) qk_s = d;
    }
    __syncthreads();
    if (tid < D) {
        float pj = 0.f, rj = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) {
            pj += red_p[ww][tid];
            rj += red_r[ww][tid];
        }
        const float uj = ld_elem(v, nh * D + tid) - a * pj;
        bu[tid] = b * uj;
        st_elem(out, nh * D + tid, fmaf(a, rj, b * qk_s * uj));
    }
    __syncthreads();
    const float4 u4 = reinterpret_cast<const float4 *>(bu)[lane];
#pragma unroll
    for (int e = 0; e < RW; ++e) {
        const float ki = ks[w * RW + e];
        float4 x = m[e];
        x.x = fmaf(a, x.x, ki * u4.x); x.y = fmaf(a, x.y, ki * u4.y);
        x.z = fmaf(a, x.z, ki * u4.z); x.w = fmaf(a, x.w, ki * u4.w);
        __stcs(M + (w * RW + e) * (D / 4) + lane, x);
    }
}

// Any dk, dv <= 128: thread j owns column j; two passes over the state.
template <typename TE>
__global__ void __launch_bounds__(128)
decode_generic_kernel(const TE *__restrict__ q, const TE *__restrict__ k,
                      const TE *__restrict__ v, const float *__restrict__ g,
                      const float *__restrict__ beta, float a_min, float *__restrict__ state,
                      TE *__restrict__ out, int dk, int dv) {
    __shared__ float qs[128], ks[128], part[4];
    const int64_t nh = blockIdx.x;
    const int tid = threadIdx.x;
    float *M = state + nh * dk * dv;
    float d = 0.f;
    if (tid < dk) {
        qs[tid] = ld_elem(q, nh * dk + tid);
        ks[tid] = ld_elem(k, nh * dk + tid);
        d = qs[tid] * ks[tid];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if ((tid & 31) == 0) part[tid >> 5] = d;
    __syncthreads();
    const float qk = part[0] + part[1] + part[2] + part[3];
    const float a = decay_alpha(g[nh], a_min);
    const float b = beta[nh];
    if (tid >= dv) return;
    const int j = tid;
    float pj = 0.f, rj = 0.f;
    for (int i = 0; i < dk; ++i) {
        const float mij = M[(int64_t)i * dv + j];
        pj = fmaf(mij, ks[i], pj);
        rj = fmaf(mij, qs[i], rj);
    }
    const float uj = ld_elem(v, nh * dv + j) - a * pj;
    st_elem(out, nh * dv + j, fmaf(a, rj, b * qk * uj));
    const float buj = b * uj;
    for (int i = 0; i < dk; ++i) {
        float *pm = M + (int64_t)i * dv + j;
        *pm = fmaf(a, *pm, ks[i] * buj);
    }
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float a_min, float *state, void *out, int N,
                          int H, int dk, int dv, Elem e, cudaStream_t s) {
    const int64_t NH = (int64_t)N * H;
    if (NH == 0) return cudaSuccess;
    if (NH > 0x7fffffff) return cudaErrorInvalidValue;
    // The streaming kernel moves the state in 16-byte vectors: it needs a
    // 16-byte aligned state (every (n, h) block is then aligned too).
    const bool fast = dk == 128 && dv == 128 && (reinterpret_cast<uintptr_t>(state) & 15) == 0;
    if (e == Elem::F32) {
        if (fast)
            decode128_kernel<float><<<(unsigned)NH, 256, 0, s>>>(
                (const float *)q, (const float *)k, (const float *)v, g, beta, a_min, state,
                (float *)out);
        else
            decode_generic_kernel<float><<<(unsigned)NH, 128, 0, s>>>(
                (const float *)q, (const float *)k, (const float *)v, g, beta, a_min, state,
                (float *)out, dk, dv);
    } else {
        using B16 = __nv_bfloat16;
        if (fast)
            decode128_kernel<B16><<<(unsigned)NH, 256, 0, s>>>(
                (const B16 *)q, (const B16 *)k, (const B16 *)v, g, beta, a_min, state,
                (B16 *)out);
        else
            decode_generic_kernel<B16><<<(unsigned)NH, 128, 0, s>>>(
                (const B16 *)q, (const B16 *)k, (const B16 *)v, g, beta, a_min, state,
                (B16 *)out, dk, dv);
    }
    return cudaGetLastError();
}

}  // namespace gdr
