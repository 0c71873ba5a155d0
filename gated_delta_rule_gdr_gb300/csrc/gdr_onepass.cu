// gdr_onepass.cu -- the chunked prefill in one launch on CUDA cores, with no
// scratch memory: the path of gdr_chunk_fwd for fp32 inputs and for every
// shape the tensor-core kernels do not take.
//
// One CTA owns DS value columns J of one (sequence, head) and walks its chunks
// in order.  The recurrence never mixes value columns, so the CTAs of a head
// share nothing; each recomputes the chunk's state-independent part (decay,
// A, T = (I + A)^-1 and the causal tile P) for itself.  Per chunk, rows r, s:
//
//   gamma_r = prod_{s <= r} alpha_s     (inside the chunk; gamma_C the last row)
//   A = strict_lower(diag(beta gamma) K (diag(1/gamma) K)^T),  T = (I + A)^-1
//   P = lower_incl(diag(gamma) Q (diag(1/gamma) K)^T)
//   E = V_J - diag(gamma) K M_J              (what the carried state mispredicts)
//   W = T diag(beta) E                       (= U - Wk M_J of the WY/UT form)
//   O_J = diag(gamma) Q M_J + P W
//   M_J <- gamma_C M_J + (diag(gamma_C / gamma) K)^T W
//
// (the intra-tile causal part plus the inter-tile recurrent state of "What a
// Trillion-Parameter MoE Model Reveals About the Next Stage of LLM Scaling",
// sections 3.1-3.3, with Gamma = exp(cumsum(log-decay)) of "Architecture
// Evolution and Training Engineering for Trillion-Scale Sparse Multimodal
// Models", section 3.2).  fp32 arithmetic throughout; the exponentials are the
// full-precision functions, so fp32 inputs meet a 1e-5 relative tolerance.
// The range rule (chunk * |worst log-decay| <= 80) keeps 1/gamma finite.

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

constexpr int kThreads = 256;

// Shared-memory floats of one CTA.
__host__ __device__ inline size_t onepass_smem_floats(int dk, int C, int DS) {
    return (size_t)dk * DS                   // M_J
           + 2 * (size_t)C * (dk + 1)        // K, Q (rows padded by one)
           + 3 * (size_t)C * DS              // V_J, E, W
           + 3 * (size_t)C * (C + 1)         // A, T, P
           + 4 * (size_t)C;                  // gamma, 1/gamma, beta, gamma_C / gamma
}

// Packed sequences (cu_seqlens != nullptr): q, k, v, out [total_T][H][d], g, beta
// [total_T][H], states [S][H][dk][dv]; blockIdx.y = s H + h.  Offsets are clamped
// into [0, total_T], so a malformed array cannot take a CTA out of the tensors.
template <typename TE>
__global__ void __launch_bounds__(kThreads)
onepass_kernel(const TE *__restrict__ q, const TE *__restrict__ k, const TE *__restrict__ v,
               const float *__restrict__ g, const float *__restrict__ beta, float d,
               const float *init, TE *__restrict__ out, float *final_state, int T, int dk,
               int dv, int C, int DS, const int *__restrict__ cu_seqlens, int H, int total_T) {
    extern __shared__ float sm[];
    const int j0 = blockIdx.x * DS;
    const int64_t bh = blockIdx.y;
    // token t of this (sequence, head): row (tbase + t * tstride) of q, k, v, out and
    // element (tbase + t * tstride) of g, beta
    int64_t tbase = bh * T, tstride = 1;
    if (cu_seqlens) {
        const int sq = (int)(bh / H), h = (int)(bh % H);
        const int t0 = min(max(cu_seqlens[sq], 0), total_T);
        const int t1 = min(max(cu_seqlens[sq + 1], t0), total_T);
        T = t1 - t0;
        tbase = (int64_t)t0 * H + h;
        tstride = H;
    }
    const int tid = threadIdx.x;
    const int ldk = dk + 1, ldc = C + 1;
    float *Ms = sm;                       // [dk][DS]
    float *Ks = Ms + (size_t)dk * DS;     // [C][dk+1]
    float *Qs = Ks + (size_t)C * ldk;     // [C][dk+1]
    float *Vs = Qs + (size_t)C * ldk;     // [C][DS]
    float *Es = Vs + (size_t)C * DS;      // [C][DS]
    float *Ws = Es + (size_t)C * DS;      // [C][DS]
    float *As = Ws + (size_t)C * DS;      // [C][C+1]
    float *Ts = As + (size_t)C * ldc;     // [C][C+1]
    float *Ps = Ts + (size_t)C * ldc;     // [C][C+1]
    float *gs = Ps + (size_t)C * ldc;     // [C] gamma
    float *ig = gs + C;                   // [C] 1/gamma
    float *bs = ig + C;                   // [C] beta
    float *sc = bs + C;                   // [C] gamma_C / gamma
    __shared__ float s_gC;

    for (int x = tid; x < dk * DS; x += kThreads) {
        const int i = x / DS, j = x % DS;
        Ms[x] = init ? init[(bh * dk + i) * dv + j0 + j] : 0.f;
    }
    const int NC = (T + C - 1) / C;
    for (int n = 0; n < NC; ++n) {
        const int t0 = n * C, c = min(C, T - t0);
        auto row = [&](int r) { return tbase + (int64_t)(t0 + r) * tstride; };   // token t0 + r
        __syncthreads();   // the previous chunk is done with every buffer
        for (int x = tid; x < c * dk; x += kThreads) {
            const int r = x / dk, i = x % dk;
            Ks[r * ldk + i] = ld_elem(k, row(r) * dk + i);
            Qs[r * ldk + i] = ld_elem(q, row(r) * dk + i);
        }
        for (int x = tid; x < c * DS; x += kThreads) {
            const int r = x / DS, j = x % DS;
            Vs[x] = ld_elem(v, row(r) * dv + j0 + j);
        }
        if (tid < 32) {
            // chunk-local inclusive scan of log alpha; lane l owns rows l, l + 32
            const int lane = tid;
            float la[2], incl[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = lane + 32 * e;
                la[e] = (r < c) ? log_alpha(g[row(r)], d) : 0.f;
                incl[e] = la[e];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, incl[e], off);
                    if (lane >= off) incl[e] += y;
                }
            }
            incl[1] += __shfl_sync(0xffffffffu, incl[0], 31);   // rows 32.. follow rows 0..31
            const float bC = __shfl_sync(0xffffffffu, incl[(c - 1) >> 5], (c - 1) & 31);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = lane + 32 * e;
                if (r < c) {
                    gs[r] = expf(incl[e]);
                    ig[r] = expf(-incl[e]);
                    bs[r] = beta[row(r)];
                    sc[r] = expf(bC - incl[e]);
                }
            }
            if (lane == 0) s_gC = expf(bC);
        }
        __syncthreads();

        // A (s < r) and P (s <= r): the chunk's dot products of length dk
        for (int x = tid; x < c * c; x += kThreads) {
            const int r = x / c, s = x % c;
            float a = 0.f, p = 0.f;
            if (s <= r) {
                float dkk = 0.f, dqk = 0.f;
                for (int i = 0; i < dk; ++i) {
                    const float ks = Ks[s * ldk + i];
                    dkk = fmaf(Ks[r * ldk + i], ks, dkk);
                    dqk = fmaf(Qs[r * ldk + i], ks, dqk);
                }
                p = gs[r] * dqk * ig[s];
                if (s < r) a = (bs[r] * gs[r]) * dkk * ig[s];
            }
            As[r * ldc + s] = a;
            Ps[r * ldc + s] = p;
        }
        __syncthreads();

        // T = (I + A)^-1: thread s computes column s top-down,
        // T[r][s] = -sum_{m = s}^{r - 1} A[r][m] T[m][s], T[s][s] = 1
        if (tid < c) {
            const int s = tid;
            for (int r = 0; r < s; ++r) Ts[r * ldc + s] = 0.f;
            Ts[s * ldc + s] = 1.f;
            for (int r = s + 1; r < c; ++r) {
                float acc = 0.f;
                for (int m = s; m < r; ++m) acc = fmaf(As[r * ldc + m], Ts[m * ldc + s], acc);
                Ts[r * ldc + s] = -acc;
            }
        }
        // E = V_J - diag(gamma) K M_J (independent of T)
        for (int x = tid; x < c * DS; x += kThreads) {
            const int r = x / DS, j = x % DS;
            float acc = 0.f;
            for (int i = 0; i < dk; ++i) acc = fmaf(Ks[r * ldk + i], Ms[i * DS + j], acc);
            Es[x] = fmaf(-gs[r], acc, Vs[x]);
        }
        __syncthreads();

        // W = T diag(beta) E
        for (int x = tid; x < c * DS; x += kThreads) {
            const int r = x / DS, j = x % DS;
            float acc = 0.f;
            for (int s = 0; s <= r; ++s) acc = fmaf(Ts[r * ldc + s] * bs[s], Es[s * DS + j], acc);
            Ws[x] = acc;
        }
        __syncthreads();

        // O_J = diag(gamma) Q M_J + P W  (reads M_J before the update below)
        for (int x = tid; x < c * DS; x += kThreads) {
            const int r = x / DS, j = x % DS;
            float qm = 0.f;
            for (int i = 0; i < dk; ++i) qm = fmaf(Qs[r * ldk + i], Ms[i * DS + j], qm);
            float acc = gs[r] * qm;
            for (int s = 0; s <= r; ++s) acc = fmaf(Ps[r * ldc + s], Ws[s * DS + j], acc);
            st_elem(out, row(r) * dv + j0 + j, acc);
        }
        __syncthreads();

        // M_J <- gamma_C M_J + (diag(gamma_C / gamma) K)^T W
        const float gC = s_gC;
        for (int x = tid; x < dk * DS; x += kThreads) {
            const int i = x / DS, j = x % DS;
            float acc = 0.f;
            for (int r = 0; r < c; ++r) acc = fmaf(sc[r] * Ks[r * ldk + i], Ws[r * DS + j], acc);
            Ms[x] = fmaf(gC, Ms[x], acc);
        }
    }
    __syncthreads();
    if (final_state) {
        for (int x = tid; x < dk * DS; x += kThreads) {
            const int i = x / DS, j = x % DS;
            final_state[(bh * dk + i) * dv + j0 + j] = Ms[x];
        }
    }
}

}  // namespace

cudaError_t launch_onepass(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float d, const float *init, void *out,
                           float *final_state, int BH, int T, int dk, int dv, int C, Elem e,
                           cudaStream_t s, const int *cu_seqlens, int H, int total_T) {
    if (BH == 0 || (cu_seqlens ? total_T : T) == 0) return cudaSuccess;
    if (C > 64) return cudaErrorInvalidValue;   // the decay scan covers two rows per lane
    const int DS = dv < 32 ? dv : 32;
    const size_t smem = sizeof(float) * onepass_smem_floats(dk, C, DS);
    dim3 grid((unsigned)(dv / DS), (unsigned)BH);
    cudaError_t err;
    if (e == Elem::F32) {
        if ((err = cudaFuncSetAttribute(onepass_kernel<float>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem)) != cudaSuccess)
            return err;
        onepass_kernel<float><<<grid, kThreads, smem, s>>>(
            (const float *)q, (const float *)k, (const float *)v, g, beta, d, init, (float *)out,
            final_state, T, dk, dv, C, DS, cu_seqlens, H, total_T);
    } else {
        if ((err = cudaFuncSetAttribute(onepass_kernel<__nv_bfloat16>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem)) != cudaSuccess)
            return err;
        onepass_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(
            (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, g,
            beta, d, init, (__nv_bfloat16 *)out, final_state, T, dk, dv, C, DS, cu_seqlens, H,
            total_T);
    }
    return cudaGetLastError();
}

}  // namespace gdr
