// gdr_staged.cu -- the chunked form of the gated delta rule as four plain
// CUDA-core kernels: cumulative decay, intra-chunk WY/UT transform, the
// sequential inter-chunk state pass and the chunk output.  fp32 arithmetic
// throughout (inputs may be bf16; they are widened on load).
//
// This is the path for fp32 inputs (whose tolerance, 1e-5 relative, rules
// out bf16/tf32 tensor-core operands) and for shapes the fused tensor-core
// kernel does not cover.  Each step is also exported on its own through the
// C ABI so that it can be checked against the chunked reference algebra.
//
// The chunked form follows "What a Trillion-Parameter MoE Model Reveals
// About the Next Stage of LLM Scaling", section 3.1 (intra-tile causal part,
// inter-tile recurrent state) and "Architecture Evolution and Training
// Engineering for Trillion-Scale Sparse Multimodal Models", section 3.2
// (Gamma = exp(cumsum(log-decay)); every causal tile scaled by 1/Gamma).

#include "gdr_internal.h"
#include "gdr_math.cuh"

#include <cuda_bf16.h>

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

// ---------------------------------------------------------------- step 1
// One warp per (bh, chunk): inclusive scan of log alpha inside the chunk.
__global__ void decay_kernel(const float *__restrict__ g, float a_min,
                             float *__restrict__ gamma, int BH, int T, int C, int NC) {
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= (int64_t)BH * NC) return;  // uniform per warp
    const int bh = (int)(warp / NC), n = (int)(warp % NC);
    const int t0 = n * C;
    const int per = (C + 31) / 32;  // rows per lane: 1 (C <= 32) or 2 (C = 64)
    float lam[2] = {0.f, 0.f};
    float local = 0.f;
    for (int e = 0; e < per; ++e) {
        const int r = lane * per + e, t = t0 + r;
        if (r < C && t < T) local += log_alpha(g[(int64_t)bh * T + t], a_min);
        lam[e] = local;
    }
    float incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float excl = incl - local;
    for (int e = 0; e < per; ++e) {
        const int r = lane * per + e, t = t0 + r;
        if (r < C && t < T) gamma[(int64_t)bh * T + t] = expf(excl + lam[e]);
    }
}

// ---------------------------------------------------------------- step 2
// One CTA per (chunk, bh).  A, T = (I + A)^-1, U = T diag(beta) V,
// Wk = T diag(beta gamma) K.
template <typename TE>
__global__ void wy_kernel(const TE *__restrict__ k, const TE *__restrict__ v,
                          const float *__restrict__ beta, const float *__restrict__ gamma,
                          float *__restrict__ U, float *__restrict__ Wk, int T, int dk, int dv,
                          int C) {
    extern __shared__ float sm[];
    const int n = blockIdx.x, bh = blockIdx.y;
    const int t0 = n * C;
    const int c = min(C, T - t0);
    const int ldk = dk + 1, ldc = C + 1;
    float *Ks = sm;                   // [C][dk+1]
    float *Vs = Ks + C * ldk;         // [C][dv]
    float *As = Vs + C * dv;          // [C][C+1]
    float *Ts = As + C * ldc;         // [C][C+1]
    float *gs = Ts + C * ldc;         // [C]  gamma
    float *ig = gs + C;               // [C]  1/gamma
    float *bs = ig + C;               // [C]  beta
    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t row0 = (int64_t)bh * T + t0;

    for (int x = tid; x < c * dk; x += nt) {
        const int r = x / dk, i = x % dk;
        Ks[r * ldk + i] = ld_elem(k, (row0 + r) * dk + i);
    }
    for (int x = tid; x < c * dv; x += nt) Vs[x] = ld_elem(v, row0 * dv + x);
    for (int r = tid; r < c; r += nt) {
        gs[r] = gamma[row0 + r];
        ig[r] = 1.0f / gs[r];
        bs[r] = beta[row0 + r];
    }
    __syncthreads();

    // A[r][s] = (beta_r gamma_r) (k_r . k_s) (1 / gamma_s) for s < r.
    for (int x = tid; x < c * c; x += nt) {
        const int r = x / c, s = x % c;
        float a = 0.f;
        if (s < r) {
            float d = 0.f;
            for (int i = 0; i < dk; ++i) d = fmaf(Ks[r * ldk + i], Ks[s * ldk + i], d);
            a = (bs[r] * gs[r]) * d * ig[s];
        }
        As[r * ldc + s] = a;
        Ts[r * ldc + s] = (r == s) ? 1.f : 0.f;
    }
    __syncthreads();

    // Forward substitution, one row at a time: (I + A) T = I gives
    // T[r][s] = -sum_{m=s}^{r-1} A[r][m] T[m][s] for s < r, T[r][r] = 1.
    for (int r = 1; r < c; ++r) {
        for (int s = tid; s < r; s += nt) {
            float acc = 0.f;
            for (int m = s; m < r; ++m) acc = fmaf(As[r * ldc + m], Ts[m * ldc + s], acc);
            Ts[r * ldc + s] = -acc;
        }
        __syncthreads();
    }

    for (int x = tid; x < c * dv; x += nt) {
        const int r = x / dv, j = x % dv;
        float acc = 0.f;
        for (int s = 0; s <= r; ++s) acc = fmaf(Ts[r * ldc + s] * bs[s], Vs[s * dv + j], acc);
        U[(row0 + r) * dv + j] = acc;
    }
    for (int x = tid; x < c * dk; x += nt) {
        const int r = x / dk, i = x % dk;
        float acc = 0.f;
        for (int s = 0; s <= r; ++s)
            acc = fmaf(Ts[r * ldc + s] * (bs[s] * gs[s]), Ks[s * ldk + i], acc);
        Wk[(row0 + r) * dk + i] = acc;
    }
}

// ---------------------------------------------------------------- step 3
// One CTA per (dv slice, bh), sequential over chunks.  The state slice
// M[:, j0:j0+DS] lives in shared memory for the whole pass.
template <typename TE>
__global__ void state_kernel(const TE *__restrict__ k, const float *__restrict__ gamma,
                             const float *__restrict__ U, const float *__restrict__ Wk,
                             const float *init, float *__restrict__ W, float *__restrict__ Mn,
                             float *final_state, int T, int dk, int dv, int C, int DS) {
    extern __shared__ float sm[];
    const int j0 = blockIdx.x * DS, bh = blockIdx.y;
    const int ldk = dk + 1;
    float *Ms = sm;                  // [dk][DS]
    float *Ks = Ms + dk * DS;        // [C][dk+1]
    float *Wks = Ks + C * ldk;       // [C][dk+1]
    float *Ws = Wks + C * ldk;       // [C][DS]
    float *sc = Ws + C * DS;         // [C]  gamma_C / gamma_r
    const int tid = threadIdx.x, nt = blockDim.x;
    const int NC = (T + C - 1) / C;

    for (int x = tid; x < dk * DS; x += nt) {
        const int i = x / DS, j = x % DS;
        Ms[x] = init ? init[((int64_t)bh * dk + i) * dv + j0 + j] : 0.f;
    }
    for (int n = 0; n < NC; ++n) {
        const int t0 = n * C, c = min(C, T - t0);
        const int64_t row0 = (int64_t)bh * T + t0;
        __syncthreads();
        for (int x = tid; x < c * dk; x += nt) {
            const int r = x / dk, i = x % dk;
            Ks[r * ldk + i] = ld_elem(k, (row0 + r) * dk + i);
            Wks[r * ldk + i] = Wk[(row0 + r) * dk + i];
        }
        {
            const float gC = gamma[row0 + c - 1];
            for (int r = tid; r < c; r += nt) sc[r] = gC / gamma[row0 + r];
        }
        if (Mn) {
            for (int x = tid; x < dk * DS; x += nt) {
                const int i = x / DS, j = x % DS;
                Mn[(((int64_t)bh * NC + n) * dk + i) * dv + j0 + j] = Ms[x];
            }
        }
        __syncthreads();
        // W = U - Wk M
        for (int x = tid; x < c * DS; x += nt) {
            const int r = x / DS, j = x % DS;
            float acc = U[(row0 + r) * dv + j0 + j];
            for (int i = 0; i < dk; ++i) acc = fmaf(-Wks[r * ldk + i], Ms[i * DS + j], acc);
            Ws[r * DS + j] = acc;
            W[(row0 + r) * dv + j0 + j] = acc;
        }
        __syncthreads();
        // M <- gamma_C M + (diag(gamma_C / gamma) K)^T W
        const float gC = gamma[row0 + c - 1];
        for (int x = tid; x < dk * DS; x += nt) {
            const int i = x / DS, j = x % DS;
            float acc = 0.f;
            for (int r = 0; r < c; ++r) acc = fmaf(sc[r] * Ks[r * ldk + i], Ws[r * DS + j], acc);
            Ms[x] = fmaf(gC, Ms[x], acc);
        }
    }
    __syncthreads();
    if (final_state) {
        for (int x = tid; x < dk * DS; x += nt) {
            const int i = x / DS, j = x % DS;
            final_state[((int64_t)bh * dk + i) * dv + j0 + j] = Ms[x];
        }
    }
}

// ---------------------------------------------------------------- step 4
// One CTA per (chunk, bh).  Thread (j, rg) accumulates rows r = rg + RG*m.
constexpr int kOutMaxRows = 32;

template <typename TE>
__global__ void output_kernel(const TE *__restrict__ q, const TE *__restrict__ k,
                              const float *__restrict__ gamma, const float *__restrict__ Mn,
                              const float *__restrict__ W, TE *__restrict__ out, int T, int dk,
                              int dv, int C) {
    extern __shared__ float sm[];
    const int n = blockIdx.x, bh = blockIdx.y;
    const int NC = (T + C - 1) / C;
    const int t0 = n * C, c = min(C, T - t0);
    const int ldk = dk + 1, ldc = C + 1;
    float *Qs = sm;                 // [C][dk+1]
    float *Ks = Qs + C * ldk;       // [C][dk+1]
    float *Ps = Ks + C * ldk;       // [C][C+1]
    float *gs = Ps + C * ldc;       // [C]
    float *ig = gs + C;             // [C]
    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t row0 = (int64_t)bh * T + t0;
    for (int x = tid; x < c * dk; x += nt) {
        const int r = x / dk, i = x % dk;
        Qs[r * ldk + i] = ld_elem(q, (row0 + r) * dk + i);
        Ks[r * ldk + i] = ld_elem(k, (row0 + r) * dk + i);
    }
    for (int r = tid; r < c; r += nt) {
        gs[r] = gamma[row0 + r];
        ig[r] = 1.0f / gs[r];
    }
    __syncthreads();
    // P[r][s] = gamma_r (q_r . k_s) (1 / gamma_s), s <= r  (diagonal tile, dense)
    for (int x = tid; x < c * c; x += nt) {
        const int r = x / c, s = x % c;
        float p = 0.f;
        if (s <= r) {
            float d = 0.f;
            for (int i = 0; i < dk; ++i) d = fmaf(Qs[r * ldk + i], Ks[s * ldk + i], d);
            p = gs[r] * d * ig[s];
        }
        Ps[r * ldc + s] = p;
    }
    __syncthreads();

    const int j = tid % dv, rg = tid / dv, RG = nt / dv;
    if (rg >= RG) return;
    float acc[kOutMaxRows];
#pragma unroll
    for (int m = 0; m < kOutMaxRows; ++m) acc[m] = 0.f;
    const float *Mp = Mn + ((int64_t)bh * NC + n) * dk * dv;
    for (int i = 0; i < dk; ++i) {
        const float mij = Mp[(int64_t)i * dv + j];
#pragma unroll
        for (int m = 0; m < kOutMaxRows; ++m) {
            const int r = rg + RG * m;
            if (r < c) acc[m] = fmaf(Qs[r * ldk + i], mij, acc[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < kOutMaxRows; ++m) {
        const int r = rg + RG * m;
        if (r < c) acc[m] *= gs[r];
    }
    for (int s = 0; s < c; ++s) {
        const float wsj = W[(row0 + s) * dv + j];
#pragma unroll
        for (int m = 0; m < kOutMaxRows; ++m) {
            const int r = rg + RG * m;
            if (r < c) acc[m] = fmaf(Ps[r * ldc + s], wsj, acc[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < kOutMaxRows; ++m) {
        const int r = rg + RG * m;
        if (r < c) st_elem(out, (row0 + r) * dv + j, acc[m]);
    }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)bytes);
}

}  // namespace

cudaError_t launch_decay(const float *g, float a_min, float *gamma, int BH, int T, int C,
                         cudaStream_t s) {
    const int NC = (T + C - 1) / C;
    const int64_t warps = (int64_t)BH * NC;
    if (warps == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    decay_kernel<<<(unsigned)blocks, threads, 0, s>>>(g, a_min, gamma, BH, T, C, NC);
    return cudaGetLastError();
}

cudaError_t launch_wy(const void *k, const void *v, const float *beta, const float *gamma,
                      float *U, float *Wk, int BH, int T, int dk, int dv, int C, Elem e,
                      cudaStream_t s) {
    const int NC = (T + C - 1) / C;
    if (BH == 0 || NC == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * ((size_t)C * (dk + 1) + (size_t)C * dv +
                                         2 * (size_t)C * (C + 1) + 3 * (size_t)C);
    dim3 grid(NC, BH);
    cudaError_t err;
    if (e == Elem::F32) {
        if ((err = set_smem(wy_kernel<float>, smem)) != cudaSuccess) return err;
        wy_kernel<float><<<grid, 256, smem, s>>>((const float *)k, (const float *)v, beta,
                                                 gamma, U, Wk, T, dk, dv, C);
    } else {
        if ((err = set_smem(wy_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return err;
        wy_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(
            (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, beta, gamma, U, Wk, T, dk,
            dv, C);
    }
    return cudaGetLastError();
}

cudaError_t launch_state(const void *k, const float *gamma, const float *U, const float *Wk,
                         const float *init, float *W, float *Mn, float *final_state, int BH,
                         int T, int dk, int dv, int C, Elem e, cudaStream_t s) {
    if (BH == 0 || T == 0) return cudaSuccess;
    const int DS = dv < 32 ? dv : 32;
    const size_t smem = sizeof(float) * ((size_t)dk * DS + 2 * (size_t)C * (dk + 1) +
                                         (size_t)C * DS + (size_t)C);
    dim3 grid(dv / DS, BH);
    cudaError_t err;
    if (e == Elem::F32) {
        if ((err = set_smem(state_kernel<float>, smem)) != cudaSuccess) return err;
        state_kernel<float><<<grid, 256, smem, s>>>((const float *)k, gamma, U, Wk, init, W,
                                                    Mn, final_state, T, dk, dv, C, DS);
    } else {
        if ((err = set_smem(state_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return err;
        state_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(
            (const __nv_bfloat16 *)k, gamma, U, Wk, init, W, Mn, final_state, T, dk, dv, C,
            DS);
    }
    return cudaGetLastError();
}

cudaError_t launch_output(const void *q, const void *k, const float *gamma, const float *Mn,
                          const float *W, void *out, int BH, int T, int dk, int dv, int C,
                          Elem e, cudaStream_t s) {
    const int NC = (T + C - 1) / C;
    if (BH == 0 || NC == 0) return cudaSuccess;
    // rows per thread: ceil(C / (256 / dv)) must fit kOutMaxRows
    const int RG = 256 / dv;
    if ((C + RG - 1) / RG > kOutMaxRows) return cudaErrorInvalidValue;
    const size_t smem = sizeof(float) * (2 * (size_t)C * (dk + 1) + (size_t)C * (C + 1) +
                                         2 * (size_t)C);
    dim3 grid(NC, BH);
    cudaError_t err;
    if (e == Elem::F32) {
        if ((err = set_smem(output_kernel<float>, smem)) != cudaSuccess) return err;
        output_kernel<float><<<grid, 256, smem, s>>>((const float *)q, (const float *)k,
                                                     gamma, Mn, W, (float *)out, T, dk, dv, C);
    } else {
        if ((err = set_smem(output_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return err;
        output_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(
            (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, gamma, Mn, W,
            (__nv_bfloat16 *)out, T, dk, dv, C);
    }
    return cudaGetLastError();
}

size_t staged_scratch_bytes(int64_t BH, int T, int dk, int dv, int C) {
    const int64_t NC = ((int64_t)T + C - 1) / C;
    const int64_t n_tok = BH * (int64_t)T;
    return sizeof(float) * (size_t)(n_tok * (1 + (int64_t)dv + dk + dv) + BH * NC * (int64_t)dk * dv);
}

cudaError_t launch_staged(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float d, const float *init, void *out,
                          float *final_state, void *scratch, int BH, int T, int dk, int dv,
                          int C, Elem e, cudaStream_t s) {
    if (BH == 0 || T == 0) return cudaSuccess;
    const size_t n_tok = (size_t)BH * (size_t)T;
    float *gamma = static_cast<float *>(scratch);   // [BH][T]
    float *U = gamma + n_tok;                      // [BH][T][dv]
    float *Wk = U + n_tok * dv;                    // [BH][T][dk]
    float *W = Wk + n_tok * dk;                    // [BH][T][dv]
    float *Mn = W + n_tok * dv;                    // [BH][NC][dk][dv]
    cudaError_t err = launch_decay(g, d, gamma, BH, T, C, s);
    if (err == cudaSuccess) err = launch_wy(k, v, beta, gamma, U, Wk, BH, T, dk, dv, C, e, s);
    if (err == cudaSuccess)
        err = launch_state(k, gamma, U, Wk, init, W, Mn, final_state, BH, T, dk, dv, C, e, s);
    if (err == cudaSuccess) err = launch_output(q, k, gamma, Mn, W, out, BH, T, dk, dv, C, e, s);
    return err;
}

cudaError_t launch_copy_state(const float *init, float *final_state, int64_t n, cudaStream_t s) {
    if (!final_state || n == 0) return cudaSuccess;
    if (init == final_state) return cudaSuccess;
    if (init)
        return cudaMemcpyAsync(final_state, init, sizeof(float) * (size_t)n,
                               cudaMemcpyDeviceToDevice, s);
    return cudaMemsetAsync(final_state, 0, sizeof(float) * (size_t)n, s);
}

}  // namespace gdr
