// gdr_bwd.cu -- the backward of the chunked gated delta rule: the gradients of
// a loss L with respect to q, k, v, g, beta and the initial state, given
// dL/dout and dL/dfinal_state.  fp32 CUDA-core kernels (inputs and the output
// gradients in the forward's element type, widened on load).
//
// The chunk algebra of the forward ("What a Trillion-Parameter MoE Model
// Reveals About the Next Stage of LLM Scaling", sections 3.1-3.3; the staged
// kernels of gdr_staged.cu recompute its intermediates gamma, W_n and M_n):
//   A  = strict_lower(diag(beta) D o K K^T),  D[r][s] = gamma_r / gamma_s
//   W  = (I + A)^-1 diag(beta) E,             E = V - diag(gamma) K M
//   O  = diag(gamma) Q M + P W,               P = lower_incl(D o Q K^T)
//   M' = gamma_C M + K^T diag(gamma_C / gamma) W
// differentiated in reverse (the transposed products of the same tiles).
//
// Reverse chain, sequential over chunks from the last (per value-column slice:
// the recurrence never mixes value columns), from dM' = dL/dM_{n+1}:
//   dW = P^T dO + diag(gamma_C / gamma) K dM'
//   dR = (I + A)^-T dW        (the gradient of diag(beta) E; a transposed
//                              unit-triangular solve)
//   dM = gamma_C dM' + Q^T diag(gamma) dO - K^T diag(gamma beta) dR
// It stores dR and dM' of every chunk.  Then every chunk on its own:
//   dQ = diag(gamma) dO M^T + (dP o D) K,                   dP = lower_incl(dO W^T)
//   dK = -diag(gamma beta) dR M^T + diag(gamma_C/gamma) W dM'^T
//        + (dP o D)^T Q + (dA o beta D) K + (dA o beta D)^T K, dA = -strict_lower(dR W^T)
//   dV = diag(beta) dR,   dbeta_r = (v_r - gamma_r M^T k_r) . dR_r + sum_s dA_rs D_rs k_r.k_s
//   db_r (b = the chunk's cumulative log-decay, gamma = e^b): the position-pair
//        terms of P and A, gamma_r q_r^T M dO_r - gamma_r beta_r k_r^T M dR_r,
//        -z_r with z_r = (gamma_C/gamma_r) k_r^T dM' w_r; the chunk's last row
//        also gets sum_r z_r + gamma_C <M, dM'>
//   dlog(alpha_t) = sum_{r >= t} db_r,   dg_t = dlog(alpha_t) * dlog(alpha)/dg.
// The initial state's gradient is the dM left after the first chunk.

#include "gdr_internal.h"
#include "gdr_math.cuh"

#include <cuda_bf16.h>

namespace gdr {
namespace {

__device__ __forceinline__ float ldx(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ldx(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void stx(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void stx(__nv_bfloat16 *p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// d log(alpha) / d g for the two decay forms (parameter d as in gdr_math.cuh).
__device__ __forceinline__ float dlog_alpha_dg(float g, float d) {
    const float s = 1.0f / (1.0f + expf(-g));
    return d > 0.0f ? (1.0f - d) * s * (1.0f - s) / decay_alpha(g, d) : d * s * (1.0f - s);
}

// ---------------------------------------------------------------- reverse chain
// One CTA per (value-column slice of DS, bh), sequential over chunks from the
// last.  dM[:, slice] lives in shared memory for the whole pass.
template <typename TE>
__global__ void bwd_chain_kernel(const TE *__restrict__ q, const TE *__restrict__ k,
                                 const float *__restrict__ gamma, const float *__restrict__ beta,
                                 const TE *__restrict__ dout, const float *dfinal,
                                 float *__restrict__ dR, float *__restrict__ dMn1, float *dinit,
                                 int T, int dk, int dv, int C, int DS) {
    extern __shared__ float sm[];
    const int j0 = blockIdx.x * DS, bh = blockIdx.y;
    const int ldk = dk + 1, ldc = C + 1;
    float *dMs = sm;                  // [dk][DS]
    float *Ks = dMs + dk * DS;        // [C][dk+1]
    float *Qs = Ks + C * ldk;         // [C][dk+1]
    float *Ps = Qs + C * ldk;         // [C][C+1]  P[r][s], s <= r
    float *As = Ps + C * ldc;         // [C][C+1]  A[r][s], s < r
    float *dOs = As + C * ldc;        // [C][DS]
    float *Xs = dOs + C * DS;         // [C][DS]   dW, then dR in place
    float *gs = Xs + C * DS;          // [C] gamma
    float *bs = gs + C;               // [C] beta
    const int tid = threadIdx.x, nt = blockDim.x;
    const int NC = (T + C - 1) / C;

    for (int x = tid; x < dk * DS; x += nt) {
        const int i = x / DS, j = x % DS;
        dMs[x] = dfinal ? dfinal[((int64_t)bh * dk + i) * dv + j0 + j] : 0.f;
    }
    for (int n = NC - 1; n >= 0; --n) {
        const int t0 = n * C, c = min(C, T - t0);
        const int64_t row0 = (int64_t)bh * T + t0;
        __syncthreads();   // the previous chunk is done with every buffer
        for (int x = tid; x < c * dk; x += nt) {
            const int r = x / dk, i = x % dk;
            Ks[r * ldk + i] = ldx(k, (row0 + r) * dk + i);
            Qs[r * ldk + i] = ldx(q, (row0 + r) * dk + i);
        }
        for (int x = tid; x < c * DS; x += nt) {
            const int r = x / DS, j = x % DS;
            dOs[x] = ldx(dout, (row0 + r) * dv + j0 + j);
        }
        for (int r = tid; r < c; r += nt) {
            gs[r] = gamma[row0 + r];
            bs[r] = beta[row0 + r];
        }
        // dM' of this chunk, for the per-chunk gradients
        for (int x = tid; x < dk * DS; x += nt) {
            const int i = x / DS, j = x % DS;
            dMn1[(((int64_t)bh * NC + n) * dk + i) * dv + j0 + j] = dMs[x];
        }
        __syncthreads();
        for (int x = tid; x < c * c; x += nt) {
            const int r = x / c, s = x % c;
            float p = 0.f, a = 0.f;
            if (s <= r) {
                float dq = 0.f, dkk = 0.f;
                for (int i = 0; i < dk; ++i) {
                    dq = fmaf(Qs[r * ldk + i], Ks[s * ldk + i], dq);
                    dkk = fmaf(Ks[r * ldk + i], Ks[s * ldk + i], dkk);
                }
                const float d = gs[r] / gs[s];
                p = d * dq;
                if (s < r) a = bs[r] * d * dkk;
            }
            Ps[r * ldc + s] = p;
            As[r * ldc + s] = a;
        }
        __syncthreads();
        // dW = P^T dO + diag(gamma_C / gamma) K dM'
        {
            const float gC = gs[c - 1];
            for (int x = tid; x < c * DS; x += nt) {
                const int r = x / DS, j = x % DS;
                float acc = 0.f;
                for (int m = r; m < c; ++m) acc = fmaf(Ps[m * ldc + r], dOs[m * DS + j], acc);
                float kd = 0.f;
                for (int i = 0; i < dk; ++i) kd = fmaf(Ks[r * ldk + i], dMs[i * DS + j], kd);
                Xs[x] = fmaf(gC / gs[r], kd, acc);
            }
        }
        __syncthreads();
        // (I + A)^T dR = dW: dR_r = dW_r - sum_{s > r} A[s][r] dR_s, from the last row;
        // one thread per column
        if (tid < DS) {
            const int j = tid;
            for (int r = c - 1; r >= 0; --r) {
                float acc = Xs[r * DS + j];
                for (int s = r + 1; s < c; ++s) acc = fmaf(-As[s * ldc + r], Xs[s * DS + j], acc);
                Xs[r * DS + j] = acc;
            }
        }
        __syncthreads();
        for (int x = tid; x < c * DS; x += nt) {
            const int r = x / DS, j = x % DS;
            dR[(row0 + r) * dv + j0 + j] = Xs[x];
        }
        // dM = gamma_C dM' + Q^T diag(gamma) dO - K^T diag(gamma beta) dR
        {
            const float gC = gs[c - 1];
            for (int x = tid; x < dk * DS; x += nt) {
                const int i = x / DS, j = x % DS;
                float acc = 0.f;
                for (int r = 0; r < c; ++r) {
                    acc = fmaf(gs[r] * Qs[r * ldk + i], dOs[r * DS + j], acc);
                    acc = fmaf(-gs[r] * bs[r] * Ks[r * ldk + i], Xs[r * DS + j], acc);
                }
                dMs[x] = fmaf(gC, dMs[x], acc);
            }
        }
    }
    __syncthreads();
    if (dinit) {
        for (int x = tid; x < dk * DS; x += nt) {
            const int i = x / DS, j = x % DS;
            dinit[((int64_t)bh * dk + i) * dv + j0 + j] = dMs[x];
        }
    }
}

// ---------------------------------------------------------------- per-chunk gradients
// One CTA per (chunk, bh), 256 threads.  Thread (i = tid % dk, rg = tid / dk)
// owns the dQ and dK elements of key column i in rows r = rg, rg + RG, ...
// (RG = 256 / dk), accumulated in registers over every term.
constexpr int kBwdThreads = 256;
constexpr int kBwdMaxRows = 32;   // C * dk / 256 for C = 64, dk = 128
constexpr int kBwdJB = 16;        // value columns of M and dM' staged at a time

template <typename TE>
__global__ void __launch_bounds__(kBwdThreads)
bwd_chunk_kernel(const TE *__restrict__ q, const TE *__restrict__ k, const TE *__restrict__ v,
                 const float *__restrict__ g, const float *__restrict__ beta, float d,
                 const float *__restrict__ gamma, const float *__restrict__ W,
                 const float *__restrict__ Mn, const TE *__restrict__ dout,
                 const float *__restrict__ dR, const float *__restrict__ dMn1,
                 TE *__restrict__ dq, TE *__restrict__ dk_out, TE *__restrict__ dv_out,
                 float *__restrict__ dg, float *__restrict__ dbeta, int T, int dk, int dv, int C) {
    extern __shared__ float sm[];
    const int n = blockIdx.x, bh = blockIdx.y;
    const int NC = (T + C - 1) / C;
    const int t0 = n * C, c = min(C, T - t0);
    const int64_t row0 = (int64_t)bh * T + t0;
    const int ldk = dk + 1, ldv = dv + 1, ldc = C + 1, ldj = kBwdJB + 1;
    float *Qs = sm;                     // [C][dk+1]
    float *Ks = Qs + C * ldk;           // [C][dk+1]
    float *Ws = Ks + C * ldk;           // [C][dv+1]
    float *dOs = Ws + C * ldv;          // [C][dv+1]
    float *dRs = dOs + C * ldv;         // [C][dv+1]
    float *FP = dRs + C * ldv;          // [C][C+1]  dP o D
    float *FA = FP + C * ldc;           // [C][C+1]  dA o beta D
    float *Mt = FA + C * ldc;           // [dk][JB+1]  M[:, jb]
    float *dMt = Mt + dk * ldj;         // [dk][JB+1]  dM'[:, jb]
    float *gs = dMt + dk * ldj;         // [C] gamma
    float *bs = gs + C;                 // [C] beta
    float *dbp = bs + C;                // [C] position-pair terms of db
    float *dbt = dbp + C;               // [C] position-pair terms of dbeta
    float *rq = dbt + C;                // [C] q_r^T M dO_r
    float *rk = rq + C;                 // [C] k_r^T M dR_r
    float *rz = rk + C;                 // [C] k_r^T dM' w_r
    float *red = rz + C;                // [2]: <M, dM'>, sum_r z_r
    const int tid = threadIdx.x;
    const float *Mp = Mn + ((int64_t)bh * NC + n) * dk * dv;
    const float *dMp = dMn1 + ((int64_t)bh * NC + n) * dk * dv;

    for (int x = tid; x < c * dk; x += kBwdThreads) {
        const int r = x / dk, i = x % dk;
        Qs[r * ldk + i] = ldx(q, (row0 + r) * dk + i);
        Ks[r * ldk + i] = ldx(k, (row0 + r) * dk + i);
    }
    for (int x = tid; x < c * dv; x += kBwdThreads) {
        const int r = x / dv, j = x % dv;
        Ws[r * ldv + j] = W[(row0 + r) * dv + j];
        dOs[r * ldv + j] = ldx(dout, (row0 + r) * dv + j);
        dRs[r * ldv + j] = dR[(row0 + r) * dv + j];
    }
    for (int r = tid; r < C; r += kBwdThreads) {
        gs[r] = r < c ? gamma[row0 + r] : 1.f;
        bs[r] = r < c ? beta[row0 + r] : 0.f;
        dbp[r] = dbt[r] = rq[r] = rk[r] = rz[r] = 0.f;
    }
    if (tid < 2) red[tid] = 0.f;
    __syncthreads();

    // position pairs (r, s), s <= r: P, A, dP, dA and their decay and beta terms
    for (int x = tid; x < C * C; x += kBwdThreads) {
        const int r = x / C, s = x % C;
        float fp = 0.f, fa = 0.f;
        if (r < c && s <= r) {
            float sqk = 0.f, skk = 0.f, dow = 0.f, drw = 0.f;
            for (int i = 0; i < dk; ++i) {
                sqk = fmaf(Qs[r * ldk + i], Ks[s * ldk + i], sqk);
                skk = fmaf(Ks[r * ldk + i], Ks[s * ldk + i], skk);
            }
            for (int j = 0; j < dv; ++j) {
                dow = fmaf(dOs[r * ldv + j], Ws[s * ldv + j], dow);
                drw = fmaf(dRs[r * ldv + j], Ws[s * ldv + j], drw);
            }
            const float D = gs[r] / gs[s];
            float e = dow * D * sqk;          // dP P
            fp = dow * D;
            if (s < r) {
                const float dA = -drw;
                e += dA * bs[r] * D * skk;    // dA A
                fa = dA * bs[r] * D;
                atomicAdd(&dbt[r], dA * D * skk);
            }
            if (s < r) {                      // e is zero on the diagonal's net
                atomicAdd(&dbp[r], e);
                atomicAdd(&dbp[s], -e);
            }
        }
        FP[r * ldc + s] = fp;
        FA[r * ldc + s] = fa;
    }
    __syncthreads();

    // state terms: aO = (dO M^T)[r][i], aR = (dR M^T)[r][i], aW = (W dM'^T)[r][i]
    const int i = tid % dk, rg = tid / dk, RG = kBwdThreads / dk;
    float aO[kBwdMaxRows], aR[kBwdMaxRows], aW[kBwdMaxRows];
#pragma unroll
    for (int m = 0; m < kBwdMaxRows; ++m) aO[m] = aR[m] = aW[m] = 0.f;
    float mdm = 0.f;   // this thread's share of <M, dM'>
    for (int jb = 0; jb < dv; jb += kBwdJB) {
        for (int x = tid; x < dk * kBwdJB; x += kBwdThreads) {
            const int ii = x / kBwdJB, jj = x % kBwdJB;
            const float mv = Mp[(int64_t)ii * dv + jb + jj], dmv = dMp[(int64_t)ii * dv + jb + jj];
            Mt[ii * ldj + jj] = mv;
            dMt[ii * ldj + jj] = dmv;
            mdm = fmaf(mv, dmv, mdm);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kBwdMaxRows; ++m) {
            const int r = rg + RG * m;
            if (r < c) {
                float o = aO[m], rr = aR[m], w = aW[m];
#pragma unroll
                for (int jj = 0; jj < kBwdJB; ++jj) {
                    const float mt = Mt[i * ldj + jj], dmt = dMt[i * ldj + jj];
                    o = fmaf(dOs[r * ldv + jb + jj], mt, o);
                    rr = fmaf(dRs[r * ldv + jb + jj], mt, rr);
                    w = fmaf(Ws[r * ldv + jb + jj], dmt, w);
                }
                aO[m] = o;
                aR[m] = rr;
                aW[m] = w;
            }
        }
        __syncthreads();
    }
    // row reductions over i of q.(M dO_r), k.(M dR_r), k.(dM' w_r); then the
    // state terms of dQ and dK in place of aO and aR
    {
        const float gC = gs[c - 1];
#pragma unroll
        for (int m = 0; m < kBwdMaxRows; ++m) {
            const int r = rg + RG * m;   // uniform over each warp (dk >= 32)
            if (r < c) {
                float pq = Qs[r * ldk + i] * aO[m];
                float pk = Ks[r * ldk + i] * aR[m];
                float pz = Ks[r * ldk + i] * aW[m];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    pq += __shfl_xor_sync(0xffffffffu, pq, off);
                    pk += __shfl_xor_sync(0xffffffffu, pk, off);
                    pz += __shfl_xor_sync(0xffffffffu, pz, off);
                }
                if ((tid & 31) == 0) {
                    atomicAdd(&rq[r], pq);
                    atomicAdd(&rk[r], pk);
                    atomicAdd(&rz[r], pz);
                }
                aO[m] *= gs[r];                                           // dQ
                aR[m] = fmaf(gC / gs[r], aW[m], -gs[r] * bs[r] * aR[m]);  // dK
            }
        }
    }
    for (int off = 16; off > 0; off >>= 1) mdm += __shfl_xor_sync(0xffffffffu, mdm, off);
    if ((tid & 31) == 0) atomicAdd(&red[0], mdm);

    // in-chunk terms: dQ += FP K,  dK += FP^T Q + FA K + FA^T K
#pragma unroll 4
    for (int s = 0; s < c; ++s) {
        const float ks = Ks[s * ldk + i], qs = Qs[s * ldk + i];
#pragma unroll
        for (int m = 0; m < kBwdMaxRows; ++m) {
            const int r = rg + RG * m;
            if (r < c) {
                aO[m] = fmaf(FP[r * ldc + s], ks, aO[m]);
                float t = fmaf(FP[s * ldc + r], qs, aR[m]);
                t = fmaf(FA[r * ldc + s], ks, t);
                aR[m] = fmaf(FA[s * ldc + r], ks, t);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kBwdMaxRows; ++m) {
        const int r = rg + RG * m;
        if (r < c) {
            stx(dq, (row0 + r) * dk + i, aO[m]);
            stx(dk_out, (row0 + r) * dk + i, aR[m]);
        }
    }
    for (int x = tid; x < c * dv; x += kBwdThreads) {
        const int r = x / dv, j = x % dv;
        stx(dv_out, (row0 + r) * dv + j, bs[r] * dRs[r * ldv + j]);
    }
    __syncthreads();

    // per row: dbeta, db, then dlog(alpha) as the reverse cumulative sum and dg
    if (tid < 32) {
        const float gC = gs[c - 1];
        float zsum = 0.f;
        float db[2] = {0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 2 * tid + e;
            if (r < c) {
                float vdr = 0.f;
                for (int j = 0; j < dv; ++j) vdr = fmaf(ldx(v, (row0 + r) * dv + j), dRs[r * ldv + j], vdr);
                dbeta[row0 + r] = dbt[r] + vdr - gs[r] * rk[r];
                const float z = gC / gs[r] * rz[r];
                zsum += z;
                db[e] = dbp[r] + gs[r] * rq[r] - gs[r] * bs[r] * rk[r] - z;
            }
        }
        for (int off = 16; off > 0; off >>= 1) zsum += __shfl_xor_sync(0xffffffffu, zsum, off);
        const float last = zsum + gC * red[0];   // the chunk's last row, through gamma_C
#pragma unroll
        for (int e = 0; e < 2; ++e)
            if (2 * tid + e == c - 1) db[e] += last;
        // suffix sums: dl_t = sum_{r >= t} db_r
        float tot = db[0] + db[1];
        float suf = tot;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, suf, off);
            if (tid + off < 32) suf += y;
        }
        const float dl1 = suf - db[0], dl0 = suf;
        const float dl[2] = {dl0, dl1};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 2 * tid + e;
            if (r < c) dg[row0 + r] = dl[e] * dlog_alpha_dg(g[row0 + r], d);
        }
    }
}

template <typename K>
cudaError_t bwd_set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

size_t chain_smem(int dk, int DS, int C) {
    return sizeof(float) * ((size_t)dk * DS + 2 * (size_t)C * (dk + 1) + 2 * (size_t)C * (C + 1) +
                            2 * (size_t)C * DS + 2 * (size_t)C);
}
size_t chunk_smem(int dk, int dv, int C) {
    return sizeof(float) * (2 * (size_t)C * (dk + 1) + 3 * (size_t)C * (dv + 1) +
                            2 * (size_t)C * (C + 1) + 2 * (size_t)dk * (kBwdJB + 1) + 7 * (size_t)C + 2);
}

size_t round4(size_t n) { return (n + 3) & ~(size_t)3; }

template <typename TE>
cudaError_t launch_bwd_t(const TE *q, const TE *k, const TE *v, const float *g, const float *beta,
                         float d, const float *init, const TE *dout, const float *dfinal, TE *dq,
                         TE *dk_out, TE *dv_out, float *dg, float *dbeta, float *dinit,
                         int BH, int T, int dk, int dv, int C, float *ws, Elem e, cudaStream_t s) {
    const int NC = (T + C - 1) / C;
    const size_t tok = (size_t)BH * T, st = (size_t)BH * NC * dk * dv;
    float *gamma = ws;
    float *U = gamma + round4(tok);
    float *Wk = U + round4(tok * dv);
    float *W = Wk + round4(tok * dk);
    float *Mn = W + round4(tok * dv);
    float *dR = Mn + round4(st);
    float *dMn1 = dR + round4(tok * dv);
    cudaError_t err = launch_decay(g, d, gamma, BH, T, C, s);
    if (err == cudaSuccess) err = launch_wy(k, v, beta, gamma, U, Wk, BH, T, dk, dv, C, e, s);
    if (err == cudaSuccess)
        err = launch_state(k, gamma, U, Wk, init, W, Mn, nullptr, BH, T, dk, dv, C, e, s);
    if (err != cudaSuccess) return err;
    const int DS = dv < 32 ? dv : 32;
    const size_t s1 = chain_smem(dk, DS, C);
    if ((err = bwd_set_smem(bwd_chain_kernel<TE>, s1)) != cudaSuccess) return err;
    bwd_chain_kernel<TE><<<dim3(dv / DS, BH), 256, s1, s>>>(q, k, gamma, beta, dout, dfinal, dR,
                                                           dMn1, dinit, T, dk, dv, C, DS);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    const size_t s2 = chunk_smem(dk, dv, C);
    if ((err = bwd_set_smem(bwd_chunk_kernel<TE>, s2)) != cudaSuccess) return err;
    bwd_chunk_kernel<TE><<<dim3(NC, BH), kBwdThreads, s2, s>>>(
        q, k, v, g, beta, d, gamma, W, Mn, dout, dR, dMn1, dq, dk_out, dv_out, dg, dbeta, T, dk, dv, C);
    return cudaGetLastError();
}

}  // namespace

bool bwd_supported(int dk, int dv, int C) {
    return (dk == 32 || dk == 64 || dk == 128) && (dv == 16 || dv == 32 || dv == 64 || dv == 128) &&
           (C == 16 || C == 32 || C == 64) && chunk_smem(dk, dv, C) <= 232448;
}

size_t bwd_workspace_bytes(int BH, int T, int dk, int dv, int C) {
    if (BH <= 0 || T <= 0) return 0;
    const int NC = (T + C - 1) / C;
    const size_t tok = (size_t)BH * T, st = (size_t)BH * NC * dk * dv;
    return sizeof(float) * (round4(tok) + round4(tok * dv) + round4(tok * dk) + round4(tok * dv) +
                            round4(st) + round4(tok * dv) + round4(st));
}

cudaError_t launch_bwd(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, float d, const float *init, const void *dout,
                       const float *dfinal, void *dq, void *dk_out, void *dv_out, float *dg,
                       float *dbeta, float *dinit, int BH, int T, int dk, int dv, int C,
                       void *ws, Elem e, cudaStream_t s) {
    if (BH == 0) return cudaSuccess;
    if (T == 0) {   // no tokens: dinit = dfinal
        if (!dinit) return cudaSuccess;
        if (dfinal)
            return cudaMemcpyAsync(dinit, dfinal, sizeof(float) * (size_t)BH * dk * dv,
                                   cudaMemcpyDeviceToDevice, s);
        return cudaMemsetAsync(dinit, 0, sizeof(float) * (size_t)BH * dk * dv, s);
    }
    float *w = static_cast<float *>(ws);
    if (e == Elem::F32)
        return launch_bwd_t<float>((const float *)q, (const float *)k, (const float *)v, g, beta, d,
                                   init, (const float *)dout, dfinal, (float *)dq, (float *)dk_out,
                                   (float *)dv_out, dg, dbeta, dinit, BH, T, dk, dv, C, w, e, s);
    return launch_bwd_t<__nv_bfloat16>(
        (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, g, beta, d,
        init, (const __nv_bfloat16 *)dout, dfinal, (__nv_bfloat16 *)dq, (__nv_bfloat16 *)dk_out,
        (__nv_bfloat16 *)dv_out, dg, dbeta, dinit, BH, T, dk, dv, C, w, e, s);
}

}  // namespace gdr
