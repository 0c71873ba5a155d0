// gdr_bwd.cu -- the backward of the chunked gated delta rule: the gradients of
// a loss L with respect to q, k, v, g, beta and the initial state, given
// dL/dout and dL/dfinal_state.  fp32 CUDA-core kernels (inputs and the output
// gradients in the forward's element type, widened on load), except for the bf16
// d = 128, chunk-64 shape, whose four kernels run on warp MMAs (below).
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
#include "gdr_sm100.cuh"

#include <cuda_bf16.h>
#include <type_traits>

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
__device__ __forceinline__ float dlog_alpha_dg(float g, float d) { return decay_dlog_dg(g, d); }

// ---------------------------------------------------------------- chunk tiles
// One CTA per (chunk, bh), all in parallel, 256 threads:
//   P[r][s]  = (gamma_r / gamma_s) q_r.k_s  (s <= r),
//   DK[r][s] = (gamma_r / gamma_s) k_r.k_s  (s < r; A = diag(beta) DK),
//   T = (I + A)^-1 (unit lower triangular, row by row),
//   U = T diag(beta) V,   Wk = T diag(beta gamma) K
// of every chunk, fp32: P, DK, T [BH][NC][C][C] (rows past a ragged chunk's end
// zero in P and DK, identity in T), U [BH,T,dv], Wk [BH,T,dk].  The products run in
// 4 x 4 (pairs) and 4 x 8 (U, Wk) register tiles.
template <typename TE>
__global__ void __launch_bounds__(256)
bwd_tiles_kernel(const TE *__restrict__ q, const TE *__restrict__ k, const TE *__restrict__ v,
                 const float *__restrict__ gamma, const float *__restrict__ beta,
                 float *__restrict__ Pt, float *__restrict__ Tt, float *__restrict__ DKt,
                 float *__restrict__ U, float *__restrict__ Wk, int T, int dk, int dv, int C) {
    extern __shared__ __align__(16) float sm[];
    const int n = blockIdx.x, bh = blockIdx.y;
    const int NC = (T + C - 1) / C;
    const int t0 = n * C, c = min(C, T - t0);
    const int64_t row0 = (int64_t)bh * T + t0;
    const int ldk = dk + 4, ldx4 = (dk > dv ? dk : dv) + 4, ldc = C + 1;
    float *Ks = sm;                 // [C][dk+4]  k, then diag(beta gamma) k
    float *QV = Ks + C * ldk;       // [C][max(dk,dv)+4]  q, then diag(beta) v
    float *As = QV + C * ldx4;      // [C][C+1]
    float *Ts = As + C * ldc;       // [C][C+1]
    float *gs = Ts + C * ldc;       // [C]
    float *bs = gs + C;             // [C]
    const int tid = threadIdx.x;
    const int64_t tb = ((int64_t)bh * NC + n) * C * C;
    for (int x = tid; x < C * dk; x += 256) {
        const int r = x / dk, i = x % dk;
        QV[r * ldx4 + i] = r < c ? ldx(q, (row0 + r) * dk + i) : 0.f;
        Ks[r * ldk + i] = r < c ? ldx(k, (row0 + r) * dk + i) : 0.f;
    }
    for (int r = tid; r < C; r += 256) {
        gs[r] = r < c ? gamma[row0 + r] : 1.f;
        bs[r] = r < c ? beta[row0 + r] : 0.f;
    }
    for (int x = tid; x < C * C; x += 256) Ts[(x / C) * ldc + x % C] = (x / C == x % C) ? 1.f : 0.f;
    __syncthreads();
    // position pairs in 4 x 4 tiles
    {
        const int TB = C / 4;
        for (int tile = tid; tile < TB * TB; tile += 256) {
            const int r0 = 4 * (tile / TB), s0 = 4 * (tile % TB);
            float aq[4][4], ak[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) aq[a][b] = ak[a][b] = 0.f;
            if (s0 <= r0 + 3) {
                for (int i = 0; i < dk; i += 4) {
                    float4 qr[4], kr[4], ks[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        qr[a] = *reinterpret_cast<const float4 *>(&QV[(r0 + a) * ldx4 + i]);
                        kr[a] = *reinterpret_cast<const float4 *>(&Ks[(r0 + a) * ldk + i]);
                        ks[a] = *reinterpret_cast<const float4 *>(&Ks[(s0 + a) * ldk + i]);
                    }
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            aq[a][b] = fmaf(qr[a].x, ks[b].x, fmaf(qr[a].y, ks[b].y,
                                       fmaf(qr[a].z, ks[b].z, fmaf(qr[a].w, ks[b].w, aq[a][b]))));
                            ak[a][b] = fmaf(kr[a].x, ks[b].x, fmaf(kr[a].y, ks[b].y,
                                       fmaf(kr[a].z, ks[b].z, fmaf(kr[a].w, ks[b].w, ak[a][b]))));
                        }
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int r = r0 + a, s = s0 + b;
                    float p = 0.f, dkk = 0.f;
                    if (r < c && s <= r) {
                        const float D = gs[r] / gs[s];
                        p = D * aq[a][b];
                        if (s < r) dkk = D * ak[a][b];
                    }
                    Pt[tb + r * C + s] = p;
                    DKt[tb + r * C + s] = dkk;
                    As[r * ldc + s] = bs[r] * dkk;
                }
        }
    }
    __syncthreads();
    // diag(beta) v over q, diag(beta gamma) k in place
    for (int x = tid; x < C * dv; x += 256) {
        const int r = x / dv, j = x % dv;
        QV[r * ldx4 + j] = r < c ? bs[r] * ldx(v, (row0 + r) * dv + j) : 0.f;
    }
    for (int x = tid; x < C * dk; x += 256) {
        const int r = x / dk, i = x % dk;
        Ks[r * ldk + i] *= bs[r] * gs[r];
    }
    // forward substitution, one row at a time: T[r][s] = -sum_{m=s}^{r-1} A[r][m] T[m][s]
    for (int r = 1; r < c; ++r) {
        __syncthreads();
        for (int s = tid; s < r; s += 256) {
            float acc = 0.f;
            for (int m = s; m < r; ++m) acc = fmaf(As[r * ldc + m], Ts[m * ldc + s], acc);
            Ts[r * ldc + s] = -acc;
        }
    }
    __syncthreads();
    for (int x = tid; x < C * C; x += 256) Tt[tb + x] = Ts[(x / C) * ldc + x % C];
    // U = T diag(beta) V and Wk = T diag(beta gamma) K: tiles of 4 rows x 8 columns over
    // the dv columns of U, then the dk columns of Wk
    {
        const int GV = dv / 8, GK = dk / 8, RB = C / 4;
        for (int tile = tid; tile < RB * (GV + GK); tile += 256) {
            const int r0 = 4 * (tile / (GV + GK)), cg = tile % (GV + GK);
            const bool isU = cg < GV;
            const int j0 = 8 * (isU ? cg : cg - GV);
            const float *B = isU ? QV : Ks;
            const int ldb = isU ? ldx4 : ldk;
            float acc[4][8];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[a][e] = 0.f;
            const int smax = min(r0 + 4, C);
            for (int s = 0; s < smax; ++s) {
                const float4 b0 = *reinterpret_cast<const float4 *>(&B[s * ldb + j0]);
                const float4 b1 = *reinterpret_cast<const float4 *>(&B[s * ldb + j0 + 4]);
                const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const float t = Ts[(r0 + a) * ldc + s];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[a][e] = fmaf(t, bv[e], acc[a][e]);
                }
            }
            float *out = isU ? U : Wk;
            const int ld = isU ? dv : dk;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int r = r0 + a;
                if (r < c) {
                    *reinterpret_cast<float4 *>(&out[(row0 + r) * ld + j0]) =
                        make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
                    *reinterpret_cast<float4 *>(&out[(row0 + r) * ld + j0 + 4]) =
                        make_float4(acc[a][4], acc[a][5], acc[a][6], acc[a][7]);
                }
            }
        }
    }
}

// ---------------------------------------------------------------- reverse chain
// 16-byte vector access to the element types.
__device__ __forceinline__ uint4 ld16(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void widen16(const uint4 &u, float *f, const float *) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void widen16(const uint4 &u, float *f, const __nv_bfloat16 *) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
        f[2 * e] = t.x;
        f[2 * e + 1] = t.y;
    }
}

// Shared-memory copies of k and q keep the element type of the inputs (bf16 values
// are exact as given): one element, or four consecutive ones, widened to fp32.
__device__ __forceinline__ float sk1(const float *p) { return *p; }
__device__ __forceinline__ float sk1(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ float4 sk4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 sk4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// One chunk's inputs of the reverse chain, held in registers between their load
// and their store to shared memory, so that the loads of chunk n - 1 run while
// chunk n computes.  Per thread: 16-byte pieces of K and Q, of P and T, of the dO
// slice, and gamma, beta of row tid.
template <typename TE, int DS>
struct ChainStage {
    static constexpr int V = 16 / (int)sizeof(TE);        // elements per 16 bytes
    static constexpr int NKQ = 64 * 128 / V / 256;          // at most C = 64, dk = 128
    static constexpr int NPT = 64 * 64 / 4 / 256;
    static constexpr int NO = (64 * DS / V + 255) / 256;
    uint4 kq[2][NKQ];
    float4 pt[2][NPT];
    uint4 o[NO];
    float gb[2];

    __device__ void load(const TE *q, const TE *k, const TE *dout, const float *gamma,
                         const float *beta, const float *Pp, const float *Tp, int64_t row0, int c,
                         int C, int dk, int dv, int j0s, int tid) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < NKQ; ++u) {
            const int idx = tid + 256 * u;
            if (idx < C * dk / V) {
                const int r = idx * V / dk, col = idx * V % dk;
                kq[0][u] = r < c ? ld16(k + (row0 + r) * dk + col) : z;
                kq[1][u] = r < c ? ld16(q + (row0 + r) * dk + col) : z;
            }
        }
#pragma unroll
        for (int u = 0; u < NPT; ++u) {
            const int idx = tid + 256 * u;
            if (idx < C * C / 4) {
                pt[0][u] = __ldg(reinterpret_cast<const float4 *>(Pp) + idx);
                pt[1][u] = __ldg(reinterpret_cast<const float4 *>(Tp) + idx);
            }
        }
#pragma unroll
        for (int u = 0; u < NO; ++u) {
            const int idx = tid + 256 * u;
            if (idx < C * DS / V) {
                const int r = idx * V / DS, col = idx * V % DS;
                o[u] = r < c ? ld16(dout + (row0 + r) * dv + j0s + col) : z;
            }
        }
        if (tid < C) {
            gb[0] = tid < c ? gamma[row0 + tid] : 1.f;
            gb[1] = tid < c ? beta[row0 + tid] : 0.f;
        }
    }
    __device__ void store(TE *Ks, TE *Qs, float *Ps, float *Tsm, float *dOs, float *gs,
                          float *bs, int C, int dk, int ldk, int tid) const {
#pragma unroll
        for (int u = 0; u < NKQ; ++u) {
            const int idx = tid + 256 * u;
            if (idx < C * dk / V) {   // k and q as given: 16 bytes as loaded
                const int r = idx * V / dk, col = idx * V % dk;
                *reinterpret_cast<uint4 *>(Ks + r * ldk + col) = kq[0][u];
                *reinterpret_cast<uint4 *>(Qs + r * ldk + col) = kq[1][u];
            }
        }
#pragma unroll
        for (int u = 0; u < NPT; ++u) {
            const int idx = tid + 256 * u;
            if (idx < C * C / 4) {
                reinterpret_cast<float4 *>(Ps)[idx] = pt[0][u];
                reinterpret_cast<float4 *>(Tsm)[idx] = pt[1][u];
            }
        }
#pragma unroll
        for (int u = 0; u < NO; ++u) {
            const int idx = tid + 256 * u;
            if (idx < C * DS / V) {
                const int r = idx * V / DS, col = idx * V % DS;
                float f[V];
                widen16(o[u], f, (const TE *)nullptr);
#pragma unroll
                for (int e = 0; e < V; ++e) dOs[r * DS + col + e] = f[e];
            }
        }
        if (tid < C) {
            gs[tid] = gb[0];
            bs[tid] = gb[1];
        }
    }
};

// One CTA per (DS value columns, bh), sequential over chunks from the last;
// dM[:, slice] lives in shared memory for the whole pass.  Each product is
// register-tiled: a thread owns 2 x 4 outputs of dW and dR, 4 x 4 of dM.  The
// gamma and gamma beta scalings ride on dO and dR, so K and Q stay as given.
template <typename TE, int DS>
__global__ void __launch_bounds__(256)
bwd_chain_kernel(const TE *__restrict__ q, const TE *__restrict__ k,
                 const float *__restrict__ gamma, const float *__restrict__ beta,
                 const TE *__restrict__ dout, const float *dfinal, const float *__restrict__ Pt,
                 const float *__restrict__ Tt, float *__restrict__ dR, float *__restrict__ dMn1,
                 float *dinit, int T, int dk, int dv, int C) {
    extern __shared__ __align__(16) float sm[];
    const int j0s = blockIdx.x * DS, bh = blockIdx.y;
    const int ldk = dk + 16 / (int)sizeof(TE);   // 16-byte rows, rows 4 banks apart
    float *dMs = sm;                      // [dk][DS]
    float *Ps = dMs + dk * DS;            // [C][C]
    float *Tsm = Ps + C * C;              // [C][C]
    float *dOs = Tsm + C * C;             // [C][DS]  dO
    float *dWs = dOs + C * DS;            // [C][DS]  dW
    float *dRg = dWs + C * DS;            // [C][DS]  gamma beta dR
    float *gs = dRg + C * DS;             // [C]
    float *bs = gs + C;                   // [C]
    float *scs = bs + C;                  // [C] gamma_C / gamma
    TE *Ks = reinterpret_cast<TE *>(sm + ((dk * DS + 2 * C * C + 3 * C * DS + 3 * C + 3) & ~3));
    TE *Qs = Ks + C * ldk;                // [C][ldk]  k, q in the input element type
    const int tid = threadIdx.x;
    const int NC = (T + C - 1) / C;
    constexpr int JG = DS / 4;            // column groups of 4
    auto tile_p = [&](int n) { return Pt + ((int64_t)bh * NC + n) * C * C; };
    auto tile_t = [&](int n) { return Tt + ((int64_t)bh * NC + n) * C * C; };

    for (int x = tid; x < dk * DS; x += 256) {
        const int i = x / DS, j = x % DS;
        dMs[x] = dfinal ? dfinal[((int64_t)bh * dk + i) * dv + j0s + j] : 0.f;
    }
    ChainStage<TE, DS> stage;
    {
        const int n = NC - 1, c = T - n * C;
        stage.load(q, k, dout, gamma, beta, tile_p(n), tile_t(n), (int64_t)bh * T + n * C, c, C, dk,
                   dv, j0s, tid);
        stage.store(Ks, Qs, Ps, Tsm, dOs, gs, bs, C, dk, ldk, tid);
    }
    for (int n = NC - 1; n >= 0; --n) {
        const int t0 = n * C, c = min(C, T - t0);
        const int64_t row0 = (int64_t)bh * T + t0;
        __syncthreads();   // chunk n's inputs are in shared memory
        if (n > 0)         // the previous chunk's loads run while this one computes
            stage.load(q, k, dout, gamma, beta, tile_p(n - 1), tile_t(n - 1), row0 - C, C, C, dk, dv,
                       j0s, tid);
        for (int x = tid; x < dk * DS; x += 256) {   // dM' of this chunk
            const int i = x / DS, j = x % DS;
            dMn1[(((int64_t)bh * NC + n) * dk + i) * dv + j0s + j] = dMs[x];
        }
        const float gC = gs[c - 1];
        for (int r = tid; r < C; r += 256) scs[r] = r < c ? gC / gs[r] : 0.f;
        __syncthreads();
        // dW = P^T dO + diag(gamma_C / gamma) K dM'   (rows r0, r0 + 1; columns jq .. jq + 3)
        for (int tile = tid; tile < (C / 2) * JG; tile += 256) {
            const int r0 = 2 * (tile / JG), jq = 4 * (tile % JG);
            float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
            for (int m = r0; m < C; ++m) {
                const float2 p = *reinterpret_cast<const float2 *>(&Ps[m * C + r0]);
                const float4 b = *reinterpret_cast<const float4 *>(&dOs[m * DS + jq]);
                a0[0] = fmaf(p.x, b.x, a0[0]); a0[1] = fmaf(p.x, b.y, a0[1]);
                a0[2] = fmaf(p.x, b.z, a0[2]); a0[3] = fmaf(p.x, b.w, a0[3]);
                a1[0] = fmaf(p.y, b.x, a1[0]); a1[1] = fmaf(p.y, b.y, a1[1]);
                a1[2] = fmaf(p.y, b.z, a1[2]); a1[3] = fmaf(p.y, b.w, a1[3]);
            }
            float k0[4] = {0.f, 0.f, 0.f, 0.f}, k1[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i = 0; i < dk; ++i) {
                const float x0 = sk1(Ks + r0 * ldk + i), x1 = sk1(Ks + (r0 + 1) * ldk + i);
                const float4 b = *reinterpret_cast<const float4 *>(&dMs[i * DS + jq]);
                k0[0] = fmaf(x0, b.x, k0[0]); k0[1] = fmaf(x0, b.y, k0[1]);
                k0[2] = fmaf(x0, b.z, k0[2]); k0[3] = fmaf(x0, b.w, k0[3]);
                k1[0] = fmaf(x1, b.x, k1[0]); k1[1] = fmaf(x1, b.y, k1[1]);
                k1[2] = fmaf(x1, b.z, k1[2]); k1[3] = fmaf(x1, b.w, k1[3]);
            }
            const float s0 = scs[r0], s1 = scs[r0 + 1];
            *reinterpret_cast<float4 *>(&dWs[r0 * DS + jq]) =
                make_float4(fmaf(s0, k0[0], a0[0]), fmaf(s0, k0[1], a0[1]), fmaf(s0, k0[2], a0[2]),
                            fmaf(s0, k0[3], a0[3]));
            *reinterpret_cast<float4 *>(&dWs[(r0 + 1) * DS + jq]) =
                make_float4(fmaf(s1, k1[0], a1[0]), fmaf(s1, k1[1], a1[1]), fmaf(s1, k1[2], a1[2]),
                            fmaf(s1, k1[3], a1[3]));
        }
        __syncthreads();
        // dR = T^T dW, the gradient of diag(beta) E; gamma beta dR for the state update
        for (int tile = tid; tile < (C / 2) * JG; tile += 256) {
            const int r0 = 2 * (tile / JG), jq = 4 * (tile % JG);
            float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
            for (int m = r0; m < C; ++m) {
                const float2 t = *reinterpret_cast<const float2 *>(&Tsm[m * C + r0]);
                const float4 b = *reinterpret_cast<const float4 *>(&dWs[m * DS + jq]);
                a0[0] = fmaf(t.x, b.x, a0[0]); a0[1] = fmaf(t.x, b.y, a0[1]);
                a0[2] = fmaf(t.x, b.z, a0[2]); a0[3] = fmaf(t.x, b.w, a0[3]);
                a1[0] = fmaf(t.y, b.x, a1[0]); a1[1] = fmaf(t.y, b.y, a1[1]);
                a1[2] = fmaf(t.y, b.z, a1[2]); a1[3] = fmaf(t.y, b.w, a1[3]);
            }
            const float g0 = gs[r0] * bs[r0], g1 = gs[r0 + 1] * bs[r0 + 1];
            *reinterpret_cast<float4 *>(&dRg[r0 * DS + jq]) =
                make_float4(g0 * a0[0], g0 * a0[1], g0 * a0[2], g0 * a0[3]);
            *reinterpret_cast<float4 *>(&dRg[(r0 + 1) * DS + jq]) =
                make_float4(g1 * a1[0], g1 * a1[1], g1 * a1[2], g1 * a1[3]);
            if (r0 < c)
                *reinterpret_cast<float4 *>(&dR[(row0 + r0) * dv + j0s + jq]) =
                    make_float4(a0[0], a0[1], a0[2], a0[3]);
            if (r0 + 1 < c)
                *reinterpret_cast<float4 *>(&dR[(row0 + r0 + 1) * dv + j0s + jq]) =
                    make_float4(a1[0], a1[1], a1[2], a1[3]);
        }
        __syncthreads();
        // dM = gamma_C dM' + Q^T (gamma dO) - K^T (gamma beta dR)   (rows iq .. iq + 3)
        for (int tile = tid; tile < (dk / 4) * JG; tile += 256) {
            const int iq = 4 * (tile / JG), jq = 4 * (tile % JG);
            float acc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float4 m0 = *reinterpret_cast<const float4 *>(&dMs[(iq + a) * DS + jq]);
                acc[a][0] = gC * m0.x; acc[a][1] = gC * m0.y; acc[a][2] = gC * m0.z; acc[a][3] = gC * m0.w;
            }
            for (int r = 0; r < c; ++r) {
                const float4 qa = sk4(Qs + r * ldk + iq);
                const float4 ka = sk4(Ks + r * ldk + iq);
                const float4 ob = *reinterpret_cast<const float4 *>(&dOs[r * DS + jq]);
                const float4 rb = *reinterpret_cast<const float4 *>(&dRg[r * DS + jq]);
                const float gr = gs[r];
                const float qv[4] = {qa.x, qa.y, qa.z, qa.w}, kv[4] = {ka.x, ka.y, ka.z, ka.w};
                const float ov[4] = {gr * ob.x, gr * ob.y, gr * ob.z, gr * ob.w};
                const float rv[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(qv[a], ov[b], fmaf(-kv[a], rv[b], acc[a][b]));
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
                *reinterpret_cast<float4 *>(&dMs[(iq + a) * DS + jq]) =
                    make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        }
        __syncthreads();   // every read of chunk n's inputs is done
        if (n > 0) stage.store(Ks, Qs, Ps, Tsm, dOs, gs, bs, C, dk, ldk, tid);
    }
    __syncthreads();
    if (dinit) {
        for (int x = tid; x < dk * DS; x += 256) {
            const int i = x / DS, j = x % DS;
            dinit[((int64_t)bh * dk + i) * dv + j0s + j] = dMs[x];
        }
    }
}

// ---------------------------------------------------------------- forward states
// One chunk's inputs of the forward-state pass, staged in registers like the
// reverse chain's: K rows, Wk rows, the U slice, gamma of row tid.
template <typename TE, int DS>
struct FwdStage {
    static constexpr int V = 16 / (int)sizeof(TE);
    static constexpr int NK = 64 * 128 / V / 256;
    static constexpr int NW = 64 * 128 / 4 / 256;
    static constexpr int NU = (64 * DS / 4 + 255) / 256;
    uint4 kk[NK];
    float4 wk[NW], u[NU];
    float gm;
    __device__ void load(const TE *k, const float *Wk, const float *U, const float *gamma,
                         int64_t row0, int c, int C, int dk, int dv, int j0s, int tid) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int x = 0; x < NK; ++x) {
            const int idx = tid + 256 * x;
            if (idx < C * dk / V) {
                const int r = idx * V / dk, col = idx * V % dk;
                kk[x] = r < c ? ld16(k + (row0 + r) * dk + col) : z;
            }
        }
#pragma unroll
        for (int x = 0; x < NW; ++x) {
            const int idx = tid + 256 * x;
            if (idx < C * dk / 4) {
                const int r = idx * 4 / dk, col = idx * 4 % dk;
                wk[x] = r < c ? __ldg(reinterpret_cast<const float4 *>(Wk + (row0 + r) * dk + col)) : zf;
            }
        }
#pragma unroll
        for (int x = 0; x < NU; ++x) {
            const int idx = tid + 256 * x;
            if (idx < C * DS / 4) {
                const int r = idx * 4 / DS, col = idx * 4 % DS;
                u[x] = r < c ? __ldg(reinterpret_cast<const float4 *>(U + (row0 + r) * dv + j0s + col)) : zf;
            }
        }
        if (tid < C) gm = tid < c ? gamma[row0 + tid] : 1.f;
    }
    __device__ void store(float *Ks, float *Wks, float *Us, float *gs, int C, int dk, int ldk,
                          int tid) const {
#pragma unroll
        for (int x = 0; x < NK; ++x) {
            const int idx = tid + 256 * x;
            if (idx < C * dk / V) {
                const int r = idx * V / dk, col = idx * V % dk;
                float f[V];
                widen16(kk[x], f, (const TE *)nullptr);
#pragma unroll
                for (int e = 0; e < V; ++e) Ks[r * ldk + col + e] = f[e];
            }
        }
#pragma unroll
        for (int x = 0; x < NW; ++x) {
            const int idx = tid + 256 * x;
            if (idx < C * dk / 4) {
                const int r = idx * 4 / dk, col = idx * 4 % dk;
                *reinterpret_cast<float4 *>(&Wks[r * ldk + col]) = wk[x];
            }
        }
#pragma unroll
        for (int x = 0; x < NU; ++x) {
            const int idx = tid + 256 * x;
            if (idx < C * DS / 4) reinterpret_cast<float4 *>(Us)[idx] = u[x];
        }
        if (tid < C) gs[tid] = gm;
    }
};

// The forward's state pass again, for the backward's recompute, register-tiled
// like the reverse chain: per chunk W = U - Wk M (rows r0, r0 + 1), then
// M <- gamma_C M + K^T diag(gamma_C / gamma) W (rows iq .. iq + 3); writes W and
// the state at every chunk start.  One CTA per (DS value columns, bh).
template <typename TE, int DS>
__global__ void __launch_bounds__(256)
bwd_fwd_state_kernel(const TE *__restrict__ k, const float *__restrict__ gamma,
                     const float *__restrict__ U, const float *__restrict__ Wk, const float *init,
                     float *__restrict__ W, float *__restrict__ Mn, int T, int dk, int dv, int C) {
    extern __shared__ __align__(16) float sm[];
    const int j0s = blockIdx.x * DS, bh = blockIdx.y;
    const int ldk = dk + 4;
    float *Ms = sm;                       // [dk][DS]
    float *Ks = Ms + dk * DS;             // [C][dk+4]  k
    float *Wks = Ks + C * ldk;            // [C][dk+4]  Wk
    float *Us = Wks + C * ldk;            // [C][DS]    U slice
    float *Ws = Us + C * DS;              // [C][DS]    diag(gamma_C / gamma) W
    float *gs = Ws + C * DS;              // [C]
    const int tid = threadIdx.x;
    const int NC = (T + C - 1) / C;
    constexpr int JG = DS / 4;
    for (int x = tid; x < dk * DS; x += 256) {
        const int i = x / DS, j = x % DS;
        Ms[x] = init ? init[((int64_t)bh * dk + i) * dv + j0s + j] : 0.f;
    }
    FwdStage<TE, DS> stage;
    stage.load(k, Wk, U, gamma, (int64_t)bh * T, min(C, T), C, dk, dv, j0s, tid);
    stage.store(Ks, Wks, Us, gs, C, dk, ldk, tid);
    for (int n = 0; n < NC; ++n) {
        const int t0 = n * C, c = min(C, T - t0);
        const int64_t row0 = (int64_t)bh * T + t0;
        __syncthreads();   // chunk n's inputs are in shared memory
        if (n + 1 < NC)
            stage.load(k, Wk, U, gamma, row0 + C, min(C, T - t0 - C), C, dk, dv, j0s, tid);
        for (int x = tid; x < dk * DS; x += 256) {
            const int i = x / DS, j = x % DS;
            Mn[(((int64_t)bh * NC + n) * dk + i) * dv + j0s + j] = Ms[x];
        }
        const float gC = gs[c - 1];
        for (int tile = tid; tile < (C / 2) * JG; tile += 256) {
            const int r0 = 2 * (tile / JG), jq = 4 * (tile % JG);
            float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i = 0; i < dk; ++i) {
                const float x0 = Wks[r0 * ldk + i], x1 = Wks[(r0 + 1) * ldk + i];
                const float4 b = *reinterpret_cast<const float4 *>(&Ms[i * DS + jq]);
                a0[0] = fmaf(x0, b.x, a0[0]); a0[1] = fmaf(x0, b.y, a0[1]);
                a0[2] = fmaf(x0, b.z, a0[2]); a0[3] = fmaf(x0, b.w, a0[3]);
                a1[0] = fmaf(x1, b.x, a1[0]); a1[1] = fmaf(x1, b.y, a1[1]);
                a1[2] = fmaf(x1, b.z, a1[2]); a1[3] = fmaf(x1, b.w, a1[3]);
            }
            const float4 u0 = *reinterpret_cast<const float4 *>(&Us[r0 * DS + jq]);
            const float4 u1 = *reinterpret_cast<const float4 *>(&Us[(r0 + 1) * DS + jq]);
            const float4 w0 = make_float4(u0.x - a0[0], u0.y - a0[1], u0.z - a0[2], u0.w - a0[3]);
            const float4 w1 = make_float4(u1.x - a1[0], u1.y - a1[1], u1.z - a1[2], u1.w - a1[3]);
            const float s0 = r0 < c ? gC / gs[r0] : 0.f, s1 = r0 + 1 < c ? gC / gs[r0 + 1] : 0.f;
            *reinterpret_cast<float4 *>(&Ws[r0 * DS + jq]) = make_float4(s0 * w0.x, s0 * w0.y, s0 * w0.z, s0 * w0.w);
            *reinterpret_cast<float4 *>(&Ws[(r0 + 1) * DS + jq]) =
                make_float4(s1 * w1.x, s1 * w1.y, s1 * w1.z, s1 * w1.w);
            if (r0 < c) *reinterpret_cast<float4 *>(&W[(row0 + r0) * dv + j0s + jq]) = w0;
            if (r0 + 1 < c) *reinterpret_cast<float4 *>(&W[(row0 + r0 + 1) * dv + j0s + jq]) = w1;
        }
        __syncthreads();
        for (int tile = tid; tile < (dk / 4) * JG; tile += 256) {
            const int iq = 4 * (tile / JG), jq = 4 * (tile % JG);
            float acc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float4 m0 = *reinterpret_cast<const float4 *>(&Ms[(iq + a) * DS + jq]);
                acc[a][0] = gC * m0.x; acc[a][1] = gC * m0.y; acc[a][2] = gC * m0.z; acc[a][3] = gC * m0.w;
            }
            for (int r = 0; r < c; ++r) {
                const float4 ka = *reinterpret_cast<const float4 *>(&Ks[r * ldk + iq]);
                const float4 wb = *reinterpret_cast<const float4 *>(&Ws[r * DS + jq]);
                const float kv[4] = {ka.x, ka.y, ka.z, ka.w}, wv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(kv[a], wv[b], acc[a][b]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
                *reinterpret_cast<float4 *>(&Ms[(iq + a) * DS + jq]) =
                    make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        }
        __syncthreads();   // every read of chunk n's inputs is done
        if (n + 1 < NC) stage.store(Ks, Wks, Us, gs, C, dk, ldk, tid);
    }
}

// ---------------------------------------------------------------- per-chunk gradients
// One CTA per (chunk, bh), 256 threads, every product register-tiled:
//  1. the position pairs: dO W^T and dR W^T in 4 x 4 tiles, then FP = dP o D and
//     FA = dA o beta D written over P and DK, with their db and dbeta terms;
//  2. the state terms dO M^T, dR M^T and W dM'^T in 4 (rows) x 8 (key columns)
//     tiles, M and dM' staged 16 value columns at a time, and the row dots
//     q.(M dO), k.(M dR), k.(dM' w) the decay and beta gradients need;
//  3. the in-chunk terms FP K, FP^T Q, FA K, FA^T K on the same tiles;
//  4. dv, dbeta, db and dg per row.
constexpr int kBwdThreads = 256;
constexpr int kBwdJB = 16;        // value columns of M and dM' staged at a time

// Rows 0 .. C-1 of a row-major matrix (width elements per row, source stride ld,
// rows >= c read as zero) into shared fp32 rows of stride lds, in 16-byte pieces:
// issue() puts every load in flight, commit() stores them, so the loads of several
// matrices overlap.
template <typename TE>
struct RowLoader {
    static constexpr int V = 16 / (int)sizeof(TE);
    static constexpr int MAXV = 64 * 128 / V / kBwdThreads;
    uint4 buf[MAXV];
    __device__ __forceinline__ void issue(const TE *src, int64_t row0, int c, int C, int width, int ld,
                                          int tid) {
#pragma unroll
        for (int u = 0; u < MAXV; ++u) {
            const int idx = tid + kBwdThreads * u;
            buf[u] = make_uint4(0u, 0u, 0u, 0u);
            if (idx < C * width / V) {
                const int r = idx * V / width, col = idx * V % width;
                if (r < c) buf[u] = ld16(src + (row0 + r) * ld + col);
            }
        }
    }
    __device__ __forceinline__ void commit(float *dst, int lds, int C, int width, int tid) const {
#pragma unroll
        for (int u = 0; u < MAXV; ++u) {
            const int idx = tid + kBwdThreads * u;
            if (idx < C * width / V) {
                const int r = idx * V / width, col = idx * V % width;
                float f[V];
                widen16(buf[u], f, (const TE *)nullptr);
#pragma unroll
                for (int e = 0; e < V; ++e) dst[r * lds + col + e] = f[e];
            }
        }
    }
};

template <typename TE>
__global__ void __launch_bounds__(kBwdThreads)
bwd_chunk_kernel(const TE *__restrict__ q, const TE *__restrict__ k, const TE *__restrict__ v,
                 const float *__restrict__ g, const float *__restrict__ beta, float d,
                 const float *__restrict__ gamma, const float *__restrict__ W,
                 const float *__restrict__ Mn, const TE *__restrict__ dout,
                 const float *__restrict__ dR, const float *__restrict__ dMn1,
                 const float *__restrict__ Pt, const float *__restrict__ DKt,
                 TE *__restrict__ dq, TE *__restrict__ dk_out, TE *__restrict__ dv_out,
                 float *__restrict__ dg, float *__restrict__ dbeta, int T, int dk, int dv, int C) {
    extern __shared__ __align__(16) float sm[];
    const int n = blockIdx.x, bh = blockIdx.y;
    const int NC = (T + C - 1) / C;
    const int t0 = n * C, c = min(C, T - t0);
    const int64_t row0 = (int64_t)bh * T + t0;
    const int ldk = dk + 4, ldv = dv + 4;
    float *Qs = sm;                     // [C][dk+4]
    float *Ks = Qs + C * ldk;           // [C][dk+4]
    float *Ws = Ks + C * ldk;           // [C][dv+4]
    float *dOs = Ws + C * ldv;          // [C][dv+4]
    float *dRs = dOs + C * ldv;         // [C][dv+4]
    float *PF = dRs + C * ldv;          // [C][C]  P, then FP = dP o D
    float *DF = PF + C * C;             // [C][C]  DK, then FA = dA o beta D
    float *Mt = DF + C * C;             // [JB][dk+4]  M[:, jb + jj], transposed
    float *dMt = Mt + kBwdJB * ldk;     // [JB][dk+4]  dM'[:, jb + jj], transposed
    float *gs = dMt + kBwdJB * ldk;     // [C] gamma
    float *bs = gs + C;                 // [C] beta
    float *dbp = bs + C;                // [C] position-pair terms of db
    float *dbt = dbp + C;               // [C] position-pair terms of dbeta
    float *rq = dbt + C;                // [C] q_r^T M dO_r
    float *rk = rq + C;                 // [C] k_r^T M dR_r
    float *rz = rk + C;                 // [C] k_r^T dM' w_r
    float *vdr = rz + C;                // [C] v_r . dR_r
    float *red = vdr + C;               // [1] <M, dM'>
    const int tid = threadIdx.x;
    const float *Mp = Mn + ((int64_t)bh * NC + n) * dk * dv;
    const float *dMp = dMn1 + ((int64_t)bh * NC + n) * dk * dv;
    const float *Pp = Pt + ((int64_t)bh * NC + n) * C * C;
    const float *DKp = DKt + ((int64_t)bh * NC + n) * C * C;

    {
        RowLoader<TE> lq, lk, lo;
        RowLoader<float> lw, lr;
        lq.issue(q, row0, c, C, dk, dk, tid);
        lk.issue(k, row0, c, C, dk, dk, tid);
        lo.issue(dout, row0, c, C, dv, dv, tid);
        lw.issue(W, row0, c, C, dv, dv, tid);
        lr.issue(dR, row0, c, C, dv, dv, tid);
        for (int r = tid; r < C; r += kBwdThreads) {
            gs[r] = r < c ? gamma[row0 + r] : 1.f;
            bs[r] = r < c ? beta[row0 + r] : 0.f;
            dbp[r] = dbt[r] = rq[r] = rk[r] = rz[r] = vdr[r] = 0.f;
        }
        if (tid == 0) red[0] = 0.f;
        lq.commit(Qs, ldk, C, dk, tid);
        lk.commit(Ks, ldk, C, dk, tid);
        lo.commit(dOs, ldv, C, dv, tid);
        lw.commit(Ws, ldv, C, dv, tid);
        lr.commit(dRs, ldv, C, dv, tid);
        RowLoader<float> lp, ld;
        lp.issue(Pp, 0, C, C, C, C, tid);
        ld.issue(DKp, 0, C, C, C, C, tid);
        lp.commit(PF, C, C, C, tid);
        ld.commit(DF, C, C, C, tid);
    }
    __syncthreads();

    // 1. position pairs (r, s): thread (rho, sig) owns rows rho + TB a and columns
    //    sig + TB b (a, b < 4, TB = C / 4), so a warp's reads of W rows are 16 consecutive
    //    rows (conflict-free); pairs above the diagonal are masked
    {
        const int TB = C / 4;
        for (int tile = tid; tile < TB * TB; tile += kBwdThreads) {
            const int rho = tile / TB, sig = tile % TB;
            float ao[4][4], ar[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) ao[a][b] = ar[a][b] = 0.f;
            for (int j = 0; j < dv; j += 4) {
                float4 o[4], rr[4], w[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    o[a] = *reinterpret_cast<const float4 *>(&dOs[(rho + TB * a) * ldv + j]);
                    rr[a] = *reinterpret_cast<const float4 *>(&dRs[(rho + TB * a) * ldv + j]);
                    w[a] = *reinterpret_cast<const float4 *>(&Ws[(sig + TB * a) * ldv + j]);
                }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        ao[a][b] = fmaf(o[a].x, w[b].x, fmaf(o[a].y, w[b].y,
                                   fmaf(o[a].z, w[b].z, fmaf(o[a].w, w[b].w, ao[a][b]))));
                        ar[a][b] = fmaf(rr[a].x, w[b].x, fmaf(rr[a].y, w[b].y,
                                   fmaf(rr[a].z, w[b].z, fmaf(rr[a].w, w[b].w, ar[a][b]))));
                    }
            }
            float re[4] = {0.f, 0.f, 0.f, 0.f}, ce[4] = {0.f, 0.f, 0.f, 0.f};
            float rt[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int r = rho + TB * a, s = sig + TB * b;
                    float fp = 0.f, fa = 0.f;
                    if (r < c && s <= r) {
                        const float D = gs[r] / gs[s];
                        const float dP = ao[a][b];
                        fp = dP * D;
                        float e = dP * PF[r * C + s];
                        if (s < r) {
                            const float dA = -ar[a][b], dkk = DF[r * C + s];
                            fa = dA * bs[r] * D;
                            e = fmaf(dA * bs[r], dkk, e);
                            rt[a] = fmaf(dA, dkk, rt[a]);
                        }
                        re[a] += e;
                        ce[b] -= e;
                    }
                    PF[r * C + s] = fp;
                    DF[r * C + s] = fa;
                }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                if (rho + TB * a < c) {
                    atomicAdd(&dbp[rho + TB * a], re[a]);
                    atomicAdd(&dbt[rho + TB * a], rt[a]);
                }
                if (sig + TB * a < c) atomicAdd(&dbp[sig + TB * a], ce[a]);
            }
        }
    }

    // 2. state terms, tile (rows r0 .. r0 + 3) x (key columns c0 .. c0 + 3 and c1 .. c1 + 3:
    //    a half-warp's float4 reads of a row cover 256 contiguous bytes)
    const int IG = dk / 8;
    const int tile = tid, r0 = 4 * (tile / IG), c0 = 4 * (tile % IG), c1 = dk / 2 + c0;
    auto colx = [&](int e) { return e < 4 ? c0 + e : c1 + e - 4; };
    const bool own = tile < (C / 4) * IG;
    float aO[4][8], aR[4][8], aW[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int e = 0; e < 8; ++e) aO[a][e] = aR[a][e] = aW[a][e] = 0.f;
    float mdm = 0.f;   // this thread's share of <M, dM'>
    // M and dM' go through registers a block of 16 value columns at a time: the next
    // block's loads run while the current one computes
    constexpr int NMB = 128 * kBwdJB / 4 / kBwdThreads;
    float4 mb[NMB], db[NMB];
    auto load_blk = [&](int jb) {
#pragma unroll
        for (int u = 0; u < NMB; ++u) {
            const int idx = tid + kBwdThreads * u;
            if (idx < dk * kBwdJB / 4) {
                const int i = idx / (kBwdJB / 4), j4 = 4 * (idx % (kBwdJB / 4));
                mb[u] = __ldg(reinterpret_cast<const float4 *>(Mp + (int64_t)i * dv + jb + j4));
                db[u] = __ldg(reinterpret_cast<const float4 *>(dMp + (int64_t)i * dv + jb + j4));
            }
        }
    };
    load_blk(0);
    for (int jb = 0; jb < dv; jb += kBwdJB) {
        __syncthreads();   // the previous block's M and dM' are read (and step 1 done)
#pragma unroll
        for (int u = 0; u < NMB; ++u) {
            const int idx = tid + kBwdThreads * u;
            if (idx < dk * kBwdJB / 4) {
                const int i = idx / (kBwdJB / 4), j4 = 4 * (idx % (kBwdJB / 4));
                const float mv[4] = {mb[u].x, mb[u].y, mb[u].z, mb[u].w};
                const float dmv[4] = {db[u].x, db[u].y, db[u].z, db[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    Mt[(j4 + e) * ldk + i] = mv[e];
                    dMt[(j4 + e) * ldk + i] = dmv[e];
                    mdm = fmaf(mv[e], dmv[e], mdm);
                }
            }
        }
        if (jb + kBwdJB < dv) load_blk(jb + kBwdJB);
        __syncthreads();
        if (own) {
#pragma unroll 1
            for (int j4 = 0; j4 < kBwdJB; j4 += 4) {
                float4 o[4], rr[4], w[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    o[a] = *reinterpret_cast<const float4 *>(&dOs[(r0 + a) * ldv + jb + j4]);
                    rr[a] = *reinterpret_cast<const float4 *>(&dRs[(r0 + a) * ldv + jb + j4]);
                    w[a] = *reinterpret_cast<const float4 *>(&Ws[(r0 + a) * ldv + jb + j4]);
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const float4 m0 = *reinterpret_cast<const float4 *>(&Mt[(j4 + jj) * ldk + c0]);
                    const float4 m1 = *reinterpret_cast<const float4 *>(&Mt[(j4 + jj) * ldk + c1]);
                    const float4 d0 = *reinterpret_cast<const float4 *>(&dMt[(j4 + jj) * ldk + c0]);
                    const float4 d1 = *reinterpret_cast<const float4 *>(&dMt[(j4 + jj) * ldk + c1]);
                    const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
                    const float dmv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        const float oa = jj == 0 ? o[a].x : jj == 1 ? o[a].y : jj == 2 ? o[a].z : o[a].w;
                        const float ra = jj == 0 ? rr[a].x : jj == 1 ? rr[a].y : jj == 2 ? rr[a].z : rr[a].w;
                        const float wa = jj == 0 ? w[a].x : jj == 1 ? w[a].y : jj == 2 ? w[a].z : w[a].w;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            aO[a][e] = fmaf(oa, mv[e], aO[a][e]);
                            aR[a][e] = fmaf(ra, mv[e], aR[a][e]);
                            aW[a][e] = fmaf(wa, dmv[e], aW[a][e]);
                        }
                    }
                }
            }
        }
    }
    // row dots over the tile's key columns, reduced across the IG threads of a row
    // group (consecutive lanes); then the state terms of dQ and dK in place
    {
        const float gC = gs[c - 1];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            float pq = 0.f, pk = 0.f, pz = 0.f;
            if (own) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float qv = Qs[(r0 + a) * ldk + colx(e)], kv = Ks[(r0 + a) * ldk + colx(e)];
                    pq = fmaf(qv, aO[a][e], pq);
                    pk = fmaf(kv, aR[a][e], pk);
                    pz = fmaf(kv, aW[a][e], pz);
                }
            }
            for (int off = 1; off < IG; off <<= 1) {
                pq += __shfl_xor_sync(0xffffffffu, pq, off);
                pk += __shfl_xor_sync(0xffffffffu, pk, off);
                pz += __shfl_xor_sync(0xffffffffu, pz, off);
            }
            const int r = r0 + a;
            if (own && (tile % IG) == 0 && r < c) {
                rq[r] = pq;
                rk[r] = pk;
                rz[r] = pz;
            }
            const float gr = gs[r < C ? r : 0], sc = gC / gr, gb = gr * bs[r < C ? r : 0];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                aO[a][e] *= gr;                                   // dQ
                aR[a][e] = fmaf(sc, aW[a][e], -gb * aR[a][e]);    // dK
            }
        }
    }
    for (int off = 16; off > 0; off >>= 1) mdm += __shfl_xor_sync(0xffffffffu, mdm, off);
    if ((tid & 31) == 0) atomicAdd(&red[0], mdm);

    // 3. in-chunk terms: dQ += FP K,  dK += FP^T Q + FA K + FA^T K
    if (own) {
        for (int s4 = 0; s4 < C; s4 += 4) {
            float4 fpr[4], far[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                fpr[a] = *reinterpret_cast<const float4 *>(&PF[(r0 + a) * C + s4]);
                far[a] = *reinterpret_cast<const float4 *>(&DF[(r0 + a) * C + s4]);
            }
#pragma unroll
            for (int ss = 0; ss < 4; ++ss) {
                const int s = s4 + ss;
                const float4 k0 = *reinterpret_cast<const float4 *>(&Ks[s * ldk + c0]);
                const float4 k1 = *reinterpret_cast<const float4 *>(&Ks[s * ldk + c1]);
                const float4 q0 = *reinterpret_cast<const float4 *>(&Qs[s * ldk + c0]);
                const float4 q1 = *reinterpret_cast<const float4 *>(&Qs[s * ldk + c1]);
                const float4 fpt = *reinterpret_cast<const float4 *>(&PF[s * C + r0]);
                const float4 fat = *reinterpret_cast<const float4 *>(&DF[s * C + r0]);
                const float kv[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                const float qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                const float ft[4] = {fpt.x, fpt.y, fpt.z, fpt.w}, at[4] = {fat.x, fat.y, fat.z, fat.w};
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const float fp = ss == 0 ? fpr[a].x : ss == 1 ? fpr[a].y : ss == 2 ? fpr[a].z : fpr[a].w;
                    const float fa = ss == 0 ? far[a].x : ss == 1 ? far[a].y : ss == 2 ? far[a].z : far[a].w;
                    const float fk = fa + at[a];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        aO[a][e] = fmaf(fp, kv[e], aO[a][e]);
                        aR[a][e] = fmaf(ft[a], qv[e], fmaf(fk, kv[e], aR[a][e]));
                    }
                }
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int r = r0 + a;
            if (r < c) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    stx(dq, (row0 + r) * dk + colx(e), aO[a][e]);
                    stx(dk_out, (row0 + r) * dk + colx(e), aR[a][e]);
                }
            }
        }
    }
    {
        // dv = diag(beta) dR, and v_r . dR_r reduced over groups of min(dv, 32) lanes
        const int gw = dv < 32 ? dv : 32;
        for (int x0 = 0; x0 < C * dv; x0 += kBwdThreads) {
            const int x = x0 + tid, r = x / dv, j = x % dv;
            float p = 0.f;
            if (r < c) {
                const float dr = dRs[r * ldv + j];
                stx(dv_out, (row0 + r) * dv + j, bs[r] * dr);
                p = ldx(v, (row0 + r) * dv + j) * dr;
            }
            for (int off = 1; off < gw; off <<= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
            if ((tid % gw) == 0 && r < c) atomicAdd(&vdr[r], p);
        }
    }
    __syncthreads();

    // 4. per row: dbeta, db, then dlog(alpha) as the reverse cumulative sum and dg
    if (tid < 32) {
        const float gC = gs[c - 1];
        float zsum = 0.f;
        float db[2] = {0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 2 * tid + e;
            if (r < c) {
                dbeta[row0 + r] = dbt[r] + vdr[r] - gs[r] * rk[r];
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
        // suffix sums: dlog(alpha_t) = sum_{r >= t} db_r
        float suf = db[0] + db[1];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, suf, off);
            if (tid + off < 32) suf += y;
        }
        const float dl[2] = {suf, suf - db[0]};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = 2 * tid + e;
            if (r < c) dg[row0 + r] = dl[e] * dlog_alpha_dg(g[row0 + r], d);
        }
    }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// rows 0 .. rows-1 of a row-major matrix (row_bytes a multiple of 16) into shared rows of
// pitch sp bytes by cp.async; rows >= c are zero-filled (their source clamped to row 0)
__device__ __forceinline__ void stage_rows(uint32_t dst, const void *src, int64_t src_pitch, int row_bytes,
                                           int sp, int rows, int c, int tid, int nthreads) {
    const int per_row = row_bytes / 16;
    for (int x = tid; x < rows * per_row; x += nthreads) {
        const int r = x / per_row, p = x % per_row;
        const bool in = r < c;
        const char *s = static_cast<const char *>(src) + (in ? r * src_pitch : 0) + 16 * p;
        cp_async16(dst + r * sp + 16 * p, s, in ? 16u : 0u);
    }
}

// 64 rows of 128 bytes whose 16-byte chunks are swizzled by row (chunk p of row r at
// byte r * 128 + 16 (p ^ (r mod 8))) into plain rows sp bytes apart
__device__ __forceinline__ void stage_rows_sw128(uint32_t dst, const void *src, int sp, int tid, int nthreads) {
    for (int x = tid; x < 64 * 8; x += nthreads) {
        const int r = x >> 3, p = x & 7;
        cp_async16(dst + r * sp + 16 * p, static_cast<const char *>(src) + r * 128 + ((p ^ (r & 7)) << 4), 16u);
    }
}

// [p, p + bytes) towards L2 (16-byte aligned, a multiple of 16 bytes)
__device__ __forceinline__ void l2_prefetch(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- per-chunk gradients, warp MMA
// The per-chunk gradients of the bf16 prefill shape (dk = dv = 128, C = 64) with every
// product on warp-level MMAs (mma.sync m16n8k16, bf16 operands, fp32 accumulation):
// q, k and dO enter as given, W, dR, M and dM' are rounded to bf16 once, FP and FA
// (formed in fp32) as operands.  Same four steps as bwd_chunk_kernel; 8 warps, the
// pairs in 16 x 32 warp tiles, the state and in-chunk products in 32 x 32.  Shared
// rows carry 16 bytes of padding, so each ldmatrix reads eight rows from eight
// different bank groups.
namespace mm {
constexpr int C = 64, D = 128, LD = D + 8, LC = C + 8;
constexpr uint32_t OFF_Q = 0, OFF_K = OFF_Q + C * LD * 2, OFF_O = OFF_K + C * LD * 2,
                   OFF_W = OFF_O + C * LD * 2, OFF_R = OFF_W + D * LC * 2,
                   OFF_M = OFF_R + C * LD * 2, OFF_DM = OFF_M + D * LD * 2,
                   OFF_FP = OFF_DM + D * LD * 2, OFF_FA = OFF_FP + C * LC * 2,
                   OFF_Q2 = OFF_FA + C * LC * 2, OFF_K2 = OFF_Q2 + C * LD * 2,   // q, k: second slot
                   OFF_SC = OFF_K2 + C * LD * 2;
constexpr uint32_t SMEM = OFF_SC + (8 * C + 4) * 4;
static_assert(OFF_Q2 - OFF_FP >= C * LD * 2 && OFF_M - OFF_R >= C * LD * 2,
              "dQ and dK leave through the FP, FA and dR tiles");
}  // namespace mm

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
// A fragment (16 x 16 at row R, column Kc) of a row-major bf16 tile, ldmatrix address
__device__ __forceinline__ uint32_t a_addr(uint32_t base, int ld, int R, int Kc, int lane) {
    return base + 2u * (uint32_t)((R + (lane & 7) + ((lane >> 3) & 1) * 8) * ld + Kc + (lane >> 4) * 8);
}
// Element offset of (r, col) in a bf16 [64][64] tile of 128-byte rows whose 16-byte chunks
// are swizzled by row (chunk c of row r at chunk c ^ (r mod 8)): the layout of the T and P
// tiles the reverse chain copies in whole
__device__ __forceinline__ int sw_elem(int r, int col) {
    return r * 64 + ((((col >> 3) ^ (r & 7))) << 3) + (col & 7);
}
// A fragment of the transpose of a row-major tile X (A[r][s] = X[s][r]), for ldmatrix.trans
__device__ __forceinline__ uint32_t at_addr(uint32_t base, int ld, int R, int Kc, int lane) {
    return base + 2u * (uint32_t)((Kc + (lane & 7) + (lane >> 4) * 8) * ld + R + ((lane >> 3) & 1) * 8);
}
// B fragments of n-tiles N, N + 8 (k = Kc .. Kc + 15) from a row-major [n][k] tile
__device__ __forceinline__ uint32_t b_addr(uint32_t base, int ld, int N, int Kc, int lane) {
    return base + 2u * (uint32_t)((N + (lane & 7) + (lane >> 4) * 8) * ld + Kc + ((lane >> 3) & 1) * 8);
}
// ... and from a row-major [k][n] tile, for ldmatrix.trans
__device__ __forceinline__ uint32_t bt_addr(uint32_t base, int ld, int N, int Kc, int lane) {
    return base + 2u * (uint32_t)((Kc + (lane & 7) + ((lane >> 3) & 1) * 8) * ld + N + (lane >> 4) * 8);
}

__global__ void __launch_bounds__(256)
bwd_chunk_mma_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                     const __nv_bfloat16 *__restrict__ v, const float *__restrict__ g,
                     const float *__restrict__ beta, float d, const float *__restrict__ gamma,
                     const __nv_bfloat16 *__restrict__ Wt, const __nv_bfloat16 *__restrict__ Sb,
                     const __nv_bfloat16 *__restrict__ dout, const float *__restrict__ dR,
                     const __nv_bfloat16 *__restrict__ dSb, __nv_bfloat16 *__restrict__ dq,
                     __nv_bfloat16 *__restrict__ dk_out, __nv_bfloat16 *__restrict__ dv_out,
                     float *__restrict__ dg, float *__restrict__ dbeta, int T, int BH) {
    using namespace mm;
    using sm100::ldsm_x4;
    using sm100::ldsm_x4_t;
    using sm100::mma16816;
    extern __shared__ __align__(16) uint8_t smb[];
    const int NC = (T + C - 1) / C;
    const int ntask = NC * BH;
    const int tid0 = threadIdx.x;
    const uint32_t sb0 = sm100::smem_u32(smb);
    // Persistent: one CTA per SM walks the chunks (task = bh * NC + n, stride gridDim.x).
    // The next chunk's tiles arrive by cp.async while this one computes: q, k into a
    // second slot right away, S, dS', dO, W^T once this chunk's state terms are done.
    auto stage_late_s = [&](int t) {   // S, dS', dO, W^T
        if (t < ntask) {
            const int64_t x = t;   // the tile index bh * NC + n
            const int n2 = t % NC, c2 = min(C, T - n2 * C);
            const int64_t r2 = (int64_t)(t / NC) * T + (int64_t)n2 * C;
            stage_rows(sb0 + OFF_M, Sb + x * D * D, D * 2, D * 2, LD * 2, D, D, tid0, 256);
            stage_rows(sb0 + OFF_DM, dSb + x * D * D, D * 2, D * 2, LD * 2, D, D, tid0, 256);
            stage_rows(sb0 + OFF_O, dout + r2 * D, D * 2, D * 2, LD * 2, C, c2, tid0, 256);
            stage_rows(sb0 + OFF_W, Wt + x * D * C, C * 2, C * 2, LC * 2, D, D, tid0, 256);
            if (tid0 == 0) {   // dR and v go through registers: towards L2 for now
                l2_prefetch(dR + r2 * D, (uint32_t)c2 * D * 4);
                l2_prefetch(v + r2 * D, (uint32_t)c2 * D * 2);
            }
        }
        cp_async_commit();
    };
    auto stage_late_qk = [&](int t, int slot) {   // q, k into slot 0 or 1 (alternating chunks)
        if (t < ntask) {
            const int n2 = t % NC, c2 = min(C, T - n2 * C);
            const int64_t r2 = (int64_t)(t / NC) * T + (int64_t)n2 * C;
            stage_rows(sb0 + (slot ? OFF_Q2 : OFF_Q), q + r2 * D, D * 2, D * 2, LD * 2, C, c2, tid0, 256);
            stage_rows(sb0 + (slot ? OFF_K2 : OFF_K), k + r2 * D, D * 2, D * 2, LD * 2, C, c2, tid0, 256);
        }
        cp_async_commit();
    };
    stage_late_s(blockIdx.x);
    stage_late_qk(blockIdx.x, 0);
    for (int task = blockIdx.x, it = 0; task < ntask; task += gridDim.x, ++it) {
        const int n = task % NC, bh = task / NC;
        const uint32_t oq = (it & 1) ? OFF_Q2 : OFF_Q, ok = (it & 1) ? OFF_K2 : OFF_K;   // this chunk's q, k
        const int t0 = n * C, c = min(C, T - t0);
        const int64_t row0 = (int64_t)bh * T + t0;
        const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, t4 = lane & 3;
        const uint32_t sb = sm100::smem_u32(smb);
        float *gs = reinterpret_cast<float *>(smb + OFF_SC);
        float *bs = gs + C, *dbp = bs + C, *dbt = dbp + C, *rq = dbt + C, *rk = rq + C, *rz = rk + C;
        float *vdr = rz + C, *red = vdr + C;

        // ---- 0. loads: every tile is on its way since the previous chunk (by cp.async into
        //         shared memory as soon as that chunk was done with it); dR
        //         (rounded to bf16 on the way), v and beta through registers for dv and v.dR
        {
            float4 fr[8];
            uint2 fv[8];
            float br[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {   // 2048 float4 per C x 128 fp32 tile: warp w, row w + 8u
                const int idx = tid + 256 * u, r = idx >> 5, col = (idx & 31) * 4;
                const bool in = r < c;
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                fr[u] = in ? __ldg(reinterpret_cast<const float4 *>(dR + (row0 + r) * D + col)) : z;
                fv[u] = in ? __ldg(reinterpret_cast<const uint2 *>(v + (row0 + r) * D + col)) : make_uint2(0u, 0u);
                br[u] = in ? beta[row0 + r] : 0.f;
            }
            for (int r = tid; r < C; r += 256) {
                gs[r] = r < c ? gamma[row0 + r] : 1.f;
                bs[r] = r < c ? beta[row0 + r] : 0.f;
                dbp[r] = dbt[r] = rq[r] = rk[r] = rz[r] = 0.f;
            }
            if (tid == 0) red[0] = 0.f;
            // dv = diag(beta) dR (from the fp32 dR) and v_r . dR_r, one warp per row
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int idx = tid + 256 * u, r = idx >> 5, col = (idx & 31) * 4;
                const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&fv[u].x));
                const float2 v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&fv[u].y));
                float p = fmaf(v01.x, fr[u].x, fmaf(v01.y, fr[u].y, fmaf(v23.x, fr[u].z, v23.y * fr[u].w)));
                for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
                if (lane == 0) vdr[r] = p;
                if (r < c)
                    *reinterpret_cast<uint2 *>(dv_out + (row0 + r) * D + col) =
                        make_uint2(pack_bf2(br[u] * fr[u].x, br[u] * fr[u].y), pack_bf2(br[u] * fr[u].z, br[u] * fr[u].w));
                *reinterpret_cast<uint2 *>(smb + OFF_R + 2 * (r * LD + col)) =
                    make_uint2(pack_bf2(fr[u].x, fr[u].y), pack_bf2(fr[u].z, fr[u].w));
            }
            cp_async_wait0();
            __syncthreads();   // the copies have landed; red[0] and the row sums are zeroed
            stage_late_qk(task + (int)gridDim.x, (it + 1) & 1);   // the next chunk's q, k: the other slot
            float mdm = 0.f;   // this thread's share of <M, dM'>, from the bf16 copies
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int idx = tid + 256 * u, r = idx >> 4, col = (idx & 15) * 8;
                float fm[8], fd[8];
                widen16(*reinterpret_cast<const uint4 *>(smb + OFF_M + 2 * (r * LD + col)), fm,
                        (const __nv_bfloat16 *)nullptr);
                widen16(*reinterpret_cast<const uint4 *>(smb + OFF_DM + 2 * (r * LD + col)), fd,
                        (const __nv_bfloat16 *)nullptr);
#pragma unroll
                for (int e = 0; e < 8; ++e) mdm = fmaf(fm[e], fd[e], mdm);
            }
            for (int off = 16; off > 0; off >>= 1) mdm += __shfl_xor_sync(0xffffffffu, mdm, off);
            if (lane == 0) atomicAdd(&red[0], mdm);
        }

        // ---- 1. position pairs: dP = dO W^T, dRW = dR W^T (rows mr .. mr + 15, columns nc .. nc + 31)
        {
            const int mr = 16 * (warp >> 1), nc = 32 * (warp & 1);
            float ap[4][4], ar[4][4], xq[4][4], xk[4][4];
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int e = 0; e < 4; ++e) ap[x][e] = ar[x][e] = xq[x][e] = xk[x][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t ao[4], aq[4];
                ldsm_x4(ao, a_addr(sb + OFF_O, LD, mr, 16 * kk, lane));
                ldsm_x4(aq, a_addr(sb + OFF_R, LD, mr, 16 * kk, lane));
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t bw[4];
                    ldsm_x4_t(bw, bt_addr(sb + OFF_W, LC, nc + 16 * np, 16 * kk, lane));   // W^T [j][s]
                    mma16816(ap[2 * np], ao, bw[0], bw[1]);
                    mma16816(ap[2 * np + 1], ao, bw[2], bw[3]);
                    mma16816(ar[2 * np], aq, bw[0], bw[1]);
                    mma16816(ar[2 * np + 1], aq, bw[2], bw[3]);
                }
            }
            // Q K^T and K K^T again (exact products of the bf16 inputs): the P and D o K K^T
            // of the pair terms, without a round trip through memory; the two tiles wholly
            // above the diagonal skip them
            if (nc <= mr + 15) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t a_q[4], a_k[4];
                    ldsm_x4(a_q, a_addr(sb + oq, LD, mr, 16 * kk, lane));
                    ldsm_x4(a_k, a_addr(sb + ok, LD, mr, 16 * kk, lane));
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        uint32_t b[4];
                        ldsm_x4(b, b_addr(sb + ok, LD, nc + 16 * np, 16 * kk, lane));
                        mma16816(xq[2 * np], a_q, b[0], b[1]);
                        mma16816(xq[2 * np + 1], a_q, b[2], b[3]);
                        mma16816(xk[2 * np], a_k, b[0], b[1]);
                        mma16816(xk[2 * np + 1], a_k, b[2], b[3]);
                    }
                }
            }
            // FP = dP o D, FA = dA o beta D (dA = -dRW), the db and dbeta pair terms
            float re[2] = {0.f, 0.f}, rt[2] = {0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                float ce[2] = {0.f, 0.f};
#pragma unroll
                for (int h = 0; h < 2; ++h) {   // rows gq, gq + 8
                    const int r = mr + gq + 8 * h, s0 = nc + 8 * nt + 2 * t4;
                    float fp[2] = {0.f, 0.f}, fa[2] = {0.f, 0.f};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int s = s0 + e;
                        if (r < c && s <= r) {
                            const float Dv = __fdividef(gs[r], gs[s]);
                            const float dP = ap[nt][2 * h + e];
                            fp[e] = dP * Dv;
                            float ee = dP * (Dv * xq[nt][2 * h + e]);   // dP P
                            if (s < r) {
                                const float dA = -ar[nt][2 * h + e], dkk = Dv * xk[nt][2 * h + e];
                                fa[e] = dA * bs[r] * Dv;
                                ee = fmaf(dA * bs[r], dkk, ee);
                                rt[h] = fmaf(dA, dkk, rt[h]);
                            }
                            re[h] += ee;
                            ce[e] -= ee;
                        }
                    }
                    *reinterpret_cast<uint32_t *>(smb + OFF_FP + 2 * (r * LC + s0)) = pack_bf2(fp[0], fp[1]);
                    *reinterpret_cast<uint32_t *>(smb + OFF_FA + 2 * (r * LC + s0)) = pack_bf2(fa[0], fa[1]);
                }
                // column sums over the 8 row lanes (gq) sharing the column
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float x = ce[e];
                    x += __shfl_xor_sync(0xffffffffu, x, 4);
                    x += __shfl_xor_sync(0xffffffffu, x, 8);
                    x += __shfl_xor_sync(0xffffffffu, x, 16);
                    const int s = nc + 8 * nt + 2 * t4 + e;
                    if (gq == 0 && s < c) atomicAdd(&dbp[s], x);
                }
            }
            // row sums over the 4 column lanes (t4) sharing the row
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float x = re[h], y = rt[h];
                x += __shfl_xor_sync(0xffffffffu, x, 1);
                x += __shfl_xor_sync(0xffffffffu, x, 2);
                y += __shfl_xor_sync(0xffffffffu, y, 1);
                y += __shfl_xor_sync(0xffffffffu, y, 2);
                const int r = mr + gq + 8 * h;
                if (t4 == 0 && r < c) {
                    atomicAdd(&dbp[r], x);
                    atomicAdd(&dbt[r], y);
                }
            }
        }
        __syncthreads();   // FP and FA are in shared memory

        // ---- 2. state terms (rows mr .. mr + 31, key columns nc .. nc + 31):
        //         X1 = dO M^T, X2 = dR M^T, X3 = W dM'^T
        const int mr = 32 * (warp >> 2), nc = 32 * (warp & 3);
        float x1[2][4][4], x2[2][4][4], x3[2][4][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
                for (int e = 0; e < 4; ++e) x1[a][b][e] = x2[a][b][e] = x3[a][b][e] = 0.f;
#pragma unroll 2
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t ao[2][4], aq[2][4], aw[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                ldsm_x4(ao[mt], a_addr(sb + OFF_O, LD, mr + 16 * mt, 16 * kk, lane));
                ldsm_x4(aq[mt], a_addr(sb + OFF_R, LD, mr + 16 * mt, 16 * kk, lane));
                ldsm_x4_t(aw[mt], at_addr(sb + OFF_W, LC, mr + 16 * mt, 16 * kk, lane));
            }
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bm[4], bd[4];   // the states are value-major: S[j][i] = M[i][j]
                ldsm_x4_t(bm, bt_addr(sb + OFF_M, LD, nc + 16 * np, 16 * kk, lane));
                ldsm_x4_t(bd, bt_addr(sb + OFF_DM, LD, nc + 16 * np, 16 * kk, lane));
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    mma16816(x1[mt][2 * np], ao[mt], bm[0], bm[1]);
                    mma16816(x1[mt][2 * np + 1], ao[mt], bm[2], bm[3]);
                    mma16816(x2[mt][2 * np], aq[mt], bm[0], bm[1]);
                    mma16816(x2[mt][2 * np + 1], aq[mt], bm[2], bm[3]);
                    mma16816(x3[mt][2 * np], aw[mt], bd[0], bd[1]);
                    mma16816(x3[mt][2 * np + 1], aw[mt], bd[2], bd[3]);
                }
            }
        }
        // row dots q.(M dO), k.(M dR), k.(dM' w) over this warp's 32 key columns (the four
        // column warps add up in shared memory); then the state terms of dQ (x1) and dK (x2)
        {
            const float gC = gs[c - 1];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = mr + 16 * mt + gq + 8 * h;
                    float pq = 0.f, pk = 0.f, pz = 0.f;
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        const int i = nc + 8 * nt + 2 * t4;
                        const float2 qf = __bfloat1622float2(
                            *reinterpret_cast<const __nv_bfloat162 *>(smb + oq + 2 * (r * LD + i)));
                        const float2 kf = __bfloat1622float2(
                            *reinterpret_cast<const __nv_bfloat162 *>(smb + ok + 2 * (r * LD + i)));
                        pq = fmaf(qf.x, x1[mt][nt][2 * h], fmaf(qf.y, x1[mt][nt][2 * h + 1], pq));
                        pk = fmaf(kf.x, x2[mt][nt][2 * h], fmaf(kf.y, x2[mt][nt][2 * h + 1], pk));
                        pz = fmaf(kf.x, x3[mt][nt][2 * h], fmaf(kf.y, x3[mt][nt][2 * h + 1], pz));
                    }
                    pq += __shfl_xor_sync(0xffffffffu, pq, 1);
                    pq += __shfl_xor_sync(0xffffffffu, pq, 2);
                    pk += __shfl_xor_sync(0xffffffffu, pk, 1);
                    pk += __shfl_xor_sync(0xffffffffu, pk, 2);
                    pz += __shfl_xor_sync(0xffffffffu, pz, 1);
                    pz += __shfl_xor_sync(0xffffffffu, pz, 2);
                    if (t4 == 0 && r < c) {
                        atomicAdd(&rq[r], pq);
                        atomicAdd(&rk[r], pk);
                        atomicAdd(&rz[r], pz);
                    }
                    const float gr = gs[r], sc = __fdividef(gC, gr), gb = gr * bs[r];
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            x1[mt][nt][2 * h + e] *= gr;
                            x2[mt][nt][2 * h + e] = fmaf(sc, x3[mt][nt][2 * h + e], -gb * x2[mt][nt][2 * h + e]);
                        }
                }
        }

        __syncthreads();                         // S and dS' are read: the next chunk's
        stage_late_s(task + (int)gridDim.x);

        // ---- 3. in-chunk terms: dQ += FP K,  dK += FP^T Q + FA K + FA^T K
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
            uint32_t afp[2][4], afpt[2][4], afa[2][4], afat[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                ldsm_x4(afp[mt], a_addr(sb + OFF_FP, LC, mr + 16 * mt, 16 * ks, lane));
                ldsm_x4_t(afpt[mt], at_addr(sb + OFF_FP, LC, mr + 16 * mt, 16 * ks, lane));
                ldsm_x4(afa[mt], a_addr(sb + OFF_FA, LC, mr + 16 * mt, 16 * ks, lane));
                ldsm_x4_t(afat[mt], at_addr(sb + OFF_FA, LC, mr + 16 * mt, 16 * ks, lane));
            }
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t bk[4], bq[4];
                ldsm_x4_t(bk, bt_addr(sb + ok, LD, nc + 16 * np, 16 * ks, lane));
                ldsm_x4_t(bq, bt_addr(sb + oq, LD, nc + 16 * np, 16 * ks, lane));
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int nt = 2 * np + hh;
                        const uint32_t k0 = bk[2 * hh], k1 = bk[2 * hh + 1], q0 = bq[2 * hh], q1 = bq[2 * hh + 1];
                        mma16816(x1[mt][nt], afp[mt], k0, k1);
                        mma16816(x2[mt][nt], afpt[mt], q0, q1);
                        mma16816(x2[mt][nt], afa[mt], k0, k1);
                        mma16816(x2[mt][nt], afat[mt], k0, k1);
                    }
            }
        }

        // ---- 4. dQ and dK through shared memory (into the dead FP, FA and dR tiles) into
        //         16-byte stores; then dbeta, db and dg per row
        __syncthreads();
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = mr + 16 * mt + gq + 8 * h, i = nc + 8 * nt + 2 * t4;
                    *reinterpret_cast<uint32_t *>(smb + OFF_FP + 2 * (r * LD + i)) =
                        pack_bf2(x1[mt][nt][2 * h], x1[mt][nt][2 * h + 1]);
                    *reinterpret_cast<uint32_t *>(smb + OFF_R + 2 * (r * LD + i)) =
                        pack_bf2(x2[mt][nt][2 * h], x2[mt][nt][2 * h + 1]);
                }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = tid + 256 * u, r = idx >> 4, col = (idx & 15) * 8;
            if (r < c) {
                *reinterpret_cast<uint4 *>(dq + (row0 + r) * D + col) =
                    *reinterpret_cast<const uint4 *>(smb + OFF_FP + 2 * (r * LD + col));
                *reinterpret_cast<uint4 *>(dk_out + (row0 + r) * D + col) =
                    *reinterpret_cast<const uint4 *>(smb + OFF_R + 2 * (r * LD + col));
            }
        }
        if (warp == 0) {
            const float gC = gs[c - 1];
            float zsum = 0.f;
            float db[2] = {0.f, 0.f};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = 2 * lane + e;
                if (r < c) {
                    dbeta[row0 + r] = dbt[r] + vdr[r] - gs[r] * rk[r];
                    const float z = gC / gs[r] * rz[r];
                    zsum += z;
                    db[e] = dbp[r] + gs[r] * rq[r] - gs[r] * bs[r] * rk[r] - z;
                }
            }
            for (int off = 16; off > 0; off >>= 1) zsum += __shfl_xor_sync(0xffffffffu, zsum, off);
            const float last = zsum + gC * red[0];
#pragma unroll
            for (int e = 0; e < 2; ++e)
                if (2 * lane + e == c - 1) db[e] += last;
            float suf = db[0] + db[1];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, suf, off);
                if (lane + off < 32) suf += y;
            }
            const float dl[2] = {suf, suf - db[0]};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = 2 * lane + e;
                if (r < c) dg[row0 + r] = dl[e] * dlog_alpha_dg(g[row0 + r], d);
            }
        }
        __syncthreads();   // shared memory is free for the next chunk
    }
}

// x = hi + lo in bf16 pairs
__device__ __forceinline__ void split_bf2(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = pack_bf2(a - hf.x, b - hf.y);
}


// ---------------------------------------------------------------- chunk tiles, warp MMA
// The chunk tiles of the bf16 d = 128, chunk-64 shape: Q K^T and K K^T on warp MMAs
// (bf16 inputs, exact products, fp32 sums), T = (I + A)^-1 solved blockwise in fp32
// (the four 16 x 16 diagonal blocks a column per lane, then the off-diagonal blocks
// by distance from the diagonal: T_ij = -T_ii sum_{m=j}^{i-1} A_im T_mj), and
// U = (T diag(beta)) V, Wk = (T diag(beta gamma)) K on warp MMAs with the fp32 left
// factors as bf16 hi + lo pairs (v and k exact).  Outputs: T and P as bf16 tiles for
// the reverse chain (TPb: per chunk T then P, C x C each), U (fp32) and Wk as bf16 rows
// (Wk2) for the forward state pass; the per-chunk kernel forms its fp32 P and D o K K^T
// itself from q and k.
namespace mt {
constexpr int C = 64, DK = 128, LD = DK + 8, LA = C + 4, LC = C + 8;
constexpr uint32_t OFF_K = 0, OFF_V = OFF_K + C * LD * 2, OFF_R1 = OFF_V + C * LD * 2,
                   R_BYTES = 2 * C * LC * 2, OFF_R2 = OFF_R1 + R_BYTES, OFF_X = OFF_R2 + R_BYTES,
                   OFF_G = OFF_X + 3 * 16 * 20 * 4;
constexpr uint32_t SMEM = OFF_G + 2 * C * 4;
static_assert(C * LD * 2 <= R_BYTES && C * LA * 4 <= R_BYTES, "region 1 holds q, then A");
}  // namespace mt

// T_ij = -T_ii sum_{m=j}^{i-1} A_im T_mj for one 16 x 16 block, by one warp: lane owns
// row lane / 2, columns 8 (lane % 2) .. + 7; X goes through the warp's scratch tile.
__device__ __forceinline__ void solve_offdiag(const float *As, float *Ts, float *Xs, int i, int j,
                                              int lane) {
    using namespace mt;
    const int rr = lane >> 1, cc = 8 * (lane & 1);
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.f;
    for (int m = j; m < i; ++m) {
#pragma unroll 4
        for (int q = 0; q < 16; ++q) {
            const float a = As[(16 * i + rr) * LA + 16 * m + q];
            const float4 t0 = *reinterpret_cast<const float4 *>(Ts + (16 * m + q) * LA + 16 * j + cc);
            const float4 t1 = *reinterpret_cast<const float4 *>(Ts + (16 * m + q) * LA + 16 * j + cc + 4);
            x[0] = fmaf(a, t0.x, x[0]); x[1] = fmaf(a, t0.y, x[1]);
            x[2] = fmaf(a, t0.z, x[2]); x[3] = fmaf(a, t0.w, x[3]);
            x[4] = fmaf(a, t1.x, x[4]); x[5] = fmaf(a, t1.y, x[5]);
            x[6] = fmaf(a, t1.z, x[6]); x[7] = fmaf(a, t1.w, x[7]);
        }
    }
    *reinterpret_cast<float4 *>(Xs + rr * 20 + cc) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4 *>(Xs + rr * 20 + cc + 4) = make_float4(x[4], x[5], x[6], x[7]);
    __syncwarp();
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll 4
    for (int q = 0; q < 16; ++q) {
        const float a = Ts[(16 * i + rr) * LA + 16 * i + q];
        const float4 x0 = *reinterpret_cast<const float4 *>(Xs + q * 20 + cc);
        const float4 x1 = *reinterpret_cast<const float4 *>(Xs + q * 20 + cc + 4);
        y[0] = fmaf(a, x0.x, y[0]); y[1] = fmaf(a, x0.y, y[1]);
        y[2] = fmaf(a, x0.z, y[2]); y[3] = fmaf(a, x0.w, y[3]);
        y[4] = fmaf(a, x1.x, y[4]); y[5] = fmaf(a, x1.y, y[5]);
        y[6] = fmaf(a, x1.z, y[6]); y[7] = fmaf(a, x1.w, y[7]);
    }
    *reinterpret_cast<float4 *>(Ts + (16 * i + rr) * LA + 16 * j + cc) = make_float4(-y[0], -y[1], -y[2], -y[3]);
    *reinterpret_cast<float4 *>(Ts + (16 * i + rr) * LA + 16 * j + cc + 4) = make_float4(-y[4], -y[5], -y[6], -y[7]);
}

__global__ void __launch_bounds__(256, 2)
bwd_tiles_mma_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                     const __nv_bfloat16 *__restrict__ v, const float *__restrict__ gamma,
                     const float *__restrict__ beta, __nv_bfloat16 *__restrict__ TPb,
                     float *__restrict__ U, __nv_bfloat16 *__restrict__ Wk2, int T, int want_uw,
                     const float *__restrict__ g, float d, float *__restrict__ tsc) {
    using namespace mt;
    using sm100::ldsm_x4;
    using sm100::ldsm_x4_t;
    using sm100::mma16816;
    extern __shared__ __align__(16) uint8_t smb[];
    const int n = blockIdx.x, bh = blockIdx.y;
    const int NC = (T + C - 1) / C;
    const int t0 = n * C, c = min(C, T - t0);
    const int64_t row0 = (int64_t)bh * T + t0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, t4 = lane & 3;
    const uint32_t sb = sm100::smem_u32(smb);
    float *As = reinterpret_cast<float *>(smb + OFF_R1);   // after the pair products
    float *Ts = reinterpret_cast<float *>(smb + OFF_R2);
    float *gs = reinterpret_cast<float *>(smb + OFF_G), *bs = gs + C;
    const int64_t tb = ((int64_t)bh * NC + n) * C * C;
    __nv_bfloat16 *Tb = TPb + 2 * tb, *Pb = Tb + C * C;

    {   // q (into region 1), k, v as given; rows past the chunk's end zero
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        uint4 bq[4], bk[4], bv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = tid + 256 * u, r = idx >> 4, col = (idx & 15) * 8;
            const bool in = r < c;
            bq[u] = in ? ld16(q + (row0 + r) * DK + col) : z;
            bk[u] = in ? ld16(k + (row0 + r) * DK + col) : z;
            bv[u] = (in && want_uw) ? ld16(v + (row0 + r) * DK + col) : z;   // v only feeds U
        }
        if (tid < C) {
            gs[tid] = tid < c ? gamma[row0 + tid] : 1.f;
            bs[tid] = tid < c ? beta[row0 + tid] : 0.f;
            if (tsc) {   // the chunk's row scalars for the per-chunk gradient kernel
                float *blk = tsc + ((int64_t)bh * NC + n) * 4 * C;
                blk[tid] = gs[tid];
                blk[C + tid] = 1.0f / gs[tid];
                blk[2 * C + tid] = bs[tid];
                blk[3 * C + tid] = tid < c ? dlog_alpha_dg(g[row0 + tid], d) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = tid + 256 * u, r = idx >> 4, col = (idx & 15) * 8;
            *reinterpret_cast<uint4 *>(smb + OFF_R1 + 2 * (r * LD + col)) = bq[u];
            *reinterpret_cast<uint4 *>(smb + OFF_K + 2 * (r * LD + col)) = bk[u];
            *reinterpret_cast<uint4 *>(smb + OFF_V + 2 * (r * LD + col)) = bv[u];
        }
    }
    __syncthreads();

    // Q K^T and K K^T: warp tile rows 16 (w >> 1), columns 32 (w & 1) (the two tiles
    // wholly above the diagonal skip the products)
    const int mb = warp >> 1, nh = warp & 1;
    float aq[4][4], ak[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int e = 0; e < 4; ++e) aq[x][e] = ak[x][e] = 0.f;
    if (32 * nh <= 16 * mb + 15) {
#pragma unroll 2
        for (int kk = 0; kk < DK / 16; ++kk) {
            uint32_t a_q[4], a_k[4];
            ldsm_x4(a_q, a_addr(sb + OFF_R1, LD, 16 * mb, 16 * kk, lane));
            ldsm_x4(a_k, a_addr(sb + OFF_K, LD, 16 * mb, 16 * kk, lane));
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t b[4];
                ldsm_x4(b, b_addr(sb + OFF_K, LD, 32 * nh + 16 * np, 16 * kk, lane));
                mma16816(aq[2 * np], a_q, b[0], b[1]);
                mma16816(aq[2 * np + 1], a_q, b[2], b[3]);
                mma16816(ak[2 * np], a_k, b[0], b[1]);
                mma16816(ak[2 * np + 1], a_k, b[2], b[3]);
            }
        }
    }
    __syncthreads();   // q is read: region 1 takes A
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = 16 * mb + gq + 8 * h, s0 = 32 * nh + 8 * nt + 2 * t4;
            float p[2], dd[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int s = s0 + e;
                const float D = __fdividef(gs[r], gs[s]);
                p[e] = (r < c && s <= r) ? D * aq[nt][2 * h + e] : 0.f;
                dd[e] = (r < c && s < r) ? D * ak[nt][2 * h + e] : 0.f;
            }
            *reinterpret_cast<uint32_t *>(Pb + sw_elem(r, s0)) = pack_bf2(p[0], p[1]);
            *reinterpret_cast<float2 *>(As + r * LA + s0) = make_float2(bs[r] * dd[0], bs[r] * dd[1]);
        }
    // the blocks of T above the diagonal are zero
    for (int x = tid; x < 6 * 256; x += 256) {
        const int b = x >> 8, e = x & 255;   // blocks (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
        const int bi = b < 3 ? 0 : (b < 5 ? 1 : 2), bj = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
        Ts[(16 * bi + (e >> 4)) * LA + 16 * bj + (e & 15)] = 0.f;
    }
    __syncthreads();
    // diagonal blocks: warp 0 blocks 0, 1, warp 1 blocks 2, 3; lane % 16 = the column
    if (warp < 2) {
        const int b = 2 * warp + (lane >> 4), s = lane & 15;
        const float *Ab = As + 16 * b * LA + 16 * b;
        float t[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float a = 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) a = fmaf(Ab[r * LA + m], t[m], a);
            t[r] = r == s ? 1.f : (r > s ? -a : 0.f);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Ts[(16 * b + r) * LA + 16 * b + s] = t[r];
    }
    __syncthreads();
    float *Xs = reinterpret_cast<float *>(smb + OFF_X) + (warp < 3 ? warp : 0) * 16 * 20;
    if (warp < 3) solve_offdiag(As, Ts, Xs, warp + 1, warp, lane);   // (1,0) (2,1) (3,2)
    __syncthreads();
    if (warp < 2) solve_offdiag(As, Ts, Xs, warp + 2, warp, lane);   // (2,0) (3,1)
    __syncthreads();
    if (warp == 0) solve_offdiag(As, Ts, Xs, 3, 0, lane);            // (3,0)
    __syncthreads();

    // T out (fp32); T diag(beta) and T diag(beta gamma) as hi + lo pairs into regions 1, 2
    {
        float4 tv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = tid + 256 * u, r = idx >> 4, s = (idx & 15) * 4;
            tv[u] = *reinterpret_cast<const float4 *>(Ts + r * LA + s);
            *reinterpret_cast<uint2 *>(Tb + sw_elem(r, s)) =
                make_uint2(pack_bf2(tv[u].x, tv[u].y), pack_bf2(tv[u].z, tv[u].w));
        }
        // U and Wk feed only the forward-state recomputation, which saved states replace
        // (want_uw is uniform over the CTA: every thread leaves here together)
        if (!want_uw) return;
        __syncthreads();   // T is read: region 2 takes T diag(beta gamma)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = tid + 256 * u, r = idx >> 4, s = (idx & 15) * 4;
            const float tt[4] = {tv[u].x, tv[u].y, tv[u].z, tv[u].w};
            float xb[4], xg[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                xb[e] = tt[e] * bs[s + e];
                xg[e] = xb[e] * gs[s + e];
            }
            uint32_t h0, l0, h1, l1;
            const uint32_t o = 2 * (r * LC + s);
            split_bf2(xb[0], xb[1], h0, l0);
            split_bf2(xb[2], xb[3], h1, l1);
            *reinterpret_cast<uint2 *>(smb + OFF_R1 + o) = make_uint2(h0, h1);
            *reinterpret_cast<uint2 *>(smb + OFF_R1 + C * LC * 2 + o) = make_uint2(l0, l1);
            split_bf2(xg[0], xg[1], h0, l0);
            split_bf2(xg[2], xg[3], h1, l1);
            *reinterpret_cast<uint2 *>(smb + OFF_R2 + o) = make_uint2(h0, h1);
            *reinterpret_cast<uint2 *>(smb + OFF_R2 + C * LC * 2 + o) = make_uint2(l0, l1);
        }
    }
    __syncthreads();

    // U = (T diag(beta)) V, Wk = (T diag(beta gamma)) K: warp tile rows 16 (w >> 1),
    // columns 64 (w & 1); T is lower triangular, so row block mb meets k blocks <= mb
#pragma unroll 1
    for (int pr = 0; pr < 2; ++pr) {
        const uint32_t ah_base = sb + (pr == 0 ? OFF_R1 : OFF_R2), al_base = ah_base + C * LC * 2;
        const uint32_t b_base = sb + (pr == 0 ? OFF_V : OFF_K);
        float acc[8][4];
#pragma unroll
        for (int x = 0; x < 8; ++x)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[x][e] = 0.f;
        for (int ks = 0; ks <= mb; ++ks) {
            uint32_t ah[4], al[4];
            ldsm_x4(ah, a_addr(ah_base, LC, 16 * mb, 16 * ks, lane));
            ldsm_x4(al, a_addr(al_base, LC, 16 * mb, 16 * ks, lane));
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b[4];
                ldsm_x4_t(b, bt_addr(b_base, LD, 64 * nh + 16 * np, 16 * ks, lane));
                mma16816(acc[2 * np], ah, b[0], b[1]);
                mma16816(acc[2 * np + 1], ah, b[2], b[3]);
                mma16816(acc[2 * np], al, b[0], b[1]);
                mma16816(acc[2 * np + 1], al, b[2], b[3]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = 16 * mb + gq + 8 * h, j = 64 * nh + 8 * nt + 2 * t4;
                if (r >= c) continue;
                if (pr == 0) {
                    *reinterpret_cast<float2 *>(U + (row0 + r) * DK + j) =
                        make_float2(acc[nt][2 * h], acc[nt][2 * h + 1]);
                } else {
                    *reinterpret_cast<uint32_t *>(Wk2 + (row0 + r) * DK + j) =
                        pack_bf2(acc[nt][2 * h], acc[nt][2 * h + 1]);
                }
            }
    }
}

// ---------------------------------------------------------------- value-column chains
// The two sequential passes of the bf16 d = 128, chunk-64 shape, value-column parallel:
// the state's value columns never mix, so warp w of a CTA owns 16 of them (the CTA 64,
// grid (dv / 64, BH), one CTA per SM) and keeps its 16 x 128 slice of the state
// TRANSPOSED in fp32 MMA accumulator fragments.  The accumulator fragment of a 16-row
// tile is the A fragment of the next product over its columns (rows g, g + 8; columns
// 2t, 2t + 1 and 2t + 8, 2t + 9 of two adjacent 8-column tiles), so a chunk's products
// chain inside the warp without shared memory or barriers.  The chunk's shared inputs
// arrive by cp.async into padded, double-buffered shared memory (the next chunk's copy
// runs under this chunk's products): two barriers per chunk.  The chunk states go out
// value-major in bf16, S[j][i] = M[i][j], for the per-chunk gradients.

namespace vc {
constexpr int C = 64, DK = 128, NW = 4, NT = 32 * NW, DSC = 16 * NW, LD = DK + 8, LC = C + 8;
// forward state stage: k, Wk (bf16 [C][LD]); U[:, slice] (fp32 [C][DSC + 4]); gamma
constexpr int LU = DSC + 4;
constexpr uint32_t F_K = 0, F_WH = F_K + C * LD * 2, F_U = F_WH + C * LD * 2,
                   F_G = F_U + C * LU * 4, F_STAGE = F_G + C * 4;
// reverse chain stage, filled by TMA and bulk copies: k, q (two 64-column slabs of [C rows]
// [128 B] each), P, T, dO[:, slice] ([C rows][128 B]), all with the 128-byte swizzle; then
// gamma and beta (the chunk's scalar block: 1 and 0 past its end)
constexpr uint32_t R_K = 0, R_Q = 16384, R_P = 32768, R_T = 40960, R_O = 49152, R_G = 57344, R_B = R_G + C * 4,
                   R_STAGE = 58368;
constexpr uint32_t R_TX = 2 * 16384 + 3 * 8192 + 2 * C * 4;   // bytes landing per stage
static_assert(F_STAGE % 16 == 0 && R_STAGE % 1024 == 0 && R_B + C * 4 <= R_STAGE, "stage layout");
// from saves, the idle forward-state stages hold a third reverse-chain stage and the four
// warps' store staging (8 KB each)
static_assert(R_STAGE + NW * 8192 <= 2 * F_STAGE, "third stage and staging");
}  // namespace vc

// Byte offset of element (row, col) (col a multiple of 8) of a tile of 64-column slabs
// ([rows][128 B] each, slab bytes apart) whose 16-byte chunks are swizzled by row: the
// layout TMA writes with the 128-byte swizzle, and in which eight consecutive rows of one
// column block fall in eight different bank groups.
__device__ __forceinline__ uint32_t sw_off(int row, int col, uint32_t slab) {
    return (uint32_t)(col >> 6) * slab + (uint32_t)row * 128u +
           ((((uint32_t)(col & 63) >> 3) ^ ((uint32_t)row & 7u)) << 4);
}
// at_addr, b_addr, bt_addr on such tiles
__device__ __forceinline__ uint32_t at_sw(uint32_t base, uint32_t slab, int R, int Kc, int lane) {
    return base + sw_off(Kc + (lane & 7) + (lane >> 4) * 8, R + ((lane >> 3) & 1) * 8, slab);
}
__device__ __forceinline__ uint32_t b_sw(uint32_t base, uint32_t slab, int N, int Kc, int lane) {
    return base + sw_off(N + (lane & 7) + (lane >> 4) * 8, Kc + ((lane >> 3) & 1) * 8, slab);
}
__device__ __forceinline__ uint32_t bt_sw(uint32_t base, uint32_t slab, int N, int Kc, int lane) {
    return base + sw_off(Kc + (lane & 7) + ((lane >> 3) & 1) * 8, N + (lane >> 4) * 8, slab);
}

// Sticky error word of this file's kernels (the reverse chain's bounded waits)
__device__ unsigned g_bwd_error_word = 0;
// Bounded wait that also gives up once *abort is raised (by another warp of the CTA);
// raises it itself (and the error word) when its own limit passes.
__device__ __noinline__ bool pass_wait_ab(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort) {
    if (sm100::mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = sm100::global_timer_ns();
    while (limit_ns > 0) {
        if (sm100::mbar_try_wait_hint(bar, parity, 20000)) return true;
        if (*abort) return false;
        if (sm100::global_timer_ns() - t0 > limit_ns) break;
    }
    *abort = 1;
    atomicOr(&g_bwd_error_word, kDevErrTimeout);
    return false;
}
// Bounded wait of one thread on an mbarrier phase: false (and the error word raised)
// once limit_ns pass; limit_ns = 0 gives up at once unless the phase is complete.
__device__ __noinline__ bool pass_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (sm100::mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = sm100::global_timer_ns();
    while (limit_ns > 0) {
        if (sm100::mbar_try_wait_hint(bar, parity, 20000)) return true;
        if (sm100::global_timer_ns() - t0 > limit_ns) break;
    }
    atomicOr(&g_bwd_error_word, kDevErrTimeout);
    return false;
}

// A fragment (k block kk) from a 16-row accumulator tile acc[2 kk], acc[2 kk + 1]
__device__ __forceinline__ void acc_to_a(const float (&x0)[4], const float (&x1)[4], uint32_t (&a)[4]) {
    a[0] = pack_bf2(x0[0], x0[1]);
    a[1] = pack_bf2(x0[2], x0[3]);
    a[2] = pack_bf2(x1[0], x1[1]);
    a[3] = pack_bf2(x1[2], x1[3]);
}
__device__ __forceinline__ void acc_to_a_split(const float (&x0)[4], const float (&x1)[4], uint32_t (&h)[4],
                                               uint32_t (&l)[4]) {
    split_bf2(x0[0], x0[1], h[0], l[0]);
    split_bf2(x0[2], x0[3], h[1], l[1]);
    split_bf2(x1[0], x1[1], h[2], l[2]);
    split_bf2(x1[2], x1[3], h[3], l[3]);
}

// Forward state: per chunk W^T = U^T - M^T Wk^T (M^T as hi + lo, Wk bf16: two products)
// and M^T <- gamma_C M^T + (W diag(gamma_C / gamma))^T K (W as hi + lo); writes W^T per
// chunk ([dv][C], bf16) and the state at every chunk start (value-major, bf16): the
// per-chunk gradients take both as bf16 operands.
__device__ __forceinline__ void
fwd_state_pass(uint8_t *smb, int tid, uint32_t bar_id, const __nv_bfloat16 *__restrict__ k, const float *__restrict__ gamma,
                        const float *__restrict__ U, const __nv_bfloat16 *__restrict__ Wk2,
                        const float *init, __nv_bfloat16 *__restrict__ Wt, __nv_bfloat16 *__restrict__ Sb,
                        int T, int dv) {
    using namespace vc;
    using sm100::ldsm_x4;
    using sm100::ldsm_x4_t;
    using sm100::mma16816;
    const int j0 = blockIdx.x * DSC, bh = blockIdx.y;
    const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, t4 = lane & 3;
    const uint32_t sb = sm100::smem_u32(smb);
    const int NC = (T + C - 1) / C;
    const int jw = j0 + 16 * warp;   // this warp's first value column
    auto issue = [&](int n) {
        if (n < NC) {
            const uint32_t st = sb + (uint32_t)(n & 1) * F_STAGE;
            const int c = min(C, T - n * C);
            const int64_t row0 = (int64_t)bh * T + (int64_t)n * C;
            stage_rows(st + F_K, k + row0 * DK, DK * 2, DK * 2, LD * 2, C, c, tid, NT);
            stage_rows(st + F_WH, Wk2 + row0 * DK, DK * 2, DK * 2, LD * 2, C, c, tid, NT);
            stage_rows(st + F_U, U + row0 * dv + j0, (int64_t)dv * 4, DSC * 4, LU * 4, C, c, tid, NT);
            if (tid < C) cp_async4(st + F_G + 4 * tid, gamma + row0 + (tid < c ? tid : 0), tid < c ? 4u : 0u);
        }
        cp_async_commit();
    };
    // M^T: rows jw + gq (+ 8), key columns 8 nt + 2 t4 (+ 1)
    float mt[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = 8 * nt + 2 * t4 + (e & 1), j = jw + gq + 8 * (e >> 1);
            mt[nt][e] = init ? init[((int64_t)bh * DK + i) * dv + j] : 0.f;
        }
    issue(0);
    issue(1);
    for (int n = 0; n < NC; ++n) {
        const int c = min(C, T - n * C);
        const uint32_t st = sb + (uint32_t)(n & 1) * F_STAGE;
        const float *gs = reinterpret_cast<const float *>(smb + (n & 1) * F_STAGE + F_G);
        const float *us = reinterpret_cast<const float *>(smb + (n & 1) * F_STAGE + F_U);
        {   // the state at this chunk's start, value-major bf16
            __nv_bfloat16 *dst = Sb + ((int64_t)bh * NC + n) * DK * dv;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    *reinterpret_cast<uint32_t *>(dst + (int64_t)(jw + gq + 8 * h) * DK + 8 * nt + 2 * t4) =
                        pack_bf2(mt[nt][2 * h], mt[nt][2 * h + 1]);
        }
        cp_async_wait1();
        sm100::named_sync(bar_id, NT);   // chunk n's stage has landed
        const float gC = gs[c - 1];
        // W^T (16 x 64): w from M^T hi, w2 from M^T lo
        float w[8][4], w2[8][4];
#pragma unroll
        for (int x = 0; x < 8; ++x)
#pragma unroll
            for (int e = 0; e < 4; ++e) w[x][e] = w2[x][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
            uint32_t ah[4], al[4];
            acc_to_a_split(mt[2 * kk], mt[2 * kk + 1], ah, al);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bh4[4];
                ldsm_x4(bh4, b_addr(st + F_WH, LD, 16 * np, 16 * kk, lane));
                mma16816(w[2 * np], ah, bh4[0], bh4[1]);
                mma16816(w[2 * np + 1], ah, bh4[2], bh4[3]);
                mma16816(w2[2 * np], al, bh4[0], bh4[1]);
                mma16816(w2[2 * np + 1], al, bh4[2], bh4[3]);
            }
        }
        // W = U - (w + w2), stored; then the columns scaled by gamma_C / gamma_r (this
        // lane's 16 rows r = 8 nt + 2 t4 + e, e < 2)
        float sc[8][2];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = 8 * nt + 2 * t4 + e;
                sc[nt][e] = r < c ? __fdividef(gC, gs[r]) : 0.f;
            }
        __nv_bfloat16 *wt = Wt + ((int64_t)bh * NC + n) * dv * C;   // W^T [j][r], bf16, zero past c
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = 8 * nt + 2 * t4, jl = 16 * warp + gq + 8 * h;
                const float x0 = us[r * LU + jl] - (w[nt][2 * h] + w2[nt][2 * h]);
                const float x1 = us[(r + 1) * LU + jl] - (w[nt][2 * h + 1] + w2[nt][2 * h + 1]);
                *reinterpret_cast<uint32_t *>(wt + (int64_t)(j0 + jl) * C + r) = pack_bf2(x0, x1);
                w[nt][2 * h] = x0 * sc[nt][0];
                w[nt][2 * h + 1] = x1 * sc[nt][1];
            }
        // M^T <- gamma_C M^T + (W diag(sc))^T K
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) mt[nt][e] *= gC;
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
            uint32_t ah[4], al[4];
            acc_to_a_split(w[2 * ks], w[2 * ks + 1], ah, al);
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t b[4];
                ldsm_x4_t(b, bt_addr(st + F_K, LD, 16 * np, 16 * ks, lane));
                mma16816(mt[2 * np], ah, b[0], b[1]);
                mma16816(mt[2 * np + 1], ah, b[2], b[3]);
                mma16816(mt[2 * np], al, b[0], b[1]);
                mma16816(mt[2 * np + 1], al, b[2], b[3]);
            }
        }
        sm100::named_sync(bar_id, NT);   // every warp of the pass is done with this stage
        issue(n + 2);
    }
}

// Reverse chain: per chunk dW^T = dO^T P + (dM'^T K^T) diag(gamma_C / gamma),
// dR^T = dW^T T (stored as dR [token][dv], fp32), and
// dM^T <- gamma_C dM'^T + (diag(gamma) dO)^T Q + (-diag(gamma beta) dR)^T K; writes dM'
// of every chunk (value-major bf16) and the initial state's gradient (fp32).  Thread 0
// of the pass fills the two stages by TMA (k, q, dO) and bulk copies (the swizzled T and
// P tiles, the chunk's scalar block); each warp's lane 0 waits (bounded) on the stage's
// mbarrier, and the warps leave together if a wait runs out.
__device__ __forceinline__ void
chain_pass(uint8_t *smb, int tid, uint32_t bar_id, const CUtensorMap *tm_q, const CUtensorMap *tm_k,
           const CUtensorMap *tm_o, const float *dfinal, const __nv_bfloat16 *__restrict__ TPb,
           float *__restrict__ dR, __nv_bfloat16 *__restrict__ dSb, float *dinit, int T, int dv,
           const float *__restrict__ rows, uint64_t limit_ns, uint8_t *stg, const CUtensorMap *tm_dr,
           const CUtensorMap *tm_ds, uint64_t *r_bar, volatile int *r_abort) {
    using namespace vc;
    using sm100::ldsm_x4;
    using sm100::ldsm_x4_t;
    using sm100::mma16816;
    // ext: another warp (reverse_loader) fills the stages, and this pass's warps hand
    // each stage back through its EMPTY barrier instead of meeting at named barriers
    const bool ext = stg != nullptr;
    const int j0 = blockIdx.x * DSC, bh = blockIdx.y;
    const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, t4 = lane & 3;
    const uint32_t sb = sm100::smem_u32(smb);
    const int NC = (T + C - 1) / C;
    const int jw = j0 + 16 * warp;
    // stages: three with the loader (the third in the idle forward-state area), else two
    const int NS = ext ? 3 : 2;
    auto bar = [&](int s) { return sm100::smem_u32(&r_bar[s]); };        // FULL of stage s
    auto ebar = [&](int s) { return sm100::smem_u32(&r_bar[3 + s]); };   // EMPTY of stage s
    int issued[2] = {0, 0};   // thread 0: loads issued per stage
    // Stage s takes chunk n (n < 0: nothing): lane 0 of each warp issues a share of the
    // copies (thread 0 first arms the barrier with all the bytes; a copy that lands
    // before that only leaves the phase waiting for the arrival).
    auto issue = [&](int s, int n) {
        if (n < 0 || lane != 0) return;
        const uint32_t st = sb + (uint32_t)s * R_STAGE, b = bar(s);
        const __nv_bfloat16 *tp = TPb + ((int64_t)bh * NC + n) * 2 * C * C;
        const float *blk = rows + ((int64_t)bh * NC + n) * 4 * C;
        if (warp == 0) {
            sm100::mbar_arrive_expect_tx(b, R_TX);
            sm100::tma_load_3d(st + R_K, tm_k, b, 0, n * C, bh);
            sm100::tma_load_3d(st + R_K + 8192, tm_k, b, 64, n * C, bh);
            ++issued[s];
        } else if (warp == 1) {
            sm100::tma_load_3d(st + R_Q, tm_q, b, 0, n * C, bh);
            sm100::tma_load_3d(st + R_Q + 8192, tm_q, b, 64, n * C, bh);
        } else if (warp == 2) {
            sm100::tma_load_3d(st + R_O, tm_o, b, j0, n * C, bh);
            sm100::bulk_load(st + R_T, tp, 8192, b);
        } else {
            sm100::bulk_load(st + R_P, tp + C * C, 8192, b);
            sm100::bulk_load(st + R_G, blk, C * 4, b);
            sm100::bulk_load(st + R_B, blk + 2 * C, C * 4, b);
        }
    };
    float dm[16][4];   // dM'^T: rows jw + gq (+ 8), key columns 8 nt + 2 t4 (+ 1)
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = 8 * nt + 2 * t4 + (e & 1), j = jw + gq + 8 * (e >> 1);
            dm[nt][e] = dfinal ? dfinal[((int64_t)bh * DK + i) * dv + j] : 0.f;
        }
    if (!ext) {
        if (tid == 0) {
            sm100::tma_prefetch_desc(tm_q);
            sm100::tma_prefetch_desc(tm_k);
            sm100::tma_prefetch_desc(tm_o);
        }
        issue(0, NC - 1);
        issue(1, NC - 2);
    }
    bool ok = true;
    for (int it = 0; it < NC; ++it) {
        const int n = NC - 1 - it, s = it % NS;
        const uint32_t ph = (uint32_t)(it / NS) & 1u;   // the stage's phase of this chunk
        const int c = min(C, T - n * C);
        const int64_t row0 = (int64_t)bh * T + (int64_t)n * C;
        const uint32_t st = sb + (uint32_t)s * R_STAGE;
        const float *gs = reinterpret_cast<const float *>(smb + s * R_STAGE + R_G);
        const float *bs = reinterpret_cast<const float *>(smb + s * R_STAGE + R_B);
        if (stg) {
            // dM' of this chunk through this warp's staging tile (16 value rows, two
            // 64-column slabs, 128-byte swizzle) and a tensor store; the staging is free
            // once the previous chunk's stores have read it
            if (lane == 0) sm100::bulk_wait_read_all();
            __syncwarp();
            const uint32_t ds = sm100::smem_u32(stg) + (uint32_t)warp * 8192u + 4096u;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t jl = (uint32_t)(gq + 8 * h);
                    const uint32_t addr = ds + (uint32_t)(nt >> 3) * 2048u + jl * 128u +
                                          ((((uint32_t)nt & 7u) ^ (jl & 7u)) << 4) + (uint32_t)t4 * 4u;
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(pack_bf2(dm[nt][2 * h], dm[nt][2 * h + 1]))
                                 : "memory");
                }
            sm100::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                const int x = bh * NC + n;
                sm100::tma_store_3d(tm_ds, ds, 0, jw, x);
                sm100::tma_store_3d(tm_ds, ds + 2048u, 64, jw, x);
                sm100::bulk_commit();
            }
        } else {   // dM' of this chunk, value-major bf16
            __nv_bfloat16 *dst = dSb + ((int64_t)bh * NC + n) * DK * dv;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    *reinterpret_cast<uint32_t *>(dst + (int64_t)(jw + gq + 8 * h) * DK + 8 * nt + 2 * t4) =
                        pack_bf2(dm[nt][2 * h], dm[nt][2 * h + 1]);
        }
        // the stage has landed (each warp's lane 0 waits); all warps leave together otherwise
        bool landed = true;
        if (ext) {   // each warp on its own; a wait that runs out raises the CTA's abort flag
            if (lane == 0) landed = pass_wait_ab(bar(s), ph, limit_ns, r_abort);
            if (!__shfl_sync(0xffffffffu, landed ? 1 : 0, 0)) {
                ok = false;
                break;
            }
        } else {
            if (lane == 0) landed = pass_wait(bar(s), ph, limit_ns);
            if (!sm100::named_and(bar_id, NT, landed)) {
                ok = false;
                break;
            }
        }
        const float gC = gs[c - 1];
        // the row scales of the combine and the state update (this lane's rows r = 8 nt +
        // 2 t4 + e, e < 2), formed before the products so that their loads and divisions
        // overlap the MMAs
        float sc[8][2], gb[8][2];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = 8 * nt + 2 * t4 + e;
                sc[nt][e] = r < c ? __fdividef(gC, gs[r]) : 0.f;
                gb[nt][e] = -gs[r] * bs[r];
            }
        // dO^T fragments (k = token) and their gamma-scaled copies
        uint32_t ao[4][4], ag[4][4];
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            ldsm_x4_t(ao[ks], at_sw(st + R_O, 8192, 16 * warp, 16 * ks, lane));
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int r = 16 * ks + 2 * t4 + 8 * (x >> 1);
                const float2 o = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ao[ks][x]));
                ag[ks][x] = pack_bf2(gs[r] * o.x, gs[r + 1] * o.y);
            }
        }
        // dW^T = dO^T P (+) dM'^T K^T, the second scaled by gamma_C / gamma_r per column r
        float a1[8][4], a2[8][4];
#pragma unroll
        for (int x = 0; x < 8; ++x)
#pragma unroll
            for (int e = 0; e < 4; ++e) a1[x][e] = a2[x][e] = 0.f;
#pragma unroll
        for (int np = 0; np < 4; ++np)
#pragma unroll
            for (int ks = np; ks < 4; ++ks) {   // P is lower triangular: P[m][r] = 0 for m < r
                uint32_t b[4];
                ldsm_x4_t(b, bt_sw(st + R_P, 8192, 16 * np, 16 * ks, lane));
                mma16816(a1[2 * np], ao[ks], b[0], b[1]);
                mma16816(a1[2 * np + 1], ao[ks], b[2], b[3]);
            }
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
            uint32_t a[4];
            acc_to_a(dm[2 * kk], dm[2 * kk + 1], a);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b[4];
                ldsm_x4(b, b_sw(st + R_K, 8192, 16 * np, 16 * kk, lane));
                mma16816(a2[2 * np], a, b[0], b[1]);
                mma16816(a2[2 * np + 1], a, b[2], b[3]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) a1[nt][e] = fmaf(sc[nt][e & 1], a2[nt][e], a1[nt][e]);
        // dR^T = dW^T T (T unit lower triangular)
#pragma unroll
        for (int x = 0; x < 8; ++x)
#pragma unroll
            for (int e = 0; e < 4; ++e) a2[x][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t a[4];
            acc_to_a(a1[2 * ks], a1[2 * ks + 1], a);
#pragma unroll
            for (int np = 0; np <= ks; ++np) {
                uint32_t b[4];
                ldsm_x4_t(b, bt_sw(st + R_T, 8192, 16 * np, 16 * ks, lane));
                mma16816(a2[2 * np], a, b[0], b[1]);
                mma16816(a2[2 * np + 1], a, b[2], b[3]);
            }
        }
        // dR out; -gamma beta dR as the A operand of the state update
        if (stg) {   // through this warp's staging tile ([64 rows][16 columns] fp32) and a tensor store
            const uint32_t dr = sm100::smem_u32(stg) + (uint32_t)warp * 8192u;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t r = (uint32_t)(8 * nt + 2 * t4 + (e & 1)), jl = (uint32_t)(gq + 8 * (e >> 1));
                    asm volatile("st.shared.f32 [%0], %1;" ::"r"(dr + r * 64u + jl * 4u), "f"(a2[nt][e]) : "memory");
                    a2[nt][e] *= gb[nt][e & 1];
                }
            sm100::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {   // rows past the sequence's end are clipped
                sm100::tma_store_3d(tm_dr, dr, jw, n * C, bh);
                sm100::bulk_commit();
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = 8 * nt + 2 * t4 + (e & 1), j = jw + gq + 8 * (e >> 1);
                    if (r < c) dR[(row0 + r) * dv + j] = a2[nt][e];
                    a2[nt][e] *= gb[nt][e & 1];
                }
        }
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) dm[nt][e] *= gC;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t ar[4];
            acc_to_a(a2[2 * ks], a2[2 * ks + 1], ar);
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t bq[4], bk[4];
                ldsm_x4_t(bq, bt_sw(st + R_Q, 8192, 16 * np, 16 * ks, lane));
                ldsm_x4_t(bk, bt_sw(st + R_K, 8192, 16 * np, 16 * ks, lane));
                mma16816(dm[2 * np], ag[ks], bq[0], bq[1]);
                mma16816(dm[2 * np + 1], ag[ks], bq[2], bq[3]);
                mma16816(dm[2 * np], ar, bk[0], bk[1]);
                mma16816(dm[2 * np + 1], ar, bk[2], bk[3]);
            }
        }
        if (ext) {   // this warp is done with the stage
            __syncwarp();
            if (lane == 0) sm100::mbar_arrive(ebar(s));
        } else {
            sm100::named_sync(bar_id, NT);   // every warp of the pass is done with this stage
            issue(s, n - 2);
        }
    }
    if (stg && lane == 0) sm100::bulk_wait_all();   // this warp's tensor stores are complete
    if (!ok && !ext && tid == 0) {
        // a wait ran out: the latest copies of each stage (its phases complete in order;
        // the other warps' copies of a phase complete it together with thread 0's) land
        // before the CTA leaves
        for (int x = 0; x < 2; ++x)
            if (issued[x] > 0) sm100::mbar_wait(bar(x), (uint32_t)(issued[x] - 1) & 1u, 2000000000ull);
    }
    if (ok && dinit) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 8 * nt + 2 * t4 + (e & 1), j = jw + gq + 8 * (e >> 1);
                dinit[((int64_t)bh * DK + i) * dv + j] = dm[nt][e];
            }
    }
}

// The reverse chain's loader when the forward-state role is idle (one thread): stage s =
// it % 3 takes chunk NC - 1 - it once the four chain warps have handed the stage back;
// the copies as in chain_pass's own issue.  On a timed-out wait (or the chain's abort) it
// stops; either way it lets its copies in flight land before it leaves.
__device__ void reverse_loader(uint8_t *smb, const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                               const CUtensorMap *tm_o, const __nv_bfloat16 *__restrict__ TPb,
                               const float *__restrict__ rows, int T, uint64_t limit_ns, uint64_t *r_bar,
                               volatile int *r_abort) {
    using namespace vc;
    const int j0 = blockIdx.x * DSC, bh = blockIdx.y;
    const int NC = (T + C - 1) / C;
    const uint32_t sb = sm100::smem_u32(smb);
    sm100::tma_prefetch_desc(tm_q);
    sm100::tma_prefetch_desc(tm_k);
    sm100::tma_prefetch_desc(tm_o);
    int issued[3] = {0, 0, 0};
    for (int it = 0; it < NC; ++it) {
        const int s = it % 3, n = NC - 1 - it;
        if (it >= 3 && !pass_wait_ab(sm100::smem_u32(&r_bar[3 + s]), (uint32_t)((it - 3) / 3) & 1u, limit_ns,
                                     r_abort))
            break;
        const uint32_t st = sb + (uint32_t)s * R_STAGE, b = sm100::smem_u32(&r_bar[s]);
        const __nv_bfloat16 *tp = TPb + ((int64_t)bh * NC + n) * 2 * C * C;
        const float *blk = rows + ((int64_t)bh * NC + n) * 4 * C;
        sm100::mbar_arrive_expect_tx(b, R_TX);
        sm100::tma_load_3d(st + R_K, tm_k, b, 0, n * C, bh);
        sm100::tma_load_3d(st + R_K + 8192, tm_k, b, 64, n * C, bh);
        sm100::tma_load_3d(st + R_Q, tm_q, b, 0, n * C, bh);
        sm100::tma_load_3d(st + R_Q + 8192, tm_q, b, 64, n * C, bh);
        sm100::tma_load_3d(st + R_O, tm_o, b, j0, n * C, bh);
        sm100::bulk_load(st + R_T, tp, 8192, b);
        sm100::bulk_load(st + R_P, tp + C * C, 8192, b);
        sm100::bulk_load(st + R_G, blk, C * 4, b);
        sm100::bulk_load(st + R_B, blk + 2 * C, C * 4, b);
        ++issued[s];
    }
    // the latest copies of each stage (its phases complete in order) land before this
    // thread leaves, so the CTA cannot leave with copies in flight even if the chain warps
    // left early
    for (int x = 0; x < 3; ++x)
        if (issued[x] > 0)
            sm100::mbar_wait(sm100::smem_u32(&r_bar[x]), (uint32_t)(issued[x] - 1) & 1u, 2000000000ull);
}

// The two sequential passes in one launch: they are independent (both need only the
// tiles), so warps 0-3 of a CTA run the forward state pass and warps 4-7 the reverse
// chain for the same 64 value columns, each role with its own stages and named barrier:
// every SM sub-partition gets one warp of each, whose latencies hide each other.
__global__ void __launch_bounds__(2 * vc::NT, 1)
bwd_passes_vc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_o, const __nv_bfloat16 *__restrict__ k,
                     const float *__restrict__ gamma, const float *__restrict__ U,
                     const __nv_bfloat16 *__restrict__ Wk2, const __nv_bfloat16 *__restrict__ TPb,
                     const float *init, const float *dfinal, __nv_bfloat16 *__restrict__ Wt,
                     __nv_bfloat16 *__restrict__ Sb, float *__restrict__ dR, __nv_bfloat16 *__restrict__ dSb,
                     float *dinit, int T, int dv, int fwd_role, const float *__restrict__ rows,
                     uint64_t limit_ns, const __grid_constant__ CUtensorMap tm_dr,
                     const __grid_constant__ CUtensorMap tm_ds) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (the reverse chain's swizzled tiles), derived from the
    // __shared__ array so that accesses through it stay shared-memory accesses
    uint8_t *smb = smem_raw + ((1024u - (sm100::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ __align__(8) uint64_t r_bar[6];   // the reverse chain's FULL (3) and EMPTY (3) barriers
    __shared__ volatile int r_abort;
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int x = 0; x < 3; ++x) {
            sm100::mbar_init(sm100::smem_u32(&r_bar[x]), 1);
            sm100::mbar_init(sm100::smem_u32(&r_bar[3 + x]), vc::NW);
        }
        r_abort = 0;
        sm100::fence_mbar_init();
    }
    __syncthreads();
    // fwd_role = 0: the forward saved W^T and the states; only the reverse chain runs, its
    // stages filled by the first warp (thread 0), a third stage and the store staging in
    // the idle forward-state stages (the two roles share no barrier, so the other warps
    // leave)
    if (tid < vc::NT) {
        if (fwd_role)
            fwd_state_pass(smb + 2 * vc::R_STAGE, tid, 1, k, gamma, U, Wk2, init, Wt, Sb, T, dv);
        else if (tid == 0)
            reverse_loader(smb, &tm_q, &tm_k, &tm_o, TPb, rows, T, limit_ns, r_bar, &r_abort);
    } else
        chain_pass(smb, tid - vc::NT, 2, &tm_q, &tm_k, &tm_o, dfinal, TPb, dR, dSb, dinit, T, dv, rows, limit_ns,
                   fwd_role ? nullptr : smb + 3 * vc::R_STAGE, &tm_dr, &tm_ds, r_bar, &r_abort);
}

template <typename K>
cudaError_t bwd_set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

size_t tiles_smem(int dk, int dv, int C) {
    return sizeof(float) * ((size_t)C * (dk + 4) + (size_t)C * ((dk > dv ? dk : dv) + 4) +
                            2 * (size_t)C * (C + 1) + 2 * (size_t)C);
}
size_t chain_smem(int dk, int DS, int C, size_t es) {
    const size_t fl = ((size_t)dk * DS + 2 * (size_t)C * C + 3 * (size_t)C * DS + 3 * (size_t)C + 3) & ~(size_t)3;
    return sizeof(float) * fl + 2 * (size_t)C * (dk + 16 / es) * es;
}
size_t chunk_smem(int dk, int dv, int C) {
    return sizeof(float) * (2 * (size_t)C * (dk + 4) + 3 * (size_t)C * (dv + 4) + 2 * (size_t)C * C +
                            2 * (size_t)kBwdJB * (dk + 4) + 8 * (size_t)C + 4);
}

size_t round4(size_t n) { return (n + 3) & ~(size_t)3; }

template <typename TE>
cudaError_t launch_bwd_t(const TE *q, const TE *k, const TE *v, const float *g, const float *beta,
                         float d, const float *init, const TE *dout, const float *dfinal, TE *dq,
                         TE *dk_out, TE *dv_out, float *dg, float *dbeta, float *dinit,
                         int BH, int T, int dk, int dv, int C, float *ws, Elem e, cudaStream_t s,
                         const void *saved) {
    const int NC = (T + C - 1) / C;
    const size_t tok = (size_t)BH * T, st = (size_t)BH * NC * dk * dv;
    (void)e;
    float *gamma = ws;
    float *U = gamma + round4(tok);
    float *Wk = U + round4(tok * dv);
    float *W = Wk + round4(tok * dk);
    float *Mn = W + round4((size_t)BH * NC * C * dv);   // padded tokens: the bf16 W^T tiles
    float *dR = Mn + round4(st);
    float *dMn1 = dR + round4(tok * dv);
    float *Pt = dMn1 + round4(st);
    float *Tt = Pt + round4((size_t)BH * NC * C * C);
    float *DKt = Tt + round4((size_t)BH * NC * C * C);
    constexpr bool kBf16 = std::is_same<TE, __nv_bfloat16>::value;
    const bool tc_chunk = opt_bwd_variant() != 1;
    // From the forward's saved buffer the tensor-core per-chunk kernel needs neither the decay
    // nor the tiles kernel: the forward left T, P and every chunk's row scalars there.
    const bool from_saves = saved && tc_chunk;
    cudaError_t err = cudaSuccess;
    if (!from_saves && (err = launch_decay(g, d, gamma, BH, T, C, s)) != cudaSuccess) return err;
    // the warp-MMA kernels: bf16, d = 128, chunk 64, gradient outputs 16-byte aligned (their
    // 16-byte stores); the states they pass on are value-major, so all four go together
    const bool mma_shape = kBf16 && dk == 128 && dv == 128 && C == 64 &&
                           ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk_out) |
                             reinterpret_cast<uintptr_t>(dv_out)) & 15) == 0;
    if (mma_shape) {
        if constexpr (kBf16) {
            __nv_bfloat16 *TPb = reinterpret_cast<__nv_bfloat16 *>(Tt);   // bf16 T, P tiles
            __nv_bfloat16 *Wk2 = reinterpret_cast<__nv_bfloat16 *>(Wk);   // bf16 rows
            __nv_bfloat16 *Wtb = reinterpret_cast<__nv_bfloat16 *>(W);    // bf16 W^T per chunk
            __nv_bfloat16 *Sbb = reinterpret_cast<__nv_bfloat16 *>(Mn);   // bf16 value-major states
            __nv_bfloat16 *dSbb = reinterpret_cast<__nv_bfloat16 *>(dMn1);
            const uint8_t *sv = static_cast<const uint8_t *>(saved);
            const __nv_bfloat16 *TPin = TPb;
            const float *rows = nullptr;   // the chain's gamma, beta rows from saved scalar blocks
            if (from_saves) {
                TPin = reinterpret_cast<const __nv_bfloat16 *>(sv + saved_tp_offset(BH, T));
                rows = reinterpret_cast<const float *>(sv + saved_sc_offset(BH, T));
            } else {
                if ((err = bwd_set_smem(bwd_tiles_mma_kernel, mt::SMEM)) != cudaSuccess) return err;
                // the tensor-core per-chunk kernel takes each chunk's row scalars (gamma, 1 / gamma,
                // beta, d log(alpha) / dg; 1 KB) from the P-tile region, which this shape leaves unused
                // (also the reverse chain's gamma and beta)
                bwd_tiles_mma_kernel<<<dim3(NC, BH), 256, mt::SMEM, s>>>(q, k, v, gamma, beta, TPb, U, Wk2, T,
                                                                         saved ? 0 : 1, g, d, Pt);
                if ((err = cudaGetLastError()) != cudaSuccess) return err;
                rows = Pt;
            }
            CUtensorMap mq, mk, mo, mdr, mds;
            if (!make_rows_map(&mq, q, BH, T) || !make_rows_map(&mk, k, BH, T) || !make_rows_map(&mo, dout, BH, T) ||
                !make_dr_store_map(&mdr, dR, BH, T) || !make_ds_store_map(&mds, dSbb, (int64_t)BH * NC))
                return cudaErrorInvalidValue;
            const size_t sp = 2 * (size_t)vc::F_STAGE + 2 * (size_t)vc::R_STAGE + 1024;
            if ((err = bwd_set_smem(bwd_passes_vc_kernel, sp)) != cudaSuccess) return err;
            bwd_passes_vc_kernel<<<dim3(dv / vc::DSC, BH), 2 * vc::NT, sp, s>>>(
                mq, mk, mo, k, gamma, U, Wk2, TPin, init, dfinal, Wtb, Sbb, dR, dSbb, dinit, T, dv,
                saved ? 0 : 1, rows, opt_wait_limit_ns(), mdr, mds);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
        }
    } else {
        const size_t s0 = tiles_smem(dk, dv, C);
        if ((err = bwd_set_smem(bwd_tiles_kernel<TE>, s0)) != cudaSuccess) return err;
        bwd_tiles_kernel<TE><<<dim3(NC, BH), 256, s0, s>>>(q, k, v, gamma, beta, Pt, Tt, DKt, U, Wk, T,
                                                          dk, dv, C);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        const int DSf = dv >= 32 ? 32 : 16;
        const size_t sf = sizeof(float) * ((size_t)dk * DSf + 2 * (size_t)C * (dk + 4) +
                                           2 * (size_t)C * DSf + (size_t)C);
        if (DSf == 32) {
            if ((err = bwd_set_smem(bwd_fwd_state_kernel<TE, 32>, sf)) != cudaSuccess) return err;
            bwd_fwd_state_kernel<TE, 32><<<dim3(dv / 32, BH), 256, sf, s>>>(k, gamma, U, Wk, init, W,
                                                                          Mn, T, dk, dv, C);
        } else {
            if ((err = bwd_set_smem(bwd_fwd_state_kernel<TE, 16>, sf)) != cudaSuccess) return err;
            bwd_fwd_state_kernel<TE, 16><<<dim3(dv / 16, BH), 256, sf, s>>>(k, gamma, U, Wk, init, W,
                                                                          Mn, T, dk, dv, C);
        }
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        if (dv >= 32) {
            const size_t s1 = chain_smem(dk, 32, C, sizeof(TE));
            if ((err = bwd_set_smem(bwd_chain_kernel<TE, 32>, s1)) != cudaSuccess) return err;
            bwd_chain_kernel<TE, 32><<<dim3(dv / 32, BH), 256, s1, s>>>(
                q, k, gamma, beta, dout, dfinal, Pt, Tt, dR, dMn1, dinit, T, dk, dv, C);
        } else {
            const size_t s1 = chain_smem(dk, 16, C, sizeof(TE));
            if ((err = bwd_set_smem(bwd_chain_kernel<TE, 16>, s1)) != cudaSuccess) return err;
            bwd_chain_kernel<TE, 16><<<dim3(dv / 16, BH), 256, s1, s>>>(
                q, k, gamma, beta, dout, dfinal, Pt, Tt, dR, dMn1, dinit, T, dk, dv, C);
        }
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if constexpr (kBf16) {
        if (mma_shape) {
            if ((err = bwd_set_smem(bwd_chunk_mma_kernel, mm::SMEM)) != cudaSuccess) return err;
            int dev = 0, nsm = 0;
            if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
            if ((err = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
                return err;
            const int ntask = NC * BH, grid = ntask < nsm ? ntask : nsm;
            // the states and W^T: the forward's saved tiles, or the ones just recomputed
            const __nv_bfloat16 *Sb_in = saved ? static_cast<const __nv_bfloat16 *>(saved)
                                               : reinterpret_cast<const __nv_bfloat16 *>(Mn);
            const __nv_bfloat16 *Wt_in =
                saved ? reinterpret_cast<const __nv_bfloat16 *>(static_cast<const uint8_t *>(saved) +
                                                               saved_state_bytes(BH, T))
                      : reinterpret_cast<const __nv_bfloat16 *>(W);
            if (tc_chunk)
                return launch_bwd_chunk_tc(q, k, v,
                                           from_saves ? reinterpret_cast<const float *>(
                                                            static_cast<const uint8_t *>(saved) +
                                                            saved_sc_offset(BH, T))
                                                      : Pt,
                                           Wt_in, Sb_in, dout, dR, dMn1, dq, dk_out, dv_out, dg, dbeta, BH, T, s);
            bwd_chunk_mma_kernel<<<grid, 256, mm::SMEM, s>>>(
                q, k, v, g, beta, d, gamma, Wt_in, Sb_in, dout, dR,
                reinterpret_cast<const __nv_bfloat16 *>(dMn1), dq, dk_out, dv_out, dg, dbeta, T, BH);
            return cudaGetLastError();
        }
    }
    const size_t s2 = chunk_smem(dk, dv, C);
    if ((err = bwd_set_smem(bwd_chunk_kernel<TE>, s2)) != cudaSuccess) return err;
    bwd_chunk_kernel<TE><<<dim3(NC, BH), kBwdThreads, s2, s>>>(
        q, k, v, g, beta, d, gamma, W, Mn, dout, dR, dMn1, Pt, DKt, dq, dk_out, dv_out, dg, dbeta, T,
        dk, dv, C);
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
    return sizeof(float) * (round4(tok) + round4(tok * dv) + round4(tok * dk) +
                            round4((size_t)BH * NC * C * dv) + round4(st) + round4(tok * dv) + round4(st) +
                            3 * round4((size_t)BH * NC * C * C));
}

void bwd_free_region(int BH, int T, int dk, int dv, int C, size_t *offset, size_t *bytes) {
    const int NC = (T + C - 1) / C;
    const size_t tok = (size_t)BH * T, st = (size_t)BH * NC * dk * dv;
    *offset = sizeof(float) * round4(tok);   // after gamma: U, Wk, W, the states
    *bytes = sizeof(float) * (round4(tok * dv) + round4(tok * dk) + round4((size_t)BH * NC * C * dv) + round4(st));
}

bool bwd_saved_shape(int dk, int dv, int C, Elem e, const void *dq, const void *dk_out,
                     const void *dv_out) {
    return e == Elem::BF16 && dk == 128 && dv == 128 && C == 64 &&
           ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk_out) |
             reinterpret_cast<uintptr_t>(dv_out)) & 15) == 0;
}

cudaError_t launch_bwd(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, float d, const float *init, const void *dout,
                       const float *dfinal, void *dq, void *dk_out, void *dv_out, float *dg,
                       float *dbeta, float *dinit, int BH, int T, int dk, int dv, int C,
                       void *ws, Elem e, cudaStream_t s, const void *saved) {
    if (saved && !bwd_saved_shape(dk, dv, C, e, dq, dk_out, dv_out)) return cudaErrorInvalidValue;
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
                                   (float *)dv_out, dg, dbeta, dinit, BH, T, dk, dv, C, w, e, s,
                                   nullptr);
    return launch_bwd_t<__nv_bfloat16>(
        (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, g, beta, d,
        init, (const __nv_bfloat16 *)dout, dfinal, (__nv_bfloat16 *)dq, (__nv_bfloat16 *)dk_out,
        (__nv_bfloat16 *)dv_out, dg, dbeta, dinit, BH, T, dk, dv, C, w, e, s, saved);
}

// Reads and clears the error word of this file's kernels (synchronous).
cudaError_t take_bwd_error_word(unsigned *value) {
    unsigned word = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&word, g_bwd_error_word, sizeof(word));
    if (e != cudaSuccess) return e;
    *value = word;
    if (word != 0) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_bwd_error_word, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace gdr
