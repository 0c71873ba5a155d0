// gdr_fused.cu -- fused chunked prefill of the gated delta rule on the
// 5th-generation tensor core (tcgen05 + TMEM, operands fed by TMA).
//
// One CTA owns one (sequence, head) and walks its chunks of C = 64 tokens in
// order.  Per chunk it does the whole chunked form -- cumulative decay, the
// intra-chunk WY/UT transform, the state step and the output -- with every
// contraction on the tensor core, and the fp32 state never leaves the SM.
// HBM sees q, k, v, g, beta once, out once, and the state twice (in, out).
//
// The method: with the lower-bounded decay, gamma_r >= a_min^r inside a chunk,
// so 1/gamma and 1/gamma_C are finite and every causal tile -- the diagonal
// (intra-chunk) tile included -- is one dense product with diagonal scalings
// ("What a Trillion-Parameter MoE Model Reveals About the Next Stage of LLM
// Scaling", sections 3.1-3.3; "Architecture Evolution and Training Engineering
// for Trillion-Scale Sparse Multimodal Models", section 3.2).  Here those
// scalings are applied in fp32 on the TMEM accumulators, not folded into the
// bf16 operands, so q, k and v enter the tensor core exactly as given.
//
// Algebra per chunk (rows r, s; gamma, 1/gamma, gamma_C as usual; M = S^T):
//   A   = strict_lower(diag(beta gamma) K K^T diag(1/gamma)),  T = (I + A)^-1
//   L   = T - I (strictly lower);  Lb = L diag(beta),  Lbg = L diag(beta gamma)
//   U   = diag(beta) V + Lb V                        (identity part kept exact)
//   Wk  = diag(beta gamma) K + Lbg K
//   W   = U - Wk M_n
//   Wt  = diag(gamma_C / gamma) W
//   P   = lower_incl(Q K^T) / gamma_C
//   O   = diag(gamma) (Q M_n + P Wt)
//   M_{n+1} = gamma_C M_n + K^T Wt
// Every product is computed transposed so that its M dimension is 128
// (dv or dk):  U^T = V^T Lb^T,  Wk^T = K^T Lbg^T,  W^T = U^T - M^T Wk^T,
// O^T = M^T Q^T + Wt^T P^T,  M^T_{n+1} = gamma_C M^T + Wt^T K.
//
// Shared-memory operands (all 128-byte swizzled, 1024-byte aligned):
//   KQ[stage]  32 KB  [slab i/64][K rows 0..63 | Q rows 0..63][128 B]  (TMA)
//   V[stage]   16 KB  [slab j/64][V rows 0..63][128 B]                   (TMA)
//   MT         32 KB  M^T bf16, K-major ([j][i], two i slabs)
//   WkT        16 KB  Wk^T bf16, MN-major ([i][r])
//   WtT        16 KB  Wt^T bf16, K-major ([j][s])
//   P, Lb, Lbg  8 KB each, K-major ([r][s])
// TMEM (fp32, 128 lanes): KQK^T 64 cols, W^T 64, Wk^T 64, O^T 64, M^T 128.

#include "gdr_internal.h"
#include "gdr_math.cuh"
#include "gdr_sm100.cuh"

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>

namespace gdr {

__device__ unsigned g_device_error_word = 0;

namespace {

using namespace sm100;

constexpr int C = 64;     // chunk
constexpr int D = 128;    // dk = dv
constexpr int NT = 128;   // threads: one per TMEM lane

// shared-memory map (bytes from the 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;             // 2 x 32 KB
constexpr uint32_t KQ_BYTES = 32768;
constexpr uint32_t OFF_V = 65536;          // 2 x 16 KB
constexpr uint32_t V_BYTES = 16384;
constexpr uint32_t OFF_MT = 98304;         // 32 KB
constexpr uint32_t OFF_WKT = 131072;       // 16 KB
constexpr uint32_t OFF_WTT = 147456;       // 16 KB
constexpr uint32_t OFF_P = 163840;         // 8 KB
constexpr uint32_t OFF_LB = 172032;        // 8 KB
constexpr uint32_t OFF_LBG = 180224;       // 8 KB
constexpr int LDA = 68;                    // fp32 row stride of the solve matrices
constexpr uint32_t OFF_AS = 188416;        // 64 x 68 fp32
constexpr uint32_t OFF_TS = OFF_AS + 64 * LDA * 4;   // 64 x 68 fp32
constexpr uint32_t OFF_YS = OFF_TS + 64 * LDA * 4;   // 32 x 32 fp32
constexpr uint32_t OFF_SC = OFF_YS + 32 * 32 * 4;    // scalars: 2 stages x 4 x 64 fp32
constexpr uint32_t SMEM_USED = OFF_SC + 2 * 4 * 64 * 4;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;    // alignment slack
static_assert(SMEM_ALLOC <= 232448, "exceeds 227 KB of shared memory per CTA");

// TMEM columns
constexpr uint32_t TM_KQK = 0, TM_W = 64, TM_WK = 128, TM_O = 192, TM_M = 256;
constexpr uint32_t TM_COLS = 512;

constexpr uint64_t kCleanupLimitNs = 2000000000ull;

struct Scal {   // per-stage per-row scalars of one chunk
    float *gam, *ig, *bs, *bg;
};

__device__ __forceinline__ Scal scal(uint8_t *sm, int stage) {
    float *b = reinterpret_cast<float *>(sm + OFF_SC) + stage * 4 * 64;
    return {b, b + 64, b + 128, b + 192};
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Write 64 fp32 values as one 128-byte bf16 row of a 128B-swizzled tile.
__device__ __forceinline__ void st_row_bf16(uint8_t *tile, uint32_t row, const float *v) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint4 u;
        u.x = pack_bf16x2(v[ch * 8 + 0], v[ch * 8 + 1]);
        u.y = pack_bf16x2(v[ch * 8 + 2], v[ch * 8 + 3]);
        u.z = pack_bf16x2(v[ch * 8 + 4], v[ch * 8 + 5]);
        u.w = pack_bf16x2(v[ch * 8 + 6], v[ch * 8 + 7]);
        *reinterpret_cast<uint4 *>(tile + row * 128u + ((ch ^ (row & 7u)) << 4)) = u;
    }
}

__device__ __forceinline__ float ld_bf16_sw(const uint8_t *tile, uint32_t row, uint32_t col) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + sw128_offset(row, col)));
}

// Cumulative decay of one chunk (threads 0..63 hold row t's g and beta; all
// 128 threads must call: it contains two block barriers).
__device__ __forceinline__ void chunk_decay(int tid, float gv, float bv, int c, float a_min,
                                            Scal s, float *s_part, float *s_gC) {
    const int lane = tid & 31, warp = tid >> 5;
    float incl = 0.f;
    if (tid < 64) {
        incl = (tid < c) ? log_alpha(gv, a_min) : 0.f;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) s_part[warp] = incl;
    }
    __syncthreads();
    if (tid < 64) {
        if (warp == 1) incl += s_part[0];
        const bool valid = tid < c;
        const float gam = valid ? expf(incl) : 1.f;
        const float b = valid ? bv : 0.f;
        s.gam[tid] = gam;
        s.ig[tid] = 1.f / gam;
        s.bs[tid] = b;
        s.bg[tid] = b * gam;
        if (tid == c - 1) *s_gC = gam;
    }
    __syncthreads();
}

// T = (I + A)^-1 for the strictly lower 64 x 64 A in As (fp32), into Ts
// (lower part only is defined).  Blocked: four 16 x 16 diagonal inverses by
// forward substitution, then two merge levels T_ij = -T_ii A_ij T_jj.
__device__ __forceinline__ void solve_unit_lower(int tid, const float *As, float *Ts, float *Ys) {
    if (tid < 64) {
        const int b = tid >> 4, l = tid & 15, o = 16 * b;
        float x[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) x[m] = (m == l) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) acc = fmaf(As[(o + r) * LDA + o + m], x[m], acc);
            if (r > l) x[r] = -acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Ts[(o + r) * LDA + o + l] = x[r];
    }
    __syncthreads();
    // level 1: blocks (1,0) and (3,2), 16 x 16 each
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int idx = u * NT + tid, p = idx >> 8, r = (idx >> 4) & 15, l = idx & 15;
        const int R = 16 * (2 * p + 1), Cb = 16 * (2 * p);
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) acc = fmaf(As[(R + r) * LDA + Cb + m], Ts[(Cb + m) * LDA + Cb + l], acc);
        Ys[p * 256 + r * 16 + l] = acc;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int idx = u * NT + tid, p = idx >> 8, r = (idx >> 4) & 15, l = idx & 15;
        const int R = 16 * (2 * p + 1), Cb = 16 * (2 * p);
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m)
            if (m <= r) acc = fmaf(Ts[(R + r) * LDA + R + m], Ys[p * 256 + m * 16 + l], acc);
        Ts[(R + r) * LDA + Cb + l] = -acc;
    }
    __syncthreads();
    // level 2: block rows 32..63, cols 0..31
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int idx = u * NT + tid, r = idx >> 5, l = idx & 31;
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 32; ++m)
            if (m >= l) acc = fmaf(As[(32 + r) * LDA + m], Ts[m * LDA + l], acc);
        Ys[r * 32 + l] = acc;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int idx = u * NT + tid, r = idx >> 5, l = idx & 31;
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 32; ++m)
            if (m <= r) acc = fmaf(Ts[(32 + r) * LDA + 32 + m], Ys[m * 32 + l], acc);
        Ts[(32 + r) * LDA + l] = -acc;
    }
    __syncthreads();
}

struct FusedArgs {
    const float *g, *beta, *init;
    __nv_bfloat16 *out;
    float *final_state;
    float a_min;
    int T;
    uint64_t limit_ns;
};

__global__ void __launch_bounds__(NT, 1)
fused_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FusedArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(sm);
    __shared__ __align__(8) uint64_t bar_tma[2];
    __shared__ __align__(8) uint64_t bar_mma;
    __shared__ uint32_t s_tmem;
    __shared__ float s_part[2];
    __shared__ float s_gC[2];

    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x;
    const int T = a.T;
    const int NC = (T + C - 1) / C;
    const int64_t row_base = (int64_t)bh * T;
    const uint32_t btma0 = smem_u32(&bar_tma[0]), btma1 = smem_u32(&bar_tma[1]);
    const uint32_t bmma = smem_u32(&bar_mma);

    if (tid == 0) {
        mbar_init(btma0, 1);
        mbar_init(btma1, 1);
        mbar_init(bmma, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);   // this warp's lane quadrant

    bool tma_pending[2] = {false, false};   // meaningful in thread 0
    uint32_t tma_parity[2] = {0u, 0u};      // parity of the outstanding load per stage
    bool mma_pending = false;               // meaningful in thread 0
    uint32_t mma_phase = 0;
    bool ok = true;

    auto issue_tma = [&](int n) {
        const int st = n & 1;
        const uint32_t bar = st ? btma1 : btma0;
        const uint32_t kq = sbase + OFF_KQ + st * KQ_BYTES;
        const uint32_t vv = sbase + OFF_V + st * V_BYTES;
        mbar_arrive_expect_tx(bar, KQ_BYTES + V_BYTES);
        tma_load_3d(kq + 0, &tm_k, bar, 0, n * C, bh);
        tma_load_3d(kq + 8192, &tm_q, bar, 0, n * C, bh);
        tma_load_3d(kq + 16384, &tm_k, bar, 64, n * C, bh);
        tma_load_3d(kq + 24576, &tm_q, bar, 64, n * C, bh);
        tma_load_3d(vv + 0, &tm_v, bar, 0, n * C, bh);
        tma_load_3d(vv + 8192, &tm_v, bar, 64, n * C, bh);
        tma_pending[st] = true;
        tma_parity[st] = (uint32_t)(n >> 1) & 1u;
    };
    auto mma_wait = [&]() -> bool {
        const bool w = mbar_wait(bmma, mma_phase, a.limit_ns);
        if (w) {
            mma_phase ^= 1u;
            mma_pending = false;
        }
        return w;
    };

    if (tid == 0) {
        issue_tma(0);
        if (NC > 1) issue_tma(1);
    }

    // decay of chunk 0, prefetch of chunk 1's g / beta
    float g_next = 0.f, b_next = 0.f;
    {
        const int c0 = min(C, T);
        float gv = 0.f, bv = 0.f;
        if (tid < c0) {
            gv = a.g[row_base + tid];
            bv = a.beta[row_base + tid];
        }
        chunk_decay(tid, gv, bv, c0, a.a_min, scal(sm, 0), s_part, &s_gC[0]);
        if (NC > 1 && tid < min(C, T - C)) {
            g_next = a.g[row_base + C + tid];
            b_next = a.beta[row_base + C + tid];
        }
    }

    // initial state: TMEM M^T <- gamma_C(0) * M0^T, MT <- bf16(M0^T)
    {
        const float gC = s_gC[0];
        const int j = tid;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
            float v[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int i = cb * 32 + e;
                v[e] = a.init ? a.init[((int64_t)bh * D + i) * D + j] : 0.f;
            }
            uint8_t *slab = sm + OFF_MT + (cb >> 1) * 16384;
            // 32 values = 4 swizzle chunks of the row
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const uint32_t ch = (cb & 1) * 4 + q4;
                uint4 u;
                u.x = pack_bf16x2(v[q4 * 8 + 0], v[q4 * 8 + 1]);
                u.y = pack_bf16x2(v[q4 * 8 + 2], v[q4 * 8 + 3]);
                u.z = pack_bf16x2(v[q4 * 8 + 4], v[q4 * 8 + 5]);
                u.w = pack_bf16x2(v[q4 * 8 + 6], v[q4 * 8 + 7]);
                *reinterpret_cast<uint4 *>(slab + j * 128u + ((ch ^ (j & 7u)) << 4)) = u;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] *= gC;
            tmem_st32(tl + TM_M + cb * 32, v);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    }

    const uint32_t idesc_kqk = idesc_bf16(128, 64, false, false);
    const uint32_t idesc_u = idesc_bf16(128, 64, true, false);
    const uint32_t idesc_w = idesc_bf16(128, 64, false, true, true);
    const uint32_t idesc_o1 = idesc_bf16(128, 64, false, false);
    const uint32_t idesc_d = idesc_bf16(128, 128, false, true);

    float *As = reinterpret_cast<float *>(sm + OFF_AS);
    float *Ts = reinterpret_cast<float *>(sm + OFF_TS);
    float *Ys = reinterpret_cast<float *>(sm + OFF_YS);

#pragma unroll 1
    for (int n = 0; n < NC; ++n) {
        const int st = n & 1;
        const int t0 = n * C;
        const int c = min(C, T - t0);
        const Scal S = scal(sm, st);
        const float gC = s_gC[st];
        const float igC = 1.f / gC;
        uint8_t *kq = sm + OFF_KQ + st * KQ_BYTES;
        uint8_t *vt = sm + OFF_V + st * V_BYTES;
        const uint32_t kq_a = sbase + OFF_KQ + st * KQ_BYTES;
        const uint32_t v_a = sbase + OFF_V + st * V_BYTES;

        // ---- inputs of chunk n
        ok = mbar_wait(st ? btma1 : btma0, (uint32_t)(n >> 1) & 1u, a.limit_ns);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        if (tid == 0) tma_pending[st] = false;

        // ---- [K;Q] K^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ad = kq_a + (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16(tmem + TM_KQK, sdesc_sw128(ad, 16, 1024), sdesc_sw128(ad, 16, 1024),
                         idesc_kqk, kk > 0);
            }
            mma_commit(bmma);
            mma_pending = true;
        }
        ok = __syncthreads_and(mma_wait());
        if (!ok) break;
        tc_fence_after();
        {
            float v[64];
            tmem_ld32(tl + TM_KQK, *reinterpret_cast<float(*)[32]>(&v[0]));
            tmem_ld32(tl + TM_KQK + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
            tmem_wait_ld();
            if (tid < 64) {
                const int r = tid;
                const float br = S.bg[r];
#pragma unroll
                for (int s = 0; s < 64; ++s)
                    As[r * LDA + s] = (s < r && r < c) ? br * v[s] * S.ig[s] : 0.f;
            } else {
                const int r = tid - 64;
#pragma unroll
                for (int s = 0; s < 64; ++s) v[s] = (s <= r && r < c) ? v[s] * igC : 0.f;
                st_row_bf16(sm + OFF_P, r, v);
            }
        }
        tc_fence_before();
        __syncthreads();

        // ---- T = (I + A)^-1, then Lb, Lbg
        solve_unit_lower(tid, As, Ts, Ys);
        {
            const int r = tid & 63;
            const float *sc = (tid < 64) ? S.bs : S.bg;
            float v[64];
#pragma unroll
            for (int s = 0; s < 64; ++s) v[s] = (s < r) ? Ts[r * LDA + s] * sc[s] : 0.f;
            st_row_bf16(sm + ((tid < 64) ? OFF_LB : OFF_LBG), r, v);
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---- U^T' = V^T Lb^T, Wk^T' = K^T Lbg^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16(tmem + TM_W, sdesc_sw128(v_a + kk * 2048, 8192, 1024),
                         sdesc_sw128(sbase + OFF_LB + kk * 32, 16, 1024), idesc_u, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16(tmem + TM_WK, sdesc_sw128(kq_a + kk * 2048, 16384, 1024),
                         sdesc_sw128(sbase + OFF_LBG + kk * 32, 16, 1024), idesc_u, kk > 0);
            }
            mma_commit(bmma);
            mma_pending = true;
        }
        ok = __syncthreads_and(mma_wait());
        if (!ok) break;
        tc_fence_after();
        {   // Wk^T[i][r] = Wk^T'[i][r] + beta_r gamma_r K[r][i]  ->  WkT (MN-major, row i)
            const int i = tid;
            float v[64];
            tmem_ld32(tl + TM_WK, *reinterpret_cast<float(*)[32]>(&v[0]));
            tmem_ld32(tl + TM_WK + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
            tmem_wait_ld();
            const uint8_t *kslab = kq + (i >> 6) * 16384;
#pragma unroll
            for (int r = 0; r < 64; ++r) v[r] = fmaf(S.bg[r], ld_bf16_sw(kslab, r, i & 63), v[r]);
            st_row_bf16(sm + OFF_WKT, i, v);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- W^T = U^T' - M^T Wk^T ;  O^T = M^T Q^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ad = sbase + OFF_MT + (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16(tmem + TM_W, sdesc_sw128(ad, 16, 1024),
                         sdesc_sw128(sbase + OFF_WKT + kk * 2048, 16384, 1024), idesc_w, 1);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t ad = sbase + OFF_MT + (kk >> 2) * 16384 + (kk & 3) * 32;
                const uint32_t bd = kq_a + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32;
                mma_bf16(tmem + TM_O, sdesc_sw128(ad, 16, 1024), sdesc_sw128(bd, 16, 1024),
                         idesc_o1, kk > 0);
            }
            mma_commit(bmma);
            mma_pending = true;
        }
        ok = __syncthreads_and(mma_wait());
        if (!ok) break;
        tc_fence_after();
        {   // Wt^T[j][s] = (W^T'[j][s] + beta_s V[s][j]) * gamma_C / gamma_s  -> WtT (row j)
            const int j = tid;
            float v[64];
            tmem_ld32(tl + TM_W, *reinterpret_cast<float(*)[32]>(&v[0]));
            tmem_ld32(tl + TM_W + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
            tmem_wait_ld();
            const uint8_t *vslab = vt + (j >> 6) * 8192;
#pragma unroll
            for (int s = 0; s < 64; ++s) {
                const float w = fmaf(S.bs[s], ld_bf16_sw(vslab, s, j & 63), v[s]);
                v[s] = (s < c) ? w * (gC * S.ig[s]) : 0.f;
            }
            st_row_bf16(sm + OFF_WTT, j, v);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- M^T += Wt^T K ;  O^T += Wt^T P^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16(tmem + TM_M, sdesc_sw128(sbase + OFF_WTT + kk * 32, 16, 1024),
                         sdesc_sw128(kq_a + kk * 2048, 16384, 1024), idesc_d, 1);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16(tmem + TM_O, sdesc_sw128(sbase + OFF_WTT + kk * 32, 16, 1024),
                         sdesc_sw128(sbase + OFF_P + kk * 32, 16, 1024), idesc_o1, 1);
            }
            mma_commit(bmma);
            mma_pending = true;
        }
        // decay of the next chunk while the tensor core works
        if (n + 1 < NC) {
            const int c1 = min(C, T - (n + 1) * C);
            chunk_decay(tid, g_next, b_next, c1, a.a_min, scal(sm, st ^ 1), s_part, &s_gC[st ^ 1]);
            if (n + 2 < NC && tid < min(C, T - (n + 2) * C)) {
                g_next = a.g[row_base + (int64_t)(n + 2) * C + tid];
                b_next = a.beta[row_base + (int64_t)(n + 2) * C + tid];
            }
        }
        ok = __syncthreads_and(mma_wait());
        if (!ok) break;
        tc_fence_after();
        {   // output: out[t0 + r][j] = gamma_r * O^T[j][r]
            const int j = tid;
            float v[64];
            tmem_ld32(tl + TM_O, *reinterpret_cast<float(*)[32]>(&v[0]));
            tmem_ld32(tl + TM_O + 32, *reinterpret_cast<float(*)[32]>(&v[32]));
            tmem_wait_ld();
            __nv_bfloat16 *o = a.out + (row_base + t0) * D + j;
#pragma unroll
            for (int r = 0; r < 64; ++r)
                if (r < c) o[(int64_t)r * D] = __float2bfloat16_rn(v[r] * S.gam[r]);
        }
        {   // state: MT <- bf16(M^T_{n+1}); TMEM M^T <- gamma_C(n+1) M^T_{n+1}
            const int j = tid;
            const bool last = (n + 1 == NC);
            const float gn = last ? 1.f : s_gC[st ^ 1];
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                float v[32];
                tmem_ld32(tl + TM_M + cb * 32, v);
                tmem_wait_ld();
                if (last) {
                    if (a.final_state) {
                        float *f = a.final_state + (int64_t)bh * D * D + j;
#pragma unroll
                        for (int e = 0; e < 32; ++e) f[(int64_t)(cb * 32 + e) * D] = v[e];
                    }
                } else {
                    uint8_t *slab = sm + OFF_MT + (cb >> 1) * 16384;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const uint32_t ch = (cb & 1) * 4 + q4;
                        uint4 u;
                        u.x = pack_bf16x2(v[q4 * 8 + 0], v[q4 * 8 + 1]);
                        u.y = pack_bf16x2(v[q4 * 8 + 2], v[q4 * 8 + 3]);
                        u.z = pack_bf16x2(v[q4 * 8 + 4], v[q4 * 8 + 5]);
                        u.w = pack_bf16x2(v[q4 * 8 + 6], v[q4 * 8 + 7]);
                        *reinterpret_cast<uint4 *>(slab + j * 128u + ((ch ^ (j & 7u)) << 4)) = u;
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= gn;
                    tmem_st32(tl + TM_M + cb * 32, v);
                }
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && n + 2 < NC) issue_tma(n + 2);
    }

    if (!ok && tid == 0) {
        // A bounded wait gave up: record it, let this CTA's copies and MMAs in
        // flight land (each wait bounded again), then release TMEM below.
        atomicOr(&g_device_error_word, kDevErrTimeout);
        if (tma_pending[0]) mbar_wait(btma0, tma_parity[0], kCleanupLimitNs);
        if (tma_pending[1]) mbar_wait(btma1, tma_parity[1], kCleanupLimitNs);
        if (mma_pending) mbar_wait(bmma, mma_phase, kCleanupLimitNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// [BH][T][128] bf16 viewed as a 3-D tensor; 64 x 64 boxes, 128-byte swizzle,
// zero fill beyond T.
bool make_map(CUtensorMap *m, const void *ptr, int BH, int T) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint64_t wait_limit_ns() {
    // Test hook: GDR_FAULT_INJECT=timeout makes every bounded wait give up at
    // once, exercising the error path without any GPU fault.
    const char *e = std::getenv("GDR_FAULT_INJECT");
    if (e && std::strcmp(e, "timeout") == 0) return 0;
    return 2000000000ull;   // 2 s
}

}  // namespace

bool fused_supported(int dk, int dv, int C_, Elem e) {
    return e == Elem::BF16 && dk == D && dv == D && C_ == C;
}

cudaError_t launch_fused(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, float a_min, const float *init, void *out,
                         float *final_state, int B, int H, int T, int dk, int dv, int C_,
                         cudaStream_t s) {
    if (!fused_supported(dk, dv, C_, Elem::BF16)) return cudaErrorInvalidValue;
    const int BH = B * H;
    if (BH == 0 || T == 0) return cudaSuccess;
    // TMA needs 16-byte aligned bases
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v)) & 15)
        return cudaErrorMisalignedAddress;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, BH, T) || !make_map(&mk, k, BH, T) || !make_map(&mv, v, BH, T))
        return cudaErrorInvalidValue;
    FusedArgs a{g, beta, init, static_cast<__nv_bfloat16 *>(out), final_state, a_min, T,
                wait_limit_ns()};
    cudaError_t e = cudaFuncSetAttribute(fused_prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    fused_prefill_kernel<<<BH, NT, SMEM_ALLOC, s>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(cudaStream_t s, unsigned *value) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    unsigned word = 0;
    e = cudaMemcpyFromSymbol(&word, g_device_error_word, sizeof(word));
    if (e != cudaSuccess) return e;
    *value = word;
    if (word != 0) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace gdr
