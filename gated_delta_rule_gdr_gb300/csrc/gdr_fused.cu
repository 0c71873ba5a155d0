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
//   U   = (Lb + diag(beta)) V,  Wk = (Lbg + diag(beta gamma)) K, where each
//         diagonal is split into its bf16 value plus a bf16 residual applied
//         by a second product, so the identity part stays exact to ~2^-17
//   W   = U - Wk M_n
//   Wt  = diag(gamma_C / gamma) W
//   P   = lower_incl(Q K^T) / gamma_C
//   O   = diag(gamma) (Q M_n + P Wt)
//   M_{n+1} = gamma_C M_n + K^T Wt
// The products are computed transposed so that their M dimension is 128
// (dv or dk):  U^T = V^T Lb^T,  Wk^T = K^T Lbg^T,  W^T = U^T - M^T Wk^T,
// M^T_{n+1} = gamma_C M^T + Wt^T K -- except the output, O = Q M + P Wt, an
// M = 64 product whose TMEM rows are whole output rows, so each row leaves the
// SM as contiguous 16-byte stores without a transpose.
//
// Warp roles (416 threads):
//   prep  (warps 0-7)  chunk k: A and P from [K;Q]K^T, the triangular solve,
//                      Lb / Lbg and the U^T, Wk^T products -- state-independent
//   chain (warps 8-11) chunk n: Wk^T to bf16, W^T epilogue, state update, output
//   copy  (warp 12)    the TMA loads of the inputs and the cumulative decay
// Each warpgroup issues its own tcgen05.mma from one elected thread, so the
// preparation of chunk n+1 overlaps the state chain of chunk n.
//
// Shared-memory operands (128-byte swizzled, 1024-byte aligned):
//   KQ[stage]  32 KB  [slab i/64][K rows 0..63 | Q rows 0..63][128 B]  (TMA)
//   V[stage]   16 KB  [slab j/64][V rows 0..63][128 B]                   (TMA)
//   MT         32 KB  M^T bf16, K-major ([j][i], two i slabs)
//   WkT        16 KB  Wk^T bf16, MN-major ([i][r])
//   WtT        16 KB  Wt^T bf16, K-major ([j][s])
//   P[2]        8 KB each, K-major ([r][s]), one per stage
//   Lb, Lbg     8 KB each, K-major ([r][s]), sharing space with the fp32 A
//   Db, Dbg     8 KB each, the diagonal residuals, sharing space with the fp32 T
// TMEM (fp32, 128 lanes): KQK^T 64 cols, W^T 2 x 64, Wk^T 64, M^T 128, and O
// 128 cols in the M = 64 layout (row r in lane r % 16 + 32 (r / 16)).

#include "gdr_fused_common.cuh"

namespace gdr {
namespace {

constexpr int NT = 416;    // prep (256) + chain (128) + copy (32)

// shared-memory map (bytes from the 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;             // 2 x 32 KB
constexpr uint32_t KQ_BYTES = 32768;
constexpr uint32_t OFF_V = 65536;          // 2 x 16 KB
constexpr uint32_t V_BYTES = 16384;
constexpr uint32_t OFF_MT = 98304;         // 32 KB
constexpr uint32_t OFF_WKT = 131072;       // 16 KB
constexpr uint32_t OFF_WTT = 147456;       // 16 KB
constexpr uint32_t OFF_P = 163840;         // 2 x 8 KB
constexpr uint32_t OFF_AS = 180224;        // 64 x 68 fp32; Lb, Lbg reuse its first 16 KB
constexpr uint32_t OFF_LB = OFF_AS;
constexpr uint32_t OFF_LBG = OFF_AS + 8192;
constexpr uint32_t OFF_TS = OFF_AS + 64 * LDA * 4;   // 64 x 68 fp32; Db, Dbg reuse it
constexpr uint32_t OFF_DB = OFF_TS;
constexpr uint32_t OFF_DBG = OFF_TS + 8192;
constexpr uint32_t OFF_YS = OFF_TS + 64 * LDA * 4;   // 32 x 40 fp32
constexpr int NSCAL = 3;                   // scalar slots (chunk m uses slot m % 3)
constexpr uint32_t OFF_SC = OFF_YS + 32 * LDY * 4;   // scalars: 3 slots x 5 x 64 fp32
constexpr uint32_t SMEM_USED = OFF_SC + NSCAL * 5 * 64 * 4;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;    // alignment slack
static_assert(SMEM_ALLOC <= 232448, "exceeds 227 KB of shared memory per CTA");
static_assert(OFF_AS % 1024 == 0 && 64 * LDA * 4 >= 16384, "Lb/Lbg must fit in A's space");
static_assert(OFF_TS % 1024 == 0, "Db/Dbg must be 1024-byte aligned");

// TMEM columns
constexpr uint32_t TM_KQK = 0, TM_W = 64 /* two buffers */, TM_WK = 192, TM_O = 256 /* 128 */,
                   TM_M = 384;
constexpr uint32_t TM_COLS = 512;

constexpr int kL2Ahead = 3;   // chunks prefetched into L2 beyond the two staged in SMEM

__device__ __forceinline__ Scal scal(uint8_t *sm, int slot) {
    return scal_at(reinterpret_cast<float *>(sm + OFF_SC) + slot * 5 * 64);
}

// mbarriers of the pipeline (index into s_bar)
enum : int {
    B_FULL0 = 0, B_FULL1,      // copy: TMA inputs of a stage landed
    B_KQK,                     // prep commit: [K;Q]K^T done
    B_UWK,                     // prep commit: U^T', Wk^T' done
    B_W,                       // chain commit: W^T done
    B_D,                       // chain commit: M^T update done
    B_O2,                      // chain commit: output accumulation done
    B_SCAL0, B_SCAL1, B_SCAL2, // copy: decay scalars of a chunk written, per slot
    B_WKFREE,                  // chain: Wk^T of a chunk read out of TMEM
    B_RWFREE0, B_RWFREE1,      // chain: W^T buffer read out, per buffer
    B_OSTAGE0, B_OSTAGE1,      // chain: input stage done with (its MMAs complete)
    B_PFREE0, B_PFREE1,        // chain: P buffer read by the output product, per buffer
    B_DRAINP, B_DRAINC,        // commits of the error path (prep, chain)
    NUM_BARS
};

__global__ void __launch_bounds__(NT, 1)
fused_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FusedArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(sm);
    __shared__ __align__(8) uint64_t s_bar[NUM_BARS];
    __shared__ uint32_t s_tmem;
    __shared__ float s_gC[NSCAL];
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x;
    const int T = a.T;
    const int NC = (T + C - 1) / C;
    const int64_t row_base = (int64_t)bh * T;
    auto bar = [&](int i) { return smem_u32(&s_bar[i]); };

    if (tid == 0) {
        for (int i = 0; i < NUM_BARS; ++i) mbar_init(bar(i), 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 12) {
        tmem_alloc(smem_u32(&s_tmem), TM_COLS);
        tmem_relinquish();
        if (tid == 384) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    float *As = reinterpret_cast<float *>(sm + OFF_AS);
    float *Ts = reinterpret_cast<float *>(sm + OFF_TS);
    float *Ys = reinterpret_cast<float *>(sm + OFF_YS);

    const uint32_t idesc_kqk = idesc_bf16(128, 64, false, false);
    const uint32_t idesc_u = idesc_bf16(128, 64, true, false);
    const uint32_t idesc_w = idesc_bf16(128, 64, false, true, true);
    const uint32_t idesc_o = idesc_bf16(64, 128, false, false);
    const uint32_t idesc_d = idesc_bf16(128, 128, false, true);

    if (warp < 8) {
        // ================================================================ prep
        const int w = tid;
        const int qd = warp & 3, half = warp >> 2;   // TMEM lane quadrant, column half
        const int lrow = qd * 32 + (tid & 31);       // TMEM lane = accumulator row
        const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
        bool issued = false;
        for (int k = 0; k < NC; ++k) {
            const int st = k & 1, sl = k % NSCAL;
            const int c = min(C, T - k * C);
            const Scal S = scal(sm, sl);
            const uint32_t kq_a = sbase + OFF_KQ + st * KQ_BYTES;
            const uint32_t v_a = sbase + OFF_V + st * V_BYTES;

            bool ok = role_wait(bar(B_FULL0 + st), (uint32_t)(k >> 1) & 1u, a.limit_ns, &s_abort);
            if (!named_and(BAR_PREP, NPREP, ok)) break;
            if (w == 0) {   // [K;Q] K^T  (the accumulator was read out last chunk)
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ad = kq_a + (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + TM_KQK, sdesc_sw128(ad, 16, 1024), sdesc_sw128(ad, 16, 1024),
                             idesc_kqk, kk > 0);
                }
                mma_commit(bar(B_KQK));
                issued = true;
            }

            // A = strict_lower(diag(beta gamma) K K^T diag(1/gamma)), P = lower(Q K^T) / gamma_C
            ok = role_wait(bar(B_SCAL0 + sl), (uint32_t)(k / NSCAL) & 1u, a.limit_ns, &s_abort);
            if (ok) ok = role_wait(bar(B_KQK), (uint32_t)k & 1u, a.limit_ns, &s_abort);
            // A's space holds Lb / Lbg of chunk k-1 until its U / Wk products are done
            if (ok && k > 0) ok = role_wait(bar(B_UWK), (uint32_t)(k - 1) & 1u, a.limit_ns, &s_abort);
            // P's buffer holds P of chunk k-2 until that chunk's output product is done
            if (ok && k > 1)
                ok = role_wait(bar(B_PFREE0 + st), (uint32_t)((k - 2) >> 1) & 1u, a.limit_ns, &s_abort);
            if (!named_and(BAR_PREP, NPREP, ok)) break;
            const float igC = 1.f / s_gC[sl];
            tc_fence_after();
            {   // this thread: accumulator row lrow, columns 32 half .. 32 half + 31
                const int h = half;
                float v[32];
                tmem_ld32(tl + TM_KQK + h * 32, v);
                tmem_wait_ld();
                if (lrow < 64) {
                    const int r = lrow;
                    const float br = (r < c) ? S.bg[r] : 0.f;
#pragma unroll
                    for (int s4 = 0; s4 < 32; s4 += 4) {
                        const int s0 = h * 32 + s4;
                        const float4 ig4 = *reinterpret_cast<const float4 *>(&S.ig[s0]);
                        float4 o;
                        o.x = (s0 + 0 < r) ? br * v[s4 + 0] * ig4.x : 0.f;
                        o.y = (s0 + 1 < r) ? br * v[s4 + 1] * ig4.y : 0.f;
                        o.z = (s0 + 2 < r) ? br * v[s4 + 2] * ig4.z : 0.f;
                        o.w = (s0 + 3 < r) ? br * v[s4 + 3] * ig4.w : 0.f;
                        *reinterpret_cast<float4 *>(&As[r * LDA + s0]) = o;
                    }
                } else {
                    const int r = lrow - 64;
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = (h * 32 + e <= r && r < c) ? v[e] * igC : 0.f;
                    st_halfrow_bf16(sm + OFF_P + st * 8192, r, h, v);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_PREP, NPREP);

            solve_unit_lower(w, As, Ts, Ys);
            {   // Lb = (T - I) diag(beta) + diag(bf16(beta)), Lbg likewise with beta gamma;
                // thread -> (matrix w / 128, row w % 64, column half (w / 64) % 2)
                const int r = w & 63, mat = w >> 7;
                const float *sc = mat ? S.bg : S.bs;
                uint8_t *dst = sm + (mat ? OFF_LBG : OFF_LB);
                {
                    const int h = (w >> 6) & 1;
                    float v[32];
#pragma unroll
                    for (int s4 = 0; s4 < 32; s4 += 4) {
                        const int s0 = h * 32 + s4;
                        const float4 t = *reinterpret_cast<const float4 *>(&Ts[r * LDA + s0]);
                        const float4 f = *reinterpret_cast<const float4 *>(&sc[s0]);
                        v[s4 + 0] = (s0 + 0 < r) ? t.x * f.x : (s0 + 0 == r ? f.x : 0.f);
                        v[s4 + 1] = (s0 + 1 < r) ? t.y * f.y : (s0 + 1 == r ? f.y : 0.f);
                        v[s4 + 2] = (s0 + 2 < r) ? t.z * f.z : (s0 + 2 == r ? f.z : 0.f);
                        v[s4 + 3] = (s0 + 3 < r) ? t.w * f.w : (s0 + 3 == r ? f.w : 0.f);
                    }
                    st_halfrow_bf16(dst, r, h, v);
                }
            }
            named_sync(BAR_PREP, NPREP);     // T is read out; its space takes the residuals
            if (w < 128) {   // Db = diag(beta - bf16(beta)), Dbg = diag(beta gamma - bf16(beta gamma))
                const int r = w & 63;
                const float x = (w < 64) ? S.bs[r] : S.bg[r];
                const float lo = x - __bfloat162float(__float2bfloat16_rn(x));
                uint8_t *dst = sm + ((w < 64) ? OFF_DB : OFF_DBG);
                const __nv_bfloat16 lo16 = __float2bfloat16_rn(lo);
                const uint32_t lo_bits = (uint32_t)*reinterpret_cast<const unsigned short *>(&lo16);
                const uint32_t word = lo_bits << (16 * (r & 1));
                const int wi = (r & 7) >> 1;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const bool here = (r >> 3) == ch;
                    *reinterpret_cast<uint4 *>(dst + r * 128u + ((ch ^ (r & 7u)) << 4)) =
                        make_uint4(here && wi == 0 ? word : 0u, here && wi == 1 ? word : 0u,
                                   here && wi == 2 ? word : 0u, here && wi == 3 ? word : 0u);
                }
            }
            fence_proxy_async_smem();
            // U^T = V^T (Lb + Db)^T into W^T buffer st (free once the chain read chunk k-2's
            // W^T);  Wk^T = K^T (Lbg + Dbg)^T
            ok = (k < 2) || role_wait(bar(B_RWFREE0 + st), (uint32_t)((k - 2) >> 1) & 1u,
                                      a.limit_ns, &s_abort);
            if (ok && k > 0) ok = role_wait(bar(B_WKFREE), (uint32_t)(k - 1) & 1u, a.limit_ns, &s_abort);
            if (!named_and(BAR_PREP, NPREP, ok)) break;
            if (w == 0) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_W + st * 64, sdesc_sw128(v_a + kk * 2048, 8192, 1024),
                             sdesc_sw128(sbase + OFF_LB + kk * 32, 16, 1024), idesc_u, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_W + st * 64, sdesc_sw128(v_a + kk * 2048, 8192, 1024),
                             sdesc_sw128(sbase + OFF_DB + kk * 32, 16, 1024), idesc_u, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_WK, sdesc_sw128(kq_a + kk * 2048, 16384, 1024),
                             sdesc_sw128(sbase + OFF_LBG + kk * 32, 16, 1024), idesc_u, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_WK, sdesc_sw128(kq_a + kk * 2048, 16384, 1024),
                             sdesc_sw128(sbase + OFF_DBG + kk * 32, 16, 1024), idesc_u, 1);
                mma_commit(bar(B_UWK));
            }

        }
        if (s_abort && w == 0 && issued) {   // let this thread's MMAs land before TMEM goes away
            mma_commit(bar(B_DRAINP));
            mbar_wait(bar(B_DRAINP), 0u, kCleanupLimitNs);
        }
    } else if (warp < 12) {
        // ================================================================ chain
        const int w = tid - 256;    // = TMEM lane (row j of the transposed products)
        const int j = w;
        const int lane = w & 31;
        const uint32_t tl = tmem + ((uint32_t)((warp - 8) * 32) << 16);
        bool issued = false;
        bool ok = role_wait(bar(B_SCAL0), 0u, a.limit_ns, &s_abort);
        ok = named_and(BAR_CHAIN, 128, ok);
        if (ok) {
            // initial state: TMEM M^T <- gamma_C(0) M0^T, MT <- bf16(M0^T)
            const float gC = s_gC[0];
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int i = cb * 32 + e;
                    v[e] = a.init ? a.init[((int64_t)bh * D + i) * D + j] : 0.f;
                }
                st_halfrow_bf16(sm + OFF_MT + (cb >> 1) * 16384, j, cb & 1, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] *= gC;
                tmem_st32(tl + TM_M + cb * 32, v);
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_CHAIN, 128);
        }
        for (int n = 0; ok && n < NC; ++n) {
            const int st = n & 1, sl = n % NSCAL, sl1 = (n + 1) % NSCAL;
            const int t0 = n * C;
            const int c = min(C, T - t0);
            const Scal S = scal(sm, sl);
            const uint32_t kq_a = sbase + OFF_KQ + st * KQ_BYTES;
            const bool last = (n + 1 == NC);

            // ---- Wk^T -> WkT (bf16, MN-major, row i = this lane)
            ok = role_wait(bar(B_FULL0 + st), (uint32_t)(n >> 1) & 1u, a.limit_ns, &s_abort);
            if (ok) ok = role_wait(bar(B_UWK), (uint32_t)n & 1u, a.limit_ns, &s_abort);
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float v[32];
                tmem_ld32(tl + TM_WK + h * 32, v);
                tmem_wait_ld();
                st_halfrow_bf16(sm + OFF_WKT, w, h, v);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_CHAIN, 128);
            // ---- W^T = U^T - M^T Wk^T ;  O = Q M
            if (w == 0) {
                mbar_arrive(bar(B_WKFREE));
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + TM_W + st * 64,
                             sdesc_sw128(sbase + OFF_MT + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_WKT + kk * 2048, 16384, 1024), idesc_w, 1);
                mma_commit(bar(B_W));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + TM_O,
                             sdesc_sw128(kq_a + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_MT + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                             idesc_o, kk > 0);
                issued = true;
            }

            // ---- Wt^T[j][s] = W^T[j][s] * gamma_C / gamma_s -> WtT (row j); then D(n)
            ok = role_wait(bar(B_W), (uint32_t)n & 1u, a.limit_ns, &s_abort);
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float v[32];
                tmem_ld32(tl + TM_W + st * 64 + h * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 32; e4 += 4) {
                    const float4 f = *reinterpret_cast<const float4 *>(&S.sc[h * 32 + e4]);
                    v[e4 + 0] *= f.x;
                    v[e4 + 1] *= f.y;
                    v[e4 + 2] *= f.z;
                    v[e4 + 3] *= f.w;
                }
                st_halfrow_bf16(sm + OFF_WTT, j, h, v);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_CHAIN, 128);
            if (w == 0) {
                mbar_arrive(bar(B_RWFREE0 + st));
                tc_fence_after();
                // M^T += Wt^T K ;  O += P Wt
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_M, sdesc_sw128(sbase + OFF_WTT + kk * 32, 16, 1024),
                             sdesc_sw128(kq_a + kk * 2048, 16384, 1024), idesc_d, 1);
                mma_commit(bar(B_D));       // the state update needs only this
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_O, sdesc_sw128(sbase + OFF_P + st * 8192 + kk * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_WTT + kk * 32, 16, 1024), idesc_o, 1);
                mma_commit(bar(B_O2));
            }

            // ---- state: MT <- bf16(M^T_{n+1}); TMEM M^T <- gamma_C(n+1) M^T_{n+1}
            ok = role_wait(bar(B_D), (uint32_t)n & 1u, a.limit_ns, &s_abort);
            // every MMA that reads this input stage is complete: let the copy warp refill it
            if (w == 0 && ok) mbar_arrive(bar(B_OSTAGE0 + st));
            if (ok && !last)
                ok = role_wait(bar(B_SCAL0 + sl1), (uint32_t)((n + 1) / NSCAL) & 1u, a.limit_ns,
                               &s_abort);
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            tc_fence_after();
            {
                const float gn = last ? 1.f : s_gC[sl1];
                float va[32];
                auto consume = [&](int cb, float (&v)[32]) {
                    if (last) {
                        if (a.final_state) {
                            float *f = a.final_state + (int64_t)bh * D * D + j;
#pragma unroll
                            for (int e = 0; e < 32; ++e) f[(int64_t)(cb * 32 + e) * D] = v[e];
                        }
                    } else {
                        st_halfrow_bf16(sm + OFF_MT + (cb >> 1) * 16384, j, cb & 1, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= gn;
                        tmem_st32(tl + TM_M + cb * 32, v);
                    }
                };
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    tmem_ld32(tl + TM_M + cb * 32, va);
                    tmem_wait_ld();
                    consume(cb, va);
                }
                tmem_wait_st();
            }
            // ---- output row r = gamma_r O[r][:]: lanes 0..15 of each quadrant hold
            // rows 16 q .. 16 q + 15 (the M = 64 TMEM layout), 128 columns each
            ok = role_wait(bar(B_O2), (uint32_t)n & 1u, a.limit_ns, &s_abort);
            if (w == 0 && ok) mbar_arrive(bar(B_PFREE0 + st));
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            tc_fence_after();
            {
                const int r = 16 * (warp - 8) + (lane & 15);
                const bool has_row = (lane < 16) && (r < c);
                const float gr = S.gam[r];
                uint4 *orow = reinterpret_cast<uint4 *>(a.out + (row_base + t0 + r) * D);
                float va[32], vb[32];
                auto emit = [&](int cb, const float (&v)[32]) {
                    if (has_row) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 u;
                            u.x = pack_bf16x2(v[q4 * 8 + 0] * gr, v[q4 * 8 + 1] * gr);
                            u.y = pack_bf16x2(v[q4 * 8 + 2] * gr, v[q4 * 8 + 3] * gr);
                            u.z = pack_bf16x2(v[q4 * 8 + 4] * gr, v[q4 * 8 + 5] * gr);
                            u.w = pack_bf16x2(v[q4 * 8 + 6] * gr, v[q4 * 8 + 7] * gr);
                            __stcs(orow + cb * 4 + q4, u);
                        }
                    }
                };
                // warp-wide loads (lanes 16..31 unused); the next block loads while
                // the current one is converted and stored
                tmem_ld32(tl + TM_O + 0, va);
                tmem_wait_ld();
                tmem_ld32(tl + TM_O + 32, vb);
                emit(0, va);
                tmem_wait_ld();
                tmem_ld32(tl + TM_O + 64, va);
                emit(1, vb);
                tmem_wait_ld();
                tmem_ld32(tl + TM_O + 96, vb);
                emit(2, va);
                tmem_wait_ld();
                emit(3, vb);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_CHAIN, 128);
        }
        if (s_abort && w == 0 && issued) {
            mma_commit(bar(B_DRAINC));
            mbar_wait(bar(B_DRAINC), 0u, kCleanupLimitNs);
        }
    } else {
        // ================================================================ copy
        const int lane = tid & 31;
        uint32_t issued[2] = {0, 0};
        auto issue_tma = [&](int n) {     // lane 0 only
            const int st = n & 1;
            const uint32_t b = bar(B_FULL0 + st);
            const uint32_t kq = sbase + OFF_KQ + st * KQ_BYTES;
            const uint32_t vv = sbase + OFF_V + st * V_BYTES;
            mbar_arrive_expect_tx(b, KQ_BYTES + V_BYTES);
            tma_load_3d(kq + 0, &tm_k, b, 0, n * C, bh);
            tma_load_3d(kq + 8192, &tm_q, b, 0, n * C, bh);
            tma_load_3d(kq + 16384, &tm_k, b, 64, n * C, bh);
            tma_load_3d(kq + 24576, &tm_q, b, 64, n * C, bh);
            tma_load_3d(vv + 0, &tm_v, b, 0, n * C, bh);
            tma_load_3d(vv + 8192, &tm_v, b, 64, n * C, bh);
            ++issued[st];
        };
        // Pull the inputs of chunk n into L2 ahead of its shared-memory load, so
        // that the load (issued when a stage frees up) hits L2 rather than HBM.
        auto prefetch_l2 = [&](int n) {   // lane 0 only
            if (n >= NC) return;
            tma_prefetch_3d(&tm_k, 0, n * C, bh);
            tma_prefetch_3d(&tm_k, 64, n * C, bh);
            tma_prefetch_3d(&tm_q, 0, n * C, bh);
            tma_prefetch_3d(&tm_q, 64, n * C, bh);
            tma_prefetch_3d(&tm_v, 0, n * C, bh);
            tma_prefetch_3d(&tm_v, 64, n * C, bh);
        };
        auto load_gb = [&](int n, float (&gv)[2], float (&bv)[2]) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = n * C + 2 * lane + e;
                gv[e] = (t < T) ? a.g[row_base + t] : 0.f;
                bv[e] = (t < T) ? a.beta[row_base + t] : 0.f;
            }
        };
        auto decay = [&](int n, const float (&gv)[2], const float (&bv)[2]) {
            const int sl = n % NSCAL;
            warp_decay(lane, gv, bv, min(C, T - n * C), a.a_min, scal(sm, sl), &s_gC[sl]);
            if (lane == 0) mbar_arrive(bar(B_SCAL0 + sl));
        };
        float gv[2], bv[2];
        for (int n = 0; n < 2 && n < NC; ++n) {
            load_gb(n, gv, bv);
            if (lane == 0) issue_tma(n);
            decay(n, gv, bv);
        }
        if (lane == 0)
            for (int n = 2; n < 2 + kL2Ahead; ++n) prefetch_l2(n);
        if (NC > 2) load_gb(2, gv, bv);
        for (int n = 0; n + 2 < NC; ++n) {   // refill a stage once chunk n is done with it
            const int st = n & 1;
            bool ok = role_wait(bar(B_OSTAGE0 + st), (uint32_t)(n >> 1) & 1u, a.limit_ns, &s_abort);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                issue_tma(n + 2);
                prefetch_l2(n + 2 + kL2Ahead);
            }
            decay(n + 2, gv, bv);
            if (n + 3 < NC) load_gb(n + 3, gv, bv);
        }
        if (s_abort && lane == 0) {
            // at most the latest load of each stage can still be in flight
            for (int st = 0; st < 2; ++st)
                if (issued[st] > 0)
                    mbar_wait(bar(B_FULL0 + st), (issued[st] - 1) & 1u, kCleanupLimitNs);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 12) {
        __syncwarp();
        tmem_dealloc(tmem, TM_COLS);
    }
}

// Two CTAs per head (the value-split kernel) while they fit on the GPU in one
// wave; one CTA per head beyond that, where every SM already has a head.
// GDR_FUSED_VARIANT=single|pair overrides the choice (used by the tests to
// cover both kernels on small shapes).
bool use_pair(int BH) {
    const char *env = std::getenv("GDR_FUSED_VARIANT");
    if (env && std::strcmp(env, "single") == 0) return false;
    if (env && std::strcmp(env, "pair") == 0) return true;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    return 2 * (int64_t)BH <= sms;
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
    if (use_pair(BH))
        return launch_fused_pair(q, k, v, g, beta, a_min, init, out, final_state, BH, T, s);
    // TMA needs 16-byte aligned bases; the output rows are written as 16-byte vectors
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 15)
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
    unsigned a = 0, b = 0;
    e = take_error_word(&a);
    if (e == cudaSuccess) e = take_pair_error_word(&b);
    *value = a | b;
    return e;
}

}  // namespace gdr
