// gdr_fused.cu -- fused chunked prefill of the gated delta rule on the
// 5th-generation tensor core (tcgen05 + TMEM, operands fed by TMA).
//
// One CTA owns one (sequence, head) and walks its chunks of C = 64 tokens in
// order.  Per chunk it does the whole chunked form -- cumulative decay, the
// intra-chunk triangular transform, the state step and the output -- with
// every contraction on the tensor core, and the fp32 state never leaves the
// SM.  HBM sees q, k, v, g, beta once, out once, and the state twice.
//
// The method: with the lower-bounded decay, gamma_r >= a_min^r inside a chunk,
// so 1/gamma and 1/gamma_C are finite and every causal tile -- the diagonal
// (intra-chunk) tile included -- is one dense product with diagonal scalings
// ("What a Trillion-Parameter MoE Model Reveals About the Next Stage of LLM
// Scaling", sections 3.1-3.3; "Architecture Evolution and Training Engineering
// for Trillion-Scale Sparse Multimodal Models", section 3.2).  The scalings are
// applied in fp32 on TMEM accumulators and in registers, not folded into the
// bf16 operands, so q, k and v enter the tensor core exactly as given.
//
// Algebra per chunk (rows r, s; gamma, 1/gamma, gamma_C as usual; M = S^T):
//   A   = strict_lower(diag(beta gamma) K K^T diag(1/gamma)),  T = (I + A)^-1
//   E   = V - diag(gamma) K M_n                 (what the state mispredicts)
//   W   = T diag(beta) E = diag(beta) E + Lb E,  Lb = strict_lower(T) diag(beta)
//   Wt  = diag(gamma_C / gamma) W
//   P   = lower_incl(Q K^T) / gamma_C
//   O   = diag(gamma) (Q M_n + P Wt)
//   M_{n+1} = gamma_C M_n + K^T Wt
// W is the chunked WY/UT form U - Wk M_n (U = T diag(beta) V, Wk = T
// diag(beta gamma) K) regrouped as T diag(beta) (V - diag(gamma) K M_n): the
// same values with two products fewer, and the identity part of T (the
// dominant diag(beta) E) is added in fp32 rather than taken through bf16.
//
// Products (tcgen05.mma, bf16 operands, fp32 accumulators in TMEM):
//   prep   [K;Q] K^T              M = 128, N = 64,  K = 128
//   chain  K M_n                  M = 64,  N = 128, K = 128  -> X
//          X += Lb E              M = 64,  N = 128, K = 64   (X = W afterwards)
//          Q M_n                  M = 64,  N = 128, K = 128  -> O
//          M  += K^T Wt           M = 128, N = 128, K = 64   (M prescaled by gamma_C)
//          O  += P Wt             M = 64,  N = 128, K = 64
// X and O use the M = 64 layout (row r in lane r % 16 + 32 (r / 16)), read and
// written by all four chain warps with the 16x32bx2 TMEM shape.
//
// Warp roles (448 threads):
//   prep  (warps 0-7)  chunk k: A and P from [K;Q]K^T, the triangular solve,
//                      Lb -- state-independent, runs ahead of the chain
//   chain (warps 8-11) chunk n: E, W, Wt, the state update and the output
//   copy  (warp 12)    TMA loads of the inputs, the cumulative decay, L2
//                      prefetch of later chunks
//   MMA   (warp 13)    issues [K;Q]K^T of chunk k+1 as soon as the preparation
//                      has read chunk k's accumulator
// The chain issues its own products; the output epilogue of chunk n runs
// while K M_{n+1} is on the tensor core.
//
// Shared memory (128-byte swizzled operands, 1024-byte aligned):
//   KQ[2]   32 KB  [slab i/64][K rows 0..63 | Q rows 0..63][128 B]   (TMA)
//   V[2]    16 KB  [slab j/64][rows 0..63][128 B]                    (TMA)
//   MS      32 KB  bf16 M_n, [slab j/64][i][128 B]   (MN-major operand)
//   EW      16 KB  bf16 E, then bf16 Wt, [slab j/64][s][128 B]  (MN-major)
//   LP[2]   16 KB  bf16 Lb [r][s] and P [r][s] of one chunk  (K-major)
//   A, T    fp32 64 x 68 each, merge scratch, 4 slots of per-chunk scalars
// TMEM: [K;Q]K^T 64 cols, X 128, O 128, M 128.

#include "gdr_fused_common.cuh"

namespace gdr {
namespace {

constexpr int NT = 448;    // prep (256) + chain (128) + copy (32) + MMA issue (32)
constexpr int NSTAGE = 2;  // input stages
constexpr int NSCAL = 4;   // scalar slots (chunk m uses slot m % 4)

// shared-memory map (bytes from the 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;
constexpr uint32_t KQ_BYTES = 32768;
constexpr uint32_t OFF_V = OFF_KQ + NSTAGE * KQ_BYTES;
constexpr uint32_t V_BYTES = 16384;
constexpr uint32_t OFF_MS = OFF_V + NSTAGE * V_BYTES;     // 32 KB
constexpr uint32_t OFF_EW = OFF_MS + 32768;               // 16 KB
constexpr uint32_t OFF_LP = OFF_EW + 16384;               // 2 x (Lb 8 KB, P 8 KB)
constexpr uint32_t LP_BYTES = 16384;
constexpr uint32_t OFF_AS = OFF_LP + 2 * LP_BYTES;        // 64 x 68 fp32
constexpr uint32_t OFF_TS = OFF_AS + 64 * LDA * 4;        // 64 x 68 fp32
constexpr uint32_t OFF_YS = OFF_TS + 64 * LDA * 4;        // 32 x 40 fp32
constexpr uint32_t OFF_SC = OFF_YS + 32 * LDY * 4;        // 4 slots x 5 x 64 fp32
constexpr uint32_t SMEM_USED = OFF_SC + NSCAL * 5 * 64 * 4;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;         // alignment slack
static_assert(SMEM_ALLOC <= 232448, "exceeds 227 KB of shared memory per CTA");
static_assert(OFF_V % 1024 == 0 && OFF_MS % 1024 == 0 && OFF_EW % 1024 == 0 &&
                  OFF_LP % 1024 == 0,
              "swizzled operands must be 1024-byte aligned");

// TMEM columns
constexpr uint32_t TM_KQK = 0, TM_X = 64, TM_O = 192, TM_M = 320;
constexpr uint32_t TM_COLS = 512;

constexpr int kL2Ahead = 3;   // chunks prefetched into L2 beyond the two staged in SMEM

__device__ __forceinline__ Scal scal(uint8_t *sm, int slot) {
    return scal_at(reinterpret_cast<float *>(sm + OFF_SC) + slot * 5 * 64);
}

// mbarriers of the pipeline (index into s_bar)
enum : int {
    B_FULL0 = 0,                    // copy: TMA inputs of a stage landed (x2)
    B_KQFREE0 = B_FULL0 + NSTAGE,   // chain: every reader of a stage is done (x2)
    B_SCAL0 = B_KQFREE0 + NSTAGE,   // copy: decay scalars of a chunk written (x4)
    B_KQK = B_SCAL0 + NSCAL,        // MMA-warp commit: [K;Q]K^T done
    B_KQKFREE,                      // prep: [K;Q]K^T accumulator read out
    B_LREADY0,                      // prep: Lb and P of buffer b written (x2)
    B_LPFREE0 = B_LREADY0 + 2,      // chain: buffer b read by its last product (x2)
    B_KM = B_LPFREE0 + 2,           // chain commit: X = K M_n done
    B_C3,                           // chain commit: X = W done
    B_D,                            // chain commit: state update (and Q M_n) done
    B_O2,                           // chain commit: output accumulation done
    B_DRAINM, B_DRAINC,             // commits of the error path (MMA warp, chain)
    NUM_BARS
};

__global__ void __launch_bounds__(NT, 1)
fused_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const FusedArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the __shared__ array by pointer
    // arithmetic so that every access through it stays a shared-memory access
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    __shared__ __align__(8) uint64_t s_bar[NUM_BARS];
    __shared__ uint32_t s_tmem;
    __shared__ float s_gC[NSCAL];
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x;
    const SeqView sv = seq_view(a, bh);        // dense [B][H][T] or packed sequences
    const int T = sv.T;
    const int NC = (T + C - 1) / C;
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

    const uint32_t idesc_kqk = idesc_bf16(128, 64, false, false);
    const uint32_t idesc_x = idesc_bf16(64, 128, false, true);   // K-major A, MN-major B
    const uint32_t idesc_d = idesc_bf16(128, 128, true, true);

    if (warp < 8) {
        // ================================================================ prep
        float *As = reinterpret_cast<float *>(sm + OFF_AS);
        float *Ts = reinterpret_cast<float *>(sm + OFF_TS);
        float *Ys = reinterpret_cast<float *>(sm + OFF_YS);
        const int w = tid;
        const int qd = warp & 3, half = warp >> 2;   // TMEM lane quadrant, column half
        const int lrow = qd * 32 + (tid & 31);       // TMEM lane = accumulator row
        const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
        for (int k = 0; k < NC; ++k) {
            const int sl = k % NSCAL, b = k & 1;
            const int c = min(C, T - k * C);
            const Scal S = scal(sm, sl);
            uint8_t *lp = sm + OFF_LP + b * LP_BYTES;

            bool ok = role_wait(bar(B_SCAL0 + sl), (uint32_t)(k / NSCAL) & 1u, a.limit_ns, &s_abort);
            if (ok) ok = role_wait(bar(B_KQK), (uint32_t)k & 1u, a.limit_ns, &s_abort);
            // buffer b holds Lb, P of chunk k-2 until the chain's last product reading them is done
            if (ok && k > 1)
                ok = role_wait(bar(B_LPFREE0 + b), (uint32_t)((k - 2) >> 1) & 1u, a.limit_ns,
                               &s_abort);
            if (!named_and(BAR_PREP, NPREP, ok)) break;
            const float igC = 1.f / s_gC[sl];
            tc_fence_after();
            {   // A = strict_lower(diag(beta gamma) K K^T diag(1/gamma)), P = lower(Q K^T) / gamma_C;
                // this thread: accumulator row lrow, columns 32 half .. 32 half + 31
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
                    st_halfrow_bf16(lp + 8192, r, h, v);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_PREP, NPREP);
            if (w == 0) mbar_arrive(bar(B_KQKFREE));   // the next [K;Q]K^T may start

            solve_unit_lower(w, As, Ts, Ys);
            {   // Lb = strict_lower(T) diag(beta): thread -> row w % 64, columns 16 (w / 64) + 0..15
                const int r = w & 63, q4 = w >> 6;
                float v[16];
#pragma unroll
                for (int s4 = 0; s4 < 16; s4 += 4) {
                    const int s0 = q4 * 16 + s4;
                    const float4 t = *reinterpret_cast<const float4 *>(&Ts[r * LDA + s0]);
                    const float4 f = *reinterpret_cast<const float4 *>(&S.bs[s0]);
                    v[s4 + 0] = (s0 + 0 < r) ? t.x * f.x : 0.f;
                    v[s4 + 1] = (s0 + 1 < r) ? t.y * f.y : 0.f;
                    v[s4 + 2] = (s0 + 2 < r) ? t.z * f.z : 0.f;
                    v[s4 + 3] = (s0 + 3 < r) ? t.w * f.w : 0.f;
                }
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const uint32_t ch = (uint32_t)(q4 * 2 + h2);
                    uint4 u;
                    u.x = pack_bf16x2(v[h2 * 8 + 0], v[h2 * 8 + 1]);
                    u.y = pack_bf16x2(v[h2 * 8 + 2], v[h2 * 8 + 3]);
                    u.z = pack_bf16x2(v[h2 * 8 + 4], v[h2 * 8 + 5]);
                    u.w = pack_bf16x2(v[h2 * 8 + 6], v[h2 * 8 + 7]);
                    *reinterpret_cast<uint4 *>(lp + r * 128u + ((ch ^ (uint32_t)(r & 7)) << 4)) = u;
                }
            }
            fence_proxy_async_smem();
            named_sync(BAR_PREP, NPREP);
            if (w == 0) mbar_arrive(bar(B_LREADY0 + b));
        }
    } else if (warp == 13) {
        // ================================================================ MMA issue
        // [K;Q]K^T of chunk k+1 once stage k+1 has landed and the preparation has read
        // chunk k's accumulator.
        if ((tid & 31) == 0) {
            bool issued = false;
            auto kqk = [&](int k) {
                const uint32_t kq_a = sbase + OFF_KQ + (k & 1) * KQ_BYTES;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t ad = kq_a + (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + TM_KQK, sdesc_sw128(ad, 16, 1024), sdesc_sw128(ad, 16, 1024),
                             idesc_kqk, kk > 0);
                }
                mma_commit(bar(B_KQK));
                issued = true;
            };
            bool ok = NC > 0 && role_wait(bar(B_FULL0), 0u, a.limit_ns, &s_abort);
            if (ok) kqk(0);
            for (int k = 0; ok && k + 1 < NC; ++k) {
                ok = role_wait(bar(B_KQKFREE), (uint32_t)k & 1u, a.limit_ns, &s_abort);
                if (ok)
                    ok = role_wait(bar(B_FULL0 + ((k + 1) & 1)), (uint32_t)((k + 1) >> 1) & 1u,
                                   a.limit_ns, &s_abort);
                if (ok) kqk(k + 1);
            }
            if (s_abort && issued) {   // let this thread's MMAs land before TMEM goes away
                mma_commit(bar(B_DRAINM));
                mbar_wait(bar(B_DRAINM), 0u, kCleanupLimitNs);
            }
        }
        __syncwarp();
    } else if (warp < 12) {
        // ================================================================ chain
        const int w = tid - 256;                 // TMEM lane of the M = 128 state: row i
        const int lane = w & 31, qd = warp - 8;
        const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
        // M = 64 layout: this thread reads row 16 qd + lane % 16, columns 64 (lane / 16) + 0..63
        const int r64 = 16 * qd + (lane & 15), h64 = lane >> 4;
        bool issued = false;

        // out rows of chunk m: gamma_r O[r][:], this thread's row and column half
        auto output_epilogue = [&](int m) {
            const int cm = min(C, T - m * C);
            const Scal Sm = scal(sm, m % NSCAL);
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                float v[32];
                tmem_ld32_m64<64>(tl + TM_O + cb * 32, v);
                tmem_wait_ld();
                if (r64 < cm) {
                    const float gr = Sm.gam[r64];
                    uint4 *orow = reinterpret_cast<uint4 *>(
                        a.out + (sv.gbase + (int64_t)(m * C + r64) * sv.stride) * D + h64 * 64 + cb * 32);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 u;
                        u.x = pack_bf16x2(v[q4 * 8 + 0] * gr, v[q4 * 8 + 1] * gr);
                        u.y = pack_bf16x2(v[q4 * 8 + 2] * gr, v[q4 * 8 + 3] * gr);
                        u.z = pack_bf16x2(v[q4 * 8 + 4] * gr, v[q4 * 8 + 5] * gr);
                        u.w = pack_bf16x2(v[q4 * 8 + 6] * gr, v[q4 * 8 + 7] * gr);
                        __stcs(orow + q4, u);
                    }
                }
            }
        };
        // X = K M_n into TMEM (chunk n's stage)
        auto issue_km = [&](int n) {
            const uint32_t kq_a = sbase + OFF_KQ + (n & 1) * KQ_BYTES;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tmem + TM_X, sdesc_sw128(kq_a + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                         sdesc_sw128(sbase + OFF_MS + kk * 2048, 16384, 1024), idesc_x, kk > 0);
            mma_commit(bar(B_KM));
            issued = true;
        };

        if (NC == 0 && a.final_state) {   // an empty sequence: final state = initial state
            float *fin = a.final_state + ((int64_t)bh * D + w) * D;
            const float *src = a.init ? a.init + ((int64_t)bh * D + w) * D : nullptr;
            for (int e = 0; e < D; ++e) fin[e] = src ? src[e] : 0.f;
        }
        bool ok = NC > 0 && role_wait(bar(B_SCAL0), 0u, a.limit_ns, &s_abort);
        ok = named_and(BAR_CHAIN, 128, ok);
        if (ok) {
            // initial state: TMEM M <- gamma_C(0) M_0, MS <- bf16(M_0); thread = row i
            const float gC = s_gC[0];
            const float *src = a.init ? a.init + ((int64_t)bh * D + w) * D : nullptr;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = src ? src[cb * 32 + e] : 0.f;
                st_halfrow_bf16(sm + OFF_MS + (cb >> 1) * 16384, w, cb & 1, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] *= gC;
                tmem_st32(tl + TM_M + cb * 32, v);
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            ok = role_wait(bar(B_FULL0), 0u, a.limit_ns, &s_abort);
            ok = named_and(BAR_CHAIN, 128, ok);
            if (ok && w == 0) issue_km(0);
        }
        for (int n = 0; ok && n < NC; ++n) {
            const int st = n & 1, b = n & 1, sl = n % NSCAL, sl1 = (n + 1) % NSCAL;
            const Scal S = scal(sm, sl);
            const uint32_t kq_a = sbase + OFF_KQ + st * KQ_BYTES;
            const uint32_t lp_a = sbase + OFF_LP + b * LP_BYTES;
            const bool last = (n + 1 == NC);

            // ---- output of chunk n-1 (its O is complete once O2(n-1) lands), overlapping
            // K M_n on the tensor core
            if (n > 0) {
                ok = role_wait(bar(B_O2), (uint32_t)(n - 1) & 1u, a.limit_ns, &s_abort);
                if (w == 0 && ok) mbar_arrive_relaxed(bar(B_LPFREE0 + (b ^ 1)));
                if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
                tc_fence_after();
                output_epilogue(n - 1);
            }

            // ---- E = V - gamma K M_n -> EW (bf16); X <- beta E (fp32, the identity part of W)
            ok = role_wait(bar(B_KM), (uint32_t)n & 1u, a.limit_ns, &s_abort);
            if (ok) ok = role_wait(bar(B_LREADY0 + b), (uint32_t)(n >> 1) & 1u, a.limit_ns, &s_abort);
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            tc_fence_after();
            {
                const float gr = S.gam[r64], br = S.bs[r64];
                const uint8_t *vrow = sm + OFF_V + st * V_BYTES + h64 * 8192 + r64 * 128;
#pragma unroll 1
                for (int cb = 0; cb < 2; ++cb) {
                    float x[32];
                    tmem_ld32_m64<64>(tl + TM_X + cb * 32, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const uint32_t ch = (uint32_t)(cb * 4 + q4);
                        const uint4 u = *reinterpret_cast<const uint4 *>(
                            vrow + ((ch ^ (uint32_t)(r64 & 7)) << 4));
                        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int p2 = 0; p2 < 4; ++p2) {
                            const float2 f = __bfloat1622float2(
                                *reinterpret_cast<const __nv_bfloat162 *>(&wv[p2]));
                            x[q4 * 8 + 2 * p2 + 0] = fmaf(-gr, x[q4 * 8 + 2 * p2 + 0], f.x);
                            x[q4 * 8 + 2 * p2 + 1] = fmaf(-gr, x[q4 * 8 + 2 * p2 + 1], f.y);
                        }
                    }
                    st_halfrow_bf16(sm + OFF_EW + h64 * 8192, r64, cb, x);
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] *= br;
                    tmem_st32_m64<64>(tl + TM_X + cb * 32, x);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_CHAIN, 128);
            if (w == 0) {   // X += Lb E (so X = W) ;  O = Q M_n
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_X, sdesc_sw128(lp_a + kk * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_EW + kk * 2048, 8192, 1024), idesc_x, 1);
                mma_commit(bar(B_C3));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + TM_O,
                             sdesc_sw128(kq_a + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_MS + kk * 2048, 16384, 1024), idesc_x, kk > 0);
            }

            // ---- Wt = diag(gamma_C / gamma) W -> EW (bf16)
            ok = role_wait(bar(B_C3), (uint32_t)n & 1u, a.limit_ns, &s_abort);
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            tc_fence_after();
            {
                const float sr = S.sc[r64];
#pragma unroll 1
                for (int cb = 0; cb < 2; ++cb) {
                    float x[32];
                    tmem_ld32_m64<64>(tl + TM_X + cb * 32, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] *= sr;
                    st_halfrow_bf16(sm + OFF_EW + h64 * 8192, r64, cb, x);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_CHAIN, 128);
            if (w == 0) {   // M += K^T Wt ;  O += P Wt
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_M, sdesc_sw128(kq_a + kk * 2048, 16384, 1024),
                             sdesc_sw128(sbase + OFF_EW + kk * 2048, 8192, 1024), idesc_d, 1);
                mma_commit(bar(B_D));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_O, sdesc_sw128(lp_a + 8192 + kk * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_EW + kk * 2048, 8192, 1024), idesc_x, 1);
                mma_commit(bar(B_O2));
            }

            // ---- state: MS <- bf16(M_{n+1}); TMEM M <- gamma_C(n+1) M_{n+1}; thread = row i
            ok = role_wait(bar(B_D), (uint32_t)n & 1u, a.limit_ns, &s_abort);
            // every product reading this input stage is complete: let the copy warp refill it
            if (w == 0 && ok) mbar_arrive(bar(B_KQFREE0 + st));
            if (ok && !last)
                ok = role_wait(bar(B_SCAL0 + sl1), (uint32_t)((n + 1) / NSCAL) & 1u, a.limit_ns,
                               &s_abort);
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            tc_fence_after();
            {
                const float gn = last ? 1.f : s_gC[sl1];
                float *fin = (last && a.final_state) ? a.final_state + ((int64_t)bh * D + w) * D
                                                     : nullptr;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    float v[32];
                    tmem_ld32(tl + TM_M + cb * 32, v);
                    tmem_wait_ld();
                    if (last) {
                        if (fin) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) fin[cb * 32 + e] = v[e];
                        }
                    } else {
                        st_halfrow_bf16(sm + OFF_MS + (cb >> 1) * 16384, w, cb & 1, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= gn;
                        tmem_st32(tl + TM_M + cb * 32, v);
                    }
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            if (!last) {   // K M_{n+1} as soon as its stage has landed
                ok = role_wait(bar(B_FULL0 + (st ^ 1)), (uint32_t)((n + 1) >> 1) & 1u, a.limit_ns,
                               &s_abort);
                if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
                if (w == 0) issue_km(n + 1);
            } else {
                named_sync(BAR_CHAIN, 128);
            }
        }
        if (ok) {   // output of the last chunk
            ok = role_wait(bar(B_O2), (uint32_t)(NC - 1) & 1u, a.limit_ns, &s_abort);
            if (named_and(BAR_CHAIN, 128, ok)) {
                tc_fence_after();
                output_epilogue(NC - 1);
            }
        }
        if (s_abort && w == 0 && issued) {
            mma_commit(bar(B_DRAINC));
            mbar_wait(bar(B_DRAINC), 0u, kCleanupLimitNs);
        }
    } else {
        // ================================================================ copy
        const int lane = tid & 31;
        uint32_t issued[NSTAGE] = {0, 0};
        auto issue_tma = [&](int n) {     // lane 0 only
            const int st = n & 1;
            const uint32_t b = bar(B_FULL0 + st);
            const uint32_t kq = sbase + OFF_KQ + st * KQ_BYTES;
            const uint32_t vv = sbase + OFF_V + st * V_BYTES;
            mbar_arrive_expect_tx(b, KQ_BYTES + V_BYTES);
            tma_load_3d(kq + 0, &tm_k, b, 0, sv.tz + n * C, sv.z);
            tma_load_3d(kq + 8192, &tm_q, b, 0, sv.tz + n * C, sv.z);
            tma_load_3d(kq + 16384, &tm_k, b, 64, sv.tz + n * C, sv.z);
            tma_load_3d(kq + 24576, &tm_q, b, 64, sv.tz + n * C, sv.z);
            tma_load_3d(vv + 0, &tm_v, b, 0, sv.tz + n * C, sv.z);
            tma_load_3d(vv + 8192, &tm_v, b, 64, sv.tz + n * C, sv.z);
            ++issued[st];
        };
        // Pull the inputs of chunk n into L2 ahead of its shared-memory load, so
        // that the load (issued when a stage frees up) hits L2 rather than HBM.
        auto prefetch_l2 = [&](int n) {   // lane 0 only
            if (n >= NC) return;
            tma_prefetch_3d(&tm_k, 0, sv.tz + n * C, sv.z);
            tma_prefetch_3d(&tm_k, 64, sv.tz + n * C, sv.z);
            tma_prefetch_3d(&tm_q, 0, sv.tz + n * C, sv.z);
            tma_prefetch_3d(&tm_q, 64, sv.tz + n * C, sv.z);
            tma_prefetch_3d(&tm_v, 0, sv.tz + n * C, sv.z);
            tma_prefetch_3d(&tm_v, 64, sv.tz + n * C, sv.z);
        };
        auto load_gb = [&](int n, float (&gv)[2], float (&bv)[2]) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = n * C + 2 * lane + e;
                gv[e] = (t < T) ? a.g[sv.gbase + (int64_t)t * sv.stride] : 0.f;
                bv[e] = (t < T) ? a.beta[sv.gbase + (int64_t)t * sv.stride] : 0.f;
            }
        };
        auto decay = [&](int n, const float (&gv)[2], const float (&bv)[2]) {
            const int sl = n % NSCAL;
            warp_decay(lane, gv, bv, min(C, T - n * C), a.a_min, scal(sm, sl), &s_gC[sl]);
            if (lane == 0) mbar_arrive(bar(B_SCAL0 + sl));
        };
        float gv[2], bv[2];
        for (int n = 0; n < NSTAGE && n < NC; ++n) {
            load_gb(n, gv, bv);
            if (lane == 0) issue_tma(n);
            decay(n, gv, bv);
        }
        if (lane == 0)
            for (int n = NSTAGE; n < NSTAGE + kL2Ahead; ++n) prefetch_l2(n);
        if (NC > NSTAGE) load_gb(NSTAGE, gv, bv);
        for (int n = 0; n + NSTAGE < NC; ++n) {   // refill a stage once chunk n is done with it
            const int st = n & 1;
            bool ok = role_wait(bar(B_KQFREE0 + st), (uint32_t)(n >> 1) & 1u, a.limit_ns, &s_abort);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                issue_tma(n + NSTAGE);
                prefetch_l2(n + NSTAGE + kL2Ahead);
            }
            decay(n + NSTAGE, gv, bv);
            if (n + NSTAGE + 1 < NC) load_gb(n + NSTAGE + 1, gv, bv);
        }
        if (s_abort && lane == 0) {
            // at most the latest load of each stage can still be in flight
            for (int st = 0; st < NSTAGE; ++st)
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

// A cluster of two CTAs per head while every head's cluster is resident at
// once; one CTA per head beyond that, where every SM already has a head.
// The GDR_OPT_FUSED_VARIANT option forces one (the tests cover both kernels
// on small shapes).
bool use_pair(int BH) {
    const int forced = opt_fused_variant();
    if (forced == 1) return false;
    if (forced == 2) return true;
    return BH <= fused_pair_max_clusters();
}

}  // namespace

bool fused_uses_pair(int BH) { return use_pair(BH); }

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
        return launch_fused_pair(q, k, v, g, beta, a_min, init, out, final_state, BH, T, nullptr,
                                 H, 0, s);
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
    unsigned a = 0, b = 0, c = 0, d = 0, f = 0;
    e = take_error_word(&a);
    if (e == cudaSuccess) e = take_pair_error_word(&b);
    if (e == cudaSuccess) e = take_prep_error_word(&c);
    if (e == cudaSuccess) e = take_chain_error_word(&d);
    if (e == cudaSuccess) e = take_segment_error_word(&f);
    unsigned m = 0, t = 0;
    if (e == cudaSuccess) e = take_mla_error_word(&m);
    if (e == cudaSuccess) e = take_bwd_tc_error_word(&t);
    unsigned r = 0;
    if (e == cudaSuccess) e = take_bwd_error_word(&r);
    *value = a | b | c | d | f | m | t | r;
    return e;
}

cudaError_t launch_fused_varlen(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float a_min, const float *init, void *out,
                                float *final_state, const int *cu_seqlens, int S, int H,
                                int total_T, cudaStream_t s) {
    const int64_t SH = (int64_t)S * H;
    if (SH == 0) return cudaSuccess;
    if (use_pair((int)SH))
        return launch_fused_pair(q, k, v, g, beta, a_min, init, out, final_state, (int)SH, 0,
                                 cu_seqlens, H, total_T, s);
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 15)
        return cudaErrorMisalignedAddress;
    CUtensorMap mq, mk, mv;
    if (!make_map_packed(&mq, q, H, total_T) || !make_map_packed(&mk, k, H, total_T) ||
        !make_map_packed(&mv, v, H, total_T))
        return cudaErrorInvalidValue;
    FusedArgs a{g, beta, init, static_cast<__nv_bfloat16 *>(out), final_state, a_min, 0,
                wait_limit_ns()};
    a.cu_seqlens = cu_seqlens;
    a.H = H;
    a.total_T = total_T;
    cudaError_t e = cudaFuncSetAttribute(fused_prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    fused_prefill_kernel<<<(unsigned)SH, NT, SMEM_ALLOC, s>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

}  // namespace gdr
