// gdr_fused_pair.cu -- fused chunked prefill with the value columns of each
// head split over two CTAs.
//
// Same method and the same chunk algebra as the one-CTA-per-head kernel in
// gdr_fused.cu (the lower-bounded decay keeps 1/gamma finite, so every causal
// tile is one dense product with diagonal scalings: "What a Trillion-Parameter
// MoE Model Reveals About the Next Stage of LLM Scaling", sections 3.1-3.3).
// What changes is the split of the work.  CTA rho of head bh owns the value
// columns J = [64 rho, 64 rho + 64): its state block M_J = S^T[:, J] (dk x 64,
// fp32, in TMEM), its U_J, W_J, Wt_J, and the output columns O[:, J].  Every
// one of those products touches only J, so the two CTAs never exchange data.
// The state-independent preparation of a chunk (A and P from [K;Q]K^T, the
// triangular solve, Lb / Lbg, Wk) does not depend on J and is done by both
// CTAs; an SM that would otherwise sit idle repeats it.  With half the value
// columns the state chain per chunk halves, and the shared memory saved buys
// a third input stage, so the preparation runs further ahead of the chain.
// The launcher picks this kernel when two CTAs per head still fit on the GPU
// in one wave.
//
// Products per chunk (orientation chosen so that shared-memory copies are
// written row by row from the TMEM rows that hold them):
//   U_J^T  = V_J^T (Lb + Db)^T            M = 64,  N = 64, K = 64   (prep)
//   Wk^T   = K^T (Lbg + Dbg)^T            M = 128, N = 64, K = 64   (prep)
//   W_J^T  = U_J^T - M_J^T Wk^T           M = 64,  N = 64, K = 128  (chain)
//   O_J    = Q M_J (+ P Wt_J)             M = 64,  N = 64, K = 128 (+64)
//   M_J   += K^T Wt_J                     M = 128, N = 64, K = 64
// with the state kept as gamma_C-prescaled fp32 M_J in TMEM and a bf16 copy
// MS = bf16(M_J) ([i][j], the MN-major operand of both W_J^T and O_J).
// Lb = (T - I) diag(beta) + diag(bf16(beta)) and Db = diag(beta - bf16(beta))
// (Lbg, Dbg likewise with beta gamma): the identity part of T enters the
// products as a bf16 value plus its bf16 residual, exact to ~2^-17.
//
// Warp roles (448 threads): prep warps 0-7, chain warps 8-11, copy warp 12,
// and warp 13, which issues the preparation's tensor-core products ([K;Q]K^T
// of the next chunk as soon as its accumulator is read out, U_J^T and Wk^T
// once Lb / Lbg are written), so that the preparation warps never stall on a
// busy tensor-core queue.  The chain issues its own products.
// Shared memory: KQ[3] 32 KB, V_J[3] 8 KB, MS 16 KB, WkT 16 KB, WtT 8 KB,
// P[2] 8 KB, the fp32 solve space (A, T; Lb / Lbg take A's space and Db / Dbg
// T's once the solve is done), the merge scratch and 4 slots of per-chunk
// scalars.
// TMEM: [K;Q]K^T 64 cols, W_J^T 2 x 64 (M = 64 layout), Wk^T 2 x 64, O_J 64
// (M = 64 layout), M_J 64.

#include "gdr_fused_common.cuh"

namespace gdr {
namespace {

constexpr int NT = 448;    // prep (256) + chain (128) + copy (32) + MMA issue (32)
constexpr int DVH = 64;    // value columns per CTA
constexpr int NSTAGE = 3;  // input stages
constexpr int NSCAL = 4;   // scalar slots (chunk m uses slot m % 4)

// shared-memory map (bytes from the 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;              // 3 x 32 KB: [slab i/64][K rows | Q rows][128 B]
constexpr uint32_t KQ_BYTES = 32768;
constexpr uint32_t OFF_V = OFF_KQ + NSTAGE * KQ_BYTES;   // 3 x 8 KB: V[:, J] rows
constexpr uint32_t V_BYTES = 8192;
constexpr uint32_t OFF_MS = OFF_V + NSTAGE * V_BYTES;    // 16 KB: bf16 M_J [i][j]
constexpr uint32_t OFF_WKT = OFF_MS + 16384;             // 16 KB: bf16 Wk^T [i][s]
constexpr uint32_t OFF_WTT = OFF_WKT + 16384;            // 8 KB: bf16 Wt_J^T [j][s]
constexpr uint32_t OFF_P = OFF_WTT + 8192;               // 2 x 8 KB: bf16 P [r][s]
constexpr uint32_t OFF_AS = OFF_P + 2 * 8192;            // 64 x 68 fp32; Lb, Lbg after the solve
constexpr uint32_t OFF_LB = OFF_AS;
constexpr uint32_t OFF_LBG = OFF_AS + 8192;
constexpr uint32_t OFF_TS = OFF_AS + 64 * LDA * 4;       // 64 x 68 fp32; Db, Dbg after the solve
constexpr uint32_t OFF_DB = OFF_TS;
constexpr uint32_t OFF_DBG = OFF_TS + 8192;
constexpr uint32_t OFF_YS = OFF_TS + 64 * LDA * 4;       // 32 x 40 fp32
constexpr uint32_t OFF_SC = OFF_YS + 32 * LDY * 4;       // 4 slots x 5 x 64 fp32
constexpr uint32_t SMEM_USED = OFF_SC + NSCAL * 5 * 64 * 4;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;        // alignment slack
static_assert(SMEM_ALLOC <= 232448, "exceeds 227 KB of shared memory per CTA");
static_assert(OFF_V % 1024 == 0 && OFF_MS % 1024 == 0 && OFF_WKT % 1024 == 0 &&
                  OFF_WTT % 1024 == 0 && OFF_P % 1024 == 0 && OFF_AS % 1024 == 0 &&
                  OFF_TS % 1024 == 0,
              "swizzled operands must be 1024-byte aligned");

// TMEM columns
constexpr uint32_t TM_KQK = 0, TM_W = 64 /* 2 x 64 */, TM_WK = 192 /* 2 x 64 */, TM_O = 320,
                   TM_M = 384;
constexpr uint32_t TM_COLS = 512;

constexpr int kL2Ahead = 3;   // chunks prefetched into L2 beyond the three staged in SMEM

__device__ __forceinline__ Scal scal(uint8_t *sm, int slot) {
    return scal_at(reinterpret_cast<float *>(sm + OFF_SC) + slot * 5 * 64);
}

// mbarriers of the pipeline (index into s_bar)
enum : int {
    B_FULL0 = 0,                       // copy: TMA inputs of a stage landed (x3)
    B_OSTAGE0 = B_FULL0 + NSTAGE,      // chain: every MMA reading a stage is done (x3)
    B_SCAL0 = B_OSTAGE0 + NSTAGE,      // copy: decay scalars of a chunk written (x4)
    B_KQK = B_SCAL0 + NSCAL,           // MMA-warp commit: [K;Q]K^T done
    B_KQKFREE,                         // prep: [K;Q]K^T accumulator read out
    B_LREADY,                          // prep: Lb, Lbg, Db, Dbg of a chunk written
    B_UWK0,                            // MMA-warp commit: U_J^T, Wk^T of buffer b done (x2)
    B_W = B_UWK0 + 2,                  // chain commit: W_J^T done
    B_D,                               // chain commit: state update (and O = Q M) done
    B_O2,                              // chain commit: output accumulation done
    B_WKFREE0,                         // chain: Wk^T buffer b read out (x2)
    B_RWFREE0 = B_WKFREE0 + 2,         // chain: W_J^T buffer b read out (x2)
    B_PFREE0 = B_RWFREE0 + 2,          // chain: P buffer b read by the output product (x2)
    B_DRAINP = B_PFREE0 + 2,           // commits of the error path (MMA warp, chain)
    B_DRAINC,
    NUM_BARS
};

__global__ void __launch_bounds__(NT, 1)
fused_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
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
    const int bh = blockIdx.x >> 1, rho = blockIdx.x & 1;
    const int j0 = rho * DVH;                 // first value column of this CTA
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
    const uint32_t idesc_u = idesc_bf16(64, 64, true, false);
    const uint32_t idesc_wk = idesc_bf16(128, 64, true, false);
    const uint32_t idesc_w = idesc_bf16(64, 64, true, true, true);
    const uint32_t idesc_o1 = idesc_bf16(64, 64, false, true);
    const uint32_t idesc_d = idesc_bf16(128, 64, true, false);
    const uint32_t idesc_o2 = idesc_bf16(64, 64, false, false);

    if (warp < 8) {
        // ================================================================ prep
        const int w = tid;
        const int qd = warp & 3, half = warp >> 2;   // TMEM lane quadrant, column half
        const int lrow = qd * 32 + (tid & 31);       // TMEM lane = accumulator row
        const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
        for (int k = 0; k < NC; ++k) {
            const int sl = k % NSCAL, b = k & 1;
            const int c = min(C, T - k * C);
            const Scal S = scal(sm, sl);

            // A = strict_lower(diag(beta gamma) K K^T diag(1/gamma)), P = lower(Q K^T) / gamma_C
            bool ok = role_wait(bar(B_SCAL0 + sl), (uint32_t)(k / NSCAL) & 1u, a.limit_ns, &s_abort);
            if (ok) ok = role_wait(bar(B_KQK), (uint32_t)k & 1u, a.limit_ns, &s_abort);
            // A's space holds Lb / Lbg of chunk k-1 until its U / Wk products are done
            if (ok && k > 0)
                ok = role_wait(bar(B_UWK0 + (b ^ 1)), (uint32_t)((k - 1) >> 1) & 1u, a.limit_ns,
                               &s_abort);
            // P's buffer holds P of chunk k-2 until that chunk's output product is done
            if (ok && k > 1)
                ok = role_wait(bar(B_PFREE0 + b), (uint32_t)((k - 2) >> 1) & 1u, a.limit_ns,
                               &s_abort);
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
                    st_halfrow_bf16(sm + OFF_P + b * 8192, r, h, v);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_PREP, NPREP);
            if (w == 0) mbar_arrive(bar(B_KQKFREE));   // the next [K;Q]K^T may start

            solve_unit_lower(w, As, Ts, Ys);
            {   // Lb = (T - I) diag(beta) + diag(bf16(beta)), Lbg likewise with beta gamma;
                // thread -> (matrix w / 128, row w % 64, column half (w / 64) % 2)
                const int r = w & 63, mat = w >> 7;
                const float *sc = mat ? S.bg : S.bs;
                uint8_t *dst = sm + (mat ? OFF_LBG : OFF_LB);
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
            named_sync(BAR_PREP, NPREP);
            if (w == 0) mbar_arrive(bar(B_LREADY));    // U_J^T and Wk^T may start
        }
    } else if (warp == 13) {
        // ================================================================ MMA issue
        // [K;Q]K^T of chunk k+1 once chunk k's accumulator is read out; then U_J^T =
        // V_J^T (Lb + Db)^T into W buffer b and Wk^T = K^T (Lbg + Dbg)^T into Wk buffer b,
        // both free once the chain has read chunk k-2's.
        if ((tid & 31) == 0) {
            bool issued = false;
            auto kqk = [&](int k) {
                const uint32_t kq_a = sbase + OFF_KQ + (k % NSTAGE) * KQ_BYTES;
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
            bool ok = role_wait(bar(B_FULL0), 0u, a.limit_ns, &s_abort);
            if (ok) kqk(0);
            for (int k = 0; ok && k < NC; ++k) {
                const int st = k % NSTAGE, b = k & 1;
                if (k + 1 < NC) {
                    ok = role_wait(bar(B_KQKFREE), (uint32_t)k & 1u, a.limit_ns, &s_abort);
                    if (ok)
                        ok = role_wait(bar(B_FULL0 + (k + 1) % NSTAGE),
                                       (uint32_t)((k + 1) / NSTAGE) & 1u, a.limit_ns, &s_abort);
                    if (!ok) break;
                    kqk(k + 1);
                }
                ok = role_wait(bar(B_LREADY), (uint32_t)k & 1u, a.limit_ns, &s_abort);
                if (ok && k > 1)
                    ok = role_wait(bar(B_RWFREE0 + b), (uint32_t)((k - 2) >> 1) & 1u, a.limit_ns,
                                   &s_abort);
                if (ok && k > 1)
                    ok = role_wait(bar(B_WKFREE0 + b), (uint32_t)((k - 2) >> 1) & 1u, a.limit_ns,
                                   &s_abort);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kq_a = sbase + OFF_KQ + st * KQ_BYTES;
                const uint32_t v_a = sbase + OFF_V + st * V_BYTES;
                const uint32_t tw = tmem + TM_W + b * 64, twk = tmem + TM_WK + b * 64;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tw, sdesc_sw128(v_a + kk * 2048, 8192, 1024),
                             sdesc_sw128(sbase + OFF_LB + kk * 32, 16, 1024), idesc_u, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tw, sdesc_sw128(v_a + kk * 2048, 8192, 1024),
                             sdesc_sw128(sbase + OFF_DB + kk * 32, 16, 1024), idesc_u, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(twk, sdesc_sw128(kq_a + kk * 2048, 16384, 1024),
                             sdesc_sw128(sbase + OFF_LBG + kk * 32, 16, 1024), idesc_wk, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(twk, sdesc_sw128(kq_a + kk * 2048, 16384, 1024),
                             sdesc_sw128(sbase + OFF_DBG + kk * 32, 16, 1024), idesc_wk, 1);
                mma_commit(bar(B_UWK0 + b));
            }
            if (s_abort && issued) {   // let this thread's MMAs land before TMEM goes away
                mma_commit(bar(B_DRAINP));
                mbar_wait(bar(B_DRAINP), 0u, kCleanupLimitNs);
            }
        }
        __syncwarp();
    } else if (warp < 12) {
        // ================================================================ chain
        const int w = tid - 256;    // TMEM lane: row i of M_J and of Wk^T
        const int lane = w & 31, qd = warp - 8;
        const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
        // M = 64 layout rows: this thread reads row 16 qd + (lane % 16), column half lane / 16
        const int r64 = 16 * qd + (lane & 15), h64 = lane >> 4;
        bool issued = false;
        bool ok = role_wait(bar(B_SCAL0), 0u, a.limit_ns, &s_abort);
        ok = named_and(BAR_CHAIN, 128, ok);
        if (ok) {
            // initial state: TMEM M_J <- gamma_C(0) M0[:, J], MS <- bf16(M0[:, J])
            const float gC = s_gC[0];
            const float *src = a.init ? a.init + ((int64_t)bh * D + w) * D + j0 : nullptr;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = src ? src[h * 32 + e] : 0.f;
                st_halfrow_bf16(sm + OFF_MS, w, h, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] *= gC;
                tmem_st32(tl + TM_M + h * 32, v);
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_CHAIN, 128);
        }
        for (int n = 0; ok && n < NC; ++n) {
            const int st = n % NSTAGE, b = n & 1, sl = n % NSCAL, sl1 = (n + 1) % NSCAL;
            const int t0 = n * C;
            const int c = min(C, T - t0);
            const Scal S = scal(sm, sl);
            const uint32_t kq_a = sbase + OFF_KQ + st * KQ_BYTES;
            const bool last = (n + 1 == NC);

            // ---- Wk^T -> WkT (bf16, MN-major operand; row i = this lane)
            ok = role_wait(bar(B_FULL0 + st), (uint32_t)(n / NSTAGE) & 1u, a.limit_ns, &s_abort);
            if (ok) ok = role_wait(bar(B_UWK0 + b), (uint32_t)(n >> 1) & 1u, a.limit_ns, &s_abort);
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float v[32];
                tmem_ld32(tl + TM_WK + b * 64 + h * 32, v);
                tmem_wait_ld();
                st_halfrow_bf16(sm + OFF_WKT, w, h, v);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_CHAIN, 128);
            // ---- W_J^T = U_J^T - M_J^T Wk^T ;  O_J = Q M_J
            if (w == 0) {
                mbar_arrive(bar(B_WKFREE0 + b));
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + TM_W + b * 64, sdesc_sw128(sbase + OFF_MS + kk * 2048, 16384, 1024),
                             sdesc_sw128(sbase + OFF_WKT + kk * 2048, 16384, 1024), idesc_w, 1);
                mma_commit(bar(B_W));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + TM_O,
                             sdesc_sw128(kq_a + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_MS + kk * 2048, 16384, 1024), idesc_o1, kk > 0);
                issued = true;
            }

            // ---- Wt_J^T[j][s] = W_J^T[j][s] gamma_C / gamma_s -> WtT (row j); then the state
            // update and the output accumulation
            ok = role_wait(bar(B_W), (uint32_t)n & 1u, a.limit_ns, &s_abort);
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            tc_fence_after();
            {
                float v[32];
                tmem_ld32_m64(tl + TM_W + b * 64, v);
                tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 32; e4 += 4) {
                    const float4 f = *reinterpret_cast<const float4 *>(&S.sc[h64 * 32 + e4]);
                    v[e4 + 0] *= f.x;
                    v[e4 + 1] *= f.y;
                    v[e4 + 2] *= f.z;
                    v[e4 + 3] *= f.w;
                }
                st_halfrow_bf16(sm + OFF_WTT, r64, h64, v);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(BAR_CHAIN, 128);
            if (w == 0) {
                mbar_arrive(bar(B_RWFREE0 + b));
                tc_fence_after();
                // M_J += K^T Wt_J ;  O_J += P Wt_J
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_M, sdesc_sw128(kq_a + kk * 2048, 16384, 1024),
                             sdesc_sw128(sbase + OFF_WTT + kk * 32, 16, 1024), idesc_d, 1);
                mma_commit(bar(B_D));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_O, sdesc_sw128(sbase + OFF_P + b * 8192 + kk * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_WTT + kk * 32, 16, 1024), idesc_o2, 1);
                mma_commit(bar(B_O2));
            }

            // ---- state: MS <- bf16(M_J,n+1); TMEM M_J <- gamma_C(n+1) M_J,n+1
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
                float *fin = (last && a.final_state)
                                 ? a.final_state + ((int64_t)bh * D + w) * D + j0
                                 : nullptr;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    float v[32];
                    tmem_ld32(tl + TM_M + h * 32, v);
                    tmem_wait_ld();
                    if (last) {
                        if (fin) {
#pragma unroll
                            for (int e = 0; e < 32; ++e) fin[h * 32 + e] = v[e];
                        }
                    } else {
                        st_halfrow_bf16(sm + OFF_MS, w, h, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= gn;
                        tmem_st32(tl + TM_M + h * 32, v);
                    }
                }
                tmem_wait_st();
            }
            // ---- output row r = gamma_r O_J[r][:], the column half h64 of this thread
            ok = role_wait(bar(B_O2), (uint32_t)n & 1u, a.limit_ns, &s_abort);
            if (w == 0 && ok) mbar_arrive(bar(B_PFREE0 + b));
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            tc_fence_after();
            {
                float v[32];
                tmem_ld32_m64(tl + TM_O, v);
                tmem_wait_ld();
                if (r64 < c) {
                    const float gr = S.gam[r64];
                    uint4 *orow = reinterpret_cast<uint4 *>(a.out + (row_base + t0 + r64) * D + j0 +
                                                            h64 * 32);
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
        uint32_t issued[NSTAGE] = {0, 0, 0};
        auto issue_tma = [&](int n) {     // lane 0 only
            const int st = n % NSTAGE;
            const uint32_t b = bar(B_FULL0 + st);
            const uint32_t kq = sbase + OFF_KQ + st * KQ_BYTES;
            const uint32_t vv = sbase + OFF_V + st * V_BYTES;
            mbar_arrive_expect_tx(b, KQ_BYTES + V_BYTES);
            tma_load_3d(kq + 0, &tm_k, b, 0, n * C, bh);
            tma_load_3d(kq + 8192, &tm_q, b, 0, n * C, bh);
            tma_load_3d(kq + 16384, &tm_k, b, 64, n * C, bh);
            tma_load_3d(kq + 24576, &tm_q, b, 64, n * C, bh);
            tma_load_3d(vv, &tm_v, b, j0, n * C, bh);
            ++issued[st];
        };
        // Pull the inputs of chunk n into L2 ahead of its shared-memory load.
        auto prefetch_l2 = [&](int n) {   // lane 0 only
            if (n >= NC) return;
            tma_prefetch_3d(&tm_k, 0, n * C, bh);
            tma_prefetch_3d(&tm_k, 64, n * C, bh);
            tma_prefetch_3d(&tm_q, 0, n * C, bh);
            tma_prefetch_3d(&tm_q, 64, n * C, bh);
            tma_prefetch_3d(&tm_v, j0, n * C, bh);
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
        for (int n = 0; n < NSTAGE && n < NC; ++n) {
            load_gb(n, gv, bv);
            if (lane == 0) issue_tma(n);
            decay(n, gv, bv);
        }
        if (lane == 0)
            for (int n = NSTAGE; n < NSTAGE + kL2Ahead; ++n) prefetch_l2(n);
        if (NC > NSTAGE) load_gb(NSTAGE, gv, bv);
        for (int n = 0; n + NSTAGE < NC; ++n) {   // refill a stage once chunk n is done with it
            const int st = n % NSTAGE;
            bool ok = role_wait(bar(B_OSTAGE0 + st), (uint32_t)(n / NSTAGE) & 1u, a.limit_ns,
                                &s_abort);
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

}  // namespace

cudaError_t launch_fused_pair(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, float a_min, const float *init, void *out,
                              float *final_state, int BH, int T, cudaStream_t s) {
    if (BH == 0 || T == 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 15)
        return cudaErrorMisalignedAddress;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, q, BH, T) || !make_map(&mk, k, BH, T) || !make_map(&mv, v, BH, T))
        return cudaErrorInvalidValue;
    FusedArgs a{g, beta, init, static_cast<__nv_bfloat16 *>(out), final_state, a_min, T,
                wait_limit_ns()};
    cudaError_t e = cudaFuncSetAttribute(fused_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    fused_pair_kernel<<<2 * BH, NT, SMEM_ALLOC, s>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

cudaError_t take_pair_error_word(unsigned *value) { return take_error_word(value); }

}  // namespace gdr
