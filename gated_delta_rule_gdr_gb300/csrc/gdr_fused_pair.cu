// gdr_fused_pair.cu -- fused chunked prefill with each head on a cluster of
// two CTAs: the value columns split between them, and the state-independent
// preparation of the chunks alternated between them and shared over DSMEM.
//
// Same method and chunk algebra as the one-CTA-per-head kernel (gdr_fused.cu:
// the lower-bounded decay keeps 1/gamma finite, so every causal tile is one
// dense product with diagonal scalings -- "What a Trillion-Parameter MoE Model
// Reveals About the Next Stage of LLM Scaling", sections 3.1-3.3):
//   E = V - diag(gamma) K M_n,   W = diag(beta) E + Lb E,   Wt = diag(gamma_C/gamma) W,
//   O = diag(gamma) (Q M_n + P Wt),   M_{n+1} = gamma_C M_n + K^T Wt,
// with Lb = strict_lower(T) diag(beta), T = (I + A)^-1, P = lower_incl(Q K^T)/gamma_C.
//
// Work split.  CTA rho (the cluster rank) owns the value columns J = [64 rho,
// 64 rho + 64): the state block M_J = M[:, J] (fp32 in TMEM, bf16 copy MS), E_J,
// W_J, Wt_J and O[:, J].  Those products touch only J.  The preparation of
// chunk k -- [K;Q]K^T, A and P, the triangular solve, Lb -- does not depend on
// J: CTA (k mod 2) does it and writes Lb and P into its own shared memory and
// into its peer's (st.shared::cluster), then arrives on the peer's mbarrier.
// Each CTA so prepares every other chunk and runs the state chain of all of
// them on half the columns.
//
// Products of the chain per chunk (M = 128 accumulators, X in TMEM):
//   X  = [K;Q] MS                      N = 64, K = 128  (rows 0-63 K M_n, 64-127 Q M_n)
//   X += [Lb;0] E                      N = 64, K = 64   (rows 0-63 become W)
//   M += K^T Wt                        N = 64, K = 64
//   X += [0;P] Wt                      N = 64, K = 64   (rows 64-127 become O / gamma)
// where E's bf16 copy feeds the second product and the chain first stores
// diag(beta) E in fp32 over X's rows 0-63, so the identity part of T is exact.
// The zero halves come from an 8 KB zero tile between Lb and P.
//
// Warp roles (448 threads): prep 0-7, chain 8-11 (warps 8-9 own X rows 0-63,
// warps 10-11 rows 64-127), copy 12 (TMA of K and Q, decay, L2 prefetch of
// K, Q and V), MMA 13 ([K;Q]K^T of the chunks this CTA prepares).  The v rows
// of the next chunk are loaded by TMA (issued by a chain thread of warps 10-11)
// into a single buffer as soon as the current chunk's E step has read it.
// Every wait is done by one thread per role, suspended in mbarrier.try_wait,
// and passed on by a named barrier.
//
// Shared memory: KQ[3] 32 KB, MS 16 KB ([i][j] bf16, MN-major), EW 8 KB
// ([s][j] bf16, MN-major; E, then Wt), V 8 KB, LP[2] 24 KB ([Lb | 0 | P], K-major;
// LP[rho] holds the chunks this CTA prepares, LP[1 - rho] its peer's), the fp32
// solve space (A, T), merge scratch, 4 slots of per-chunk scalars.
// TMEM: [K;Q]K^T 64 cols, X[2] 2 x 64, M_J 64.

#include "gdr_fused_common.cuh"

namespace gdr {
namespace {

constexpr int NT = 448;    // prep (256) + chain (128) + copy (32) + MMA issue (32)
constexpr int DVH = 64;    // value columns per CTA
constexpr int NSTAGE = 3;  // input stages
constexpr int NSCAL = 4;   // scalar slots (chunk m uses slot m % 4)

// shared-memory map (bytes from the 1024-aligned base)
constexpr uint32_t OFF_KQ = 0;              // [slab i/64][K rows | Q rows][128 B]
constexpr uint32_t KQ_BYTES = 32768;
constexpr uint32_t OFF_MS = OFF_KQ + NSTAGE * KQ_BYTES;   // 16 KB
constexpr uint32_t OFF_EW = OFF_MS + 16384;               // 8 KB
constexpr uint32_t OFF_VB = OFF_EW + 8192;                // 8 KB: v[chunk rows][J] (TMA)
constexpr uint32_t OFF_LP = OFF_VB + 8192;                // 2 x [Lb 8 KB | zeros 8 KB | P 8 KB]
constexpr uint32_t LP_BYTES = 24576;
constexpr uint32_t LP_P = 16384;                          // offset of P in an LP buffer
constexpr uint32_t OFF_AS = OFF_LP + 2 * LP_BYTES;        // 64 x 68 fp32
constexpr uint32_t OFF_TS = OFF_AS + 64 * LDA * 4;        // 64 x 68 fp32
constexpr uint32_t OFF_YS = OFF_TS + 64 * LDA * 4;        // 32 x 40 fp32
constexpr uint32_t OFF_SC = OFF_YS + 32 * LDY * 4;        // 4 slots x 5 x 64 fp32
constexpr uint32_t SMEM_USED = OFF_SC + NSCAL * 5 * 64 * 4;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;         // alignment slack
static_assert(SMEM_ALLOC <= 232448, "exceeds 227 KB of shared memory per CTA");
static_assert(OFF_MS % 1024 == 0 && OFF_EW % 1024 == 0 && OFF_VB % 1024 == 0 && OFF_LP % 1024 == 0 &&
                  LP_BYTES % 1024 == 0,
              "swizzled operands must be 1024-byte aligned");

// TMEM columns
constexpr uint32_t TM_KQK = 0, TM_X = 64 /* 2 x 64 */, TM_M = 192;
constexpr uint32_t TM_COLS = 256;

constexpr int kL2Ahead = 3;   // chunks prefetched into L2 beyond the three staged in SMEM

__device__ __forceinline__ Scal scal(uint8_t *sm, int slot) {
    return scal_at(reinterpret_cast<float *>(sm + OFF_SC) + slot * 5 * 64);
}

// Output row r (< 64) of a chunk with c valid rows, this CTA's 64 columns:
// out[r][:] = gamma_r X[64 + r][:], X in TMEM at column x (this thread's lane
// = 64 + r); out0 = row 0 of the chunk, rows `orow` elements apart.  One copy
// for both call sites.
__device__ __noinline__ void emit_output_rows(uint32_t x, int r, int c, const float *gam,
                                              __nv_bfloat16 *out0, int64_t orow) {
#pragma unroll 1
    for (int cb = 0; cb < 2; ++cb) {
        float v[32];
        tmem_ld32(x + cb * 32, v);
        tmem_wait_ld();
        if (r < c) {
            const float gr = gam[r];
            uint4 *dst = reinterpret_cast<uint4 *>(out0 + (int64_t)r * orow + cb * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint4 u;
                u.x = pack_bf16x2(v[q4 * 8 + 0] * gr, v[q4 * 8 + 1] * gr);
                u.y = pack_bf16x2(v[q4 * 8 + 2] * gr, v[q4 * 8 + 3] * gr);
                u.z = pack_bf16x2(v[q4 * 8 + 4] * gr, v[q4 * 8 + 5] * gr);
                u.w = pack_bf16x2(v[q4 * 8 + 6] * gr, v[q4 * 8 + 7] * gr);
                __stcs(dst + q4, u);
            }
        }
    }
}

// mbarriers of the pipeline (index into s_bar)
enum : int {
    B_FULL0 = 0,                       // copy: TMA inputs of a stage landed (x3)
    B_KQFREE0 = B_FULL0 + NSTAGE,      // chain: every reader of a stage is done (x3)
    B_SCAL0 = B_KQFREE0 + NSTAGE,      // copy: decay scalars of a chunk written (x4)
    B_KQK = B_SCAL0 + NSCAL,           // MMA-warp commit: [K;Q]K^T done
    B_KQKFREE,                         // prep: [K;Q]K^T accumulator read out
    B_LREADY0,                         // Lb, P of LP buffer b written (x2; b = 1 - rho by the peer)
    B_LPFREE = B_LREADY0 + 2,          // own chain: LP[rho] read by its last product
    B_PEERFREE,                        // peer chain (remote arrive): its copy of LP[rho] read
    B_KM,                              // chain commit: X = [K;Q] MS done
    B_C3,                              // chain commit: X rows 0-63 = W done
    B_D,                               // chain commit: state update done
    B_O2,                              // chain commit (warp 10): X rows 64-127 = O / gamma done
    B_VFULL,                           // chain-issued TMA: v rows of the next chunk landed
    B_DRAINM, B_DRAINC, B_DRAINO,      // commits of the error path
    NUM_BARS
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NT, 1)
fused_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
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
    const int rho = (int)cluster_rank(), peer = rho ^ 1;
    const int bh = blockIdx.x >> 1;
    const int j0 = rho * DVH;                 // first value column of this CTA
    const SeqView sv = seq_view(a, bh);        // dense [B][H][T] or packed sequences
    const int T = sv.T;
    const int NC = (T + C - 1) / C;
    __nv_bfloat16 *const out0 = a.out + sv.gbase * D + j0;   // out row of token 0, columns J
    const int64_t orow = (int64_t)sv.stride * D;             // elements between token rows
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
    {   // the zero tiles between Lb and P of both LP buffers
        uint4 *z0 = reinterpret_cast<uint4 *>(sm + OFF_LP + 8192);
        uint4 *z1 = reinterpret_cast<uint4 *>(sm + OFF_LP + LP_BYTES + 8192);
        for (int i = tid; i < 512; i += NT) z0[i] = z1[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    // both CTAs' barriers are initialised before either touches the other's shared memory
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    const uint32_t idesc_kqk = idesc_bf16(128, 64, false, false);
    const uint32_t idesc_x = idesc_bf16(128, 64, false, true);   // K-major A, MN-major B
    const uint32_t idesc_d = idesc_bf16(128, 64, true, true);

    if (warp < 8) {
        // ================================================================ prep
        // the chunks k = rho, rho + 2, ...; results into LP[rho] here and at the peer
        float *As = reinterpret_cast<float *>(sm + OFF_AS);
        float *Ts = reinterpret_cast<float *>(sm + OFF_TS);
        float *Ys = reinterpret_cast<float *>(sm + OFF_YS);
        const int w = tid;
        const int qd = warp & 3, half = warp >> 2;   // TMEM lane quadrant, column half
        const int lrow = qd * 32 + (tid & 31);       // TMEM lane = accumulator row
        const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
        uint8_t *lp = sm + OFF_LP + rho * LP_BYTES;
        const uint32_t lp_peer = cluster_map(smem_u32(lp), (uint32_t)peer);
        for (int k = rho, j = 0; k < NC; k += 2, ++j) {
            const int sl = k % NSCAL;
            const int c = min(C, T - k * C);
            const Scal S = scal(sm, sl);

            bool ok = true;
            if (w == 0) {   // one thread waits; the named barrier passes the result on
                ok = role_wait(bar(B_SCAL0 + sl), (uint32_t)(k / NSCAL) & 1u, a.limit_ns, &s_abort);
                if (ok) ok = role_wait(bar(B_KQK), (uint32_t)j & 1u, a.limit_ns, &s_abort);
                // LP[rho] here and at the peer hold chunk k-2 until both chains have read it
                if (ok && j > 0)
                    ok = role_wait(bar(B_LPFREE), (uint32_t)(j - 1) & 1u, a.limit_ns, &s_abort);
                if (ok && j > 0)
                    ok = role_wait_cluster(bar(B_PEERFREE), (uint32_t)(j - 1) & 1u, a.limit_ns,
                                           &s_abort);
            }
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
                    for (int q4 = 0; q4 < 4; ++q4) {
                        float p8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int s = h * 32 + q4 * 8 + e;
                            p8[e] = (s <= r && r < c) ? v[q4 * 8 + e] * igC : 0.f;
                        }
                        uint4 u;
                        u.x = pack_bf16x2(p8[0], p8[1]);
                        u.y = pack_bf16x2(p8[2], p8[3]);
                        u.z = pack_bf16x2(p8[4], p8[5]);
                        u.w = pack_bf16x2(p8[6], p8[7]);
                        const uint32_t off =
                            LP_P + (uint32_t)r * 128u + (((uint32_t)(h * 4 + q4) ^ (uint32_t)(r & 7)) << 4);
                        *reinterpret_cast<uint4 *>(lp + off) = u;
                        st_cluster_v4(lp_peer + off, u);
                    }
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
                    const uint32_t off = (uint32_t)r * 128u + ((ch ^ (uint32_t)(r & 7)) << 4);
                    *reinterpret_cast<uint4 *>(lp + off) = u;
                    st_cluster_v4(lp_peer + off, u);
                }
            }
            fence_proxy_async_smem();
            fence_proxy_async_cluster();
            named_sync(BAR_PREP, NPREP);
            if (w == 0) {
                mbar_arrive(bar(B_LREADY0 + rho));
                mbar_arrive_remote(cluster_map(bar(B_LREADY0 + rho), (uint32_t)peer));
            }
        }
    } else if (warp == 13) {
        // ================================================================ MMA issue
        // [K;Q]K^T of this CTA's chunks k = rho, rho + 2, ...: each once its stage has
        // landed and the preparation has read the previous one's accumulator.
        if ((tid & 31) == 0) {
            bool issued = false;
            for (int k = rho, j = 0; k < NC; k += 2, ++j) {
                bool ok = (j == 0) ||
                          role_wait(bar(B_KQKFREE), (uint32_t)(j - 1) & 1u, a.limit_ns, &s_abort);
                if (ok)
                    ok = role_wait(bar(B_FULL0 + k % NSTAGE), (uint32_t)(k / NSTAGE) & 1u, a.limit_ns,
                                   &s_abort);
                if (!ok) break;
                const uint64_t dkq = sdesc_sw128(sbase + OFF_KQ + (k % NSTAGE) * KQ_BYTES, 16, 1024);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t d = sdesc_add(dkq, (kk >> 2) * 16384 + (kk & 3) * 32);
                    mma_bf16(tmem + TM_KQK, d, d, idesc_kqk, kk > 0);
                }
                mma_commit(bar(B_KQK));
                issued = true;
            }
            if (s_abort && issued) {   // let this thread's MMAs land before TMEM goes away
                mma_commit(bar(B_DRAINM));
                mbar_wait(bar(B_DRAINM), 0u, kCleanupLimitNs);
            }
        }
        __syncwarp();
    } else if (warp < 12) {
        // ================================================================ chain
        const int w = tid - 256;                 // TMEM lane = row of X and of M_J
        const int qd = warp - 8;
        const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
        bool issued = false, issued_o = false;
        uint32_t issued_v = 0;   // TMA loads of v issued (threads 0 and 64)
        const uint32_t peer_free = cluster_map(bar(B_PEERFREE), (uint32_t)peer);

        // X(n) = [K;Q] MS  (chunk n's stage)
        auto issue_km = [&](int n) {
            const uint64_t da = sdesc_sw128(sbase + OFF_KQ + (n % NSTAGE) * KQ_BYTES, 16, 1024);
            const uint64_t db = sdesc_sw128(sbase + OFF_MS, 8192, 1024);
            const uint32_t dst = tmem + TM_X + (n & 1) * 64;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(dst, sdesc_add(da, (kk >> 2) * 16384 + (kk & 3) * 32),
                         sdesc_add(db, kk * 2048), idesc_x, kk > 0);
            mma_commit(bar(B_KM));
            issued = true;
        };

        if (NC == 0 && a.final_state) {   // an empty sequence: final state = initial state
            float *fin = a.final_state + ((int64_t)bh * D + w) * D + j0;
            const float *src = a.init ? a.init + ((int64_t)bh * D + w) * D + j0 : nullptr;
            for (int e = 0; e < DVH; ++e) fin[e] = src ? src[e] : 0.f;
        }
        bool ok = NC > 0 && ((w != 0) || role_wait(bar(B_SCAL0), 0u, a.limit_ns, &s_abort));
        ok = named_and(BAR_CHAIN, 128, ok);
        if (ok) {
            // initial state: TMEM M_J <- gamma_C(0) M_0[:, J], MS <- bf16(M_0[:, J]); thread = row i
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
            if (w == 64) {
                mbar_arrive_expect_tx(bar(B_VFULL), 8192);
                tma_load_3d(sbase + OFF_VB, &tm_v, bar(B_VFULL), j0, sv.tz, sv.z);
                issued_v = 1;
            }
        }
        for (int n = 0; ok && n < NC; ++n) {
            // ---- X(n) = [K;Q] MS_n once chunk n's stage has landed (MS_n: the previous
            // iteration's state step, or the initial state)
            if (w == 0)
                ok = role_wait(bar(B_FULL0 + n % NSTAGE), (uint32_t)(n / NSTAGE) & 1u, a.limit_ns,
                               &s_abort);
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            if (w == 0) issue_km(n);
            const int st = n % NSTAGE, b = n & 1, sl = n % NSCAL, sl1 = (n + 1) % NSCAL;
            const int t0 = n * C;
            const int c = min(C, T - t0);
            const Scal S = scal(sm, sl);
            const uint32_t kq_a = sbase + OFF_KQ + st * KQ_BYTES;
            const uint32_t lp_a = sbase + OFF_LP + b * LP_BYTES;
            const uint32_t xcol = TM_X + (n & 1) * 64;
            const bool last = (n + 1 == NC);

            if (w < 64) {
                // ---- E = V - gamma K M_n -> EW (bf16); X rows 0-63 <- beta E (fp32)
                if (w == 0) ok = role_wait(bar(B_VFULL), (uint32_t)n & 1u, a.limit_ns, &s_abort);
                ok = named_and(BAR_EROWS, 64, ok);
                if (w == 0 && ok) ok = role_wait(bar(B_KM), (uint32_t)n & 1u, a.limit_ns, &s_abort);
                ok = named_and(BAR_EROWS, 64, ok);
                tc_fence_after();
                const float gr = S.gam[w], br = S.bs[w];
                // v[t0 + w][J], row w of the v buffer (zero-filled past T by the copy); the
                // buffer is refilled only after the chain barrier that follows this step
                const uint8_t *vrow = sm + OFF_VB + w * 128;
#pragma unroll 1
                for (int cb = 0; cb < (ok ? 2 : 0); ++cb) {
                    float x[32];
                    tmem_ld32(tl + xcol + cb * 32, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const uint4 u = *reinterpret_cast<const uint4 *>(
                            vrow + (((uint32_t)(cb * 4 + q4) ^ (uint32_t)(w & 7)) << 4));
                        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int p2 = 0; p2 < 4; ++p2) {
                            const float2 f = __bfloat1622float2(
                                *reinterpret_cast<const __nv_bfloat162 *>(&wv[p2]));
                            x[q4 * 8 + 2 * p2 + 0] = fmaf(-gr, x[q4 * 8 + 2 * p2 + 0], f.x);
                            x[q4 * 8 + 2 * p2 + 1] = fmaf(-gr, x[q4 * 8 + 2 * p2 + 1], f.y);
                        }
                    }
                    st_halfrow_bf16(sm + OFF_EW, w, cb, x);
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] *= br;
                    tmem_st32(tl + xcol + cb * 32, x);
                }
                tmem_wait_st();
                fence_proxy_async_smem();
            } else if (n > 0) {
                // ---- output of chunk n-1, once its last product has landed
                if (w == 64) ok = role_wait(bar(B_O2), (uint32_t)(n - 1) & 1u, a.limit_ns, &s_abort);
                ok = named_and(BAR_OROWS, 64, ok);
                if (ok) {
                    if (w == 64) {   // chunk n-1's LP buffer is read: free it for its producer
                        if (((n - 1) & 1) == rho) mbar_arrive_relaxed(bar(B_LPFREE));
                        else mbar_arrive_remote_relaxed(peer_free);
                    }
                    tc_fence_after();
                    const int m = n - 1;
                    emit_output_rows(tl + TM_X + (m & 1) * 64, w - 64, min(C, T - m * C),
                                     scal(sm, m % NSCAL).gam, out0 + (int64_t)m * C * orow, orow);
                }
            }
            // Lb of chunk n is needed from here on
            if (ok && w == 0)
                ok = role_wait_cluster(bar(B_LREADY0 + b), (uint32_t)(n >> 1) & 1u, a.limit_ns,
                                       &s_abort);
            tc_fence_before();
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            if (w == 64 && !last) {   // the v buffer is read: refill it with the next chunk's rows
                mbar_arrive_expect_tx(bar(B_VFULL), 8192);
                tma_load_3d(sbase + OFF_VB, &tm_v, bar(B_VFULL), j0, sv.tz + t0 + C, sv.z);
                ++issued_v;
            }
            if (w == 0) {   // X += [Lb; 0] E  (rows 0-63 become W)
                fence_proxy_async_smem();
                tc_fence_after();
                const uint64_t da = sdesc_sw128(lp_a, 16, 1024);
                const uint64_t db = sdesc_sw128(sbase + OFF_EW, 8192, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + xcol, sdesc_add(da, kk * 32), sdesc_add(db, kk * 2048), idesc_x, 1);
                mma_commit(bar(B_C3));
            }

            // ---- Wt = diag(gamma_C / gamma) W -> EW (bf16), warps 8-9
            if (w < 64) {
                if (w == 0) ok = role_wait(bar(B_C3), (uint32_t)n & 1u, a.limit_ns, &s_abort);
                ok = named_and(BAR_EROWS, 64, ok);
                if (ok) {
                    tc_fence_after();
                    const float sr = S.sc[w];
#pragma unroll 1
                    for (int cb = 0; cb < 2; ++cb) {
                        float x[32];
                        tmem_ld32(tl + xcol + cb * 32, x);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) x[e] *= sr;
                        st_halfrow_bf16(sm + OFF_EW, w, cb, x);
                    }
                    fence_proxy_async_smem();
                }
            }
            tc_fence_before();
            if (!named_and(BAR_CHAIN, 128, ok)) { ok = false; break; }
            if (w == 0) {   // M_J += K^T Wt
                tc_fence_after();
                const uint64_t da = sdesc_sw128(kq_a, 16384, 1024);
                const uint64_t db = sdesc_sw128(sbase + OFF_EW, 8192, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_M, sdesc_add(da, kk * 2048), sdesc_add(db, kk * 2048), idesc_d, 1);
                mma_commit(bar(B_D));
            } else if (w == 64) {   // X += [0; P] Wt  (rows 64-127 become O / gamma)
                tc_fence_after();
                const uint64_t da = sdesc_sw128(lp_a + 8192, 16, 1024);
                const uint64_t db = sdesc_sw128(sbase + OFF_EW, 8192, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + xcol, sdesc_add(da, kk * 32), sdesc_add(db, kk * 2048), idesc_x, 1);
                mma_commit(bar(B_O2));
                issued_o = true;
            }

            // ---- state: MS <- bf16(M_{n+1}); TMEM M_J <- gamma_C(n+1) M_{n+1}; thread = row i
            if (w == 0) {
                ok = role_wait(bar(B_D), (uint32_t)n & 1u, a.limit_ns, &s_abort);
                // every product reading this input stage is complete: let the copy warp refill it
                if (ok) mbar_arrive(bar(B_KQFREE0 + st));
                if (ok && !last)
                    ok = role_wait(bar(B_SCAL0 + sl1), (uint32_t)((n + 1) / NSCAL) & 1u,
                                   a.limit_ns, &s_abort);
            }
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
            fence_proxy_async_smem();
            tc_fence_before();
        }
        if (ok && w >= 64) {   // output of the last chunk
            if (w == 64) ok = role_wait(bar(B_O2), (uint32_t)(NC - 1) & 1u, a.limit_ns, &s_abort);
            ok = named_and(BAR_OROWS, 64, ok);
            if (ok) {
                tc_fence_after();
                const int m = NC - 1;
                emit_output_rows(tl + TM_X + (m & 1) * 64, w - 64, min(C, T - m * C),
                                 scal(sm, m % NSCAL).gam, out0 + (int64_t)m * C * orow, orow);
            }
        }
        if (s_abort && w == 0 && issued) {
            mma_commit(bar(B_DRAINC));
            mbar_wait(bar(B_DRAINC), 0u, kCleanupLimitNs);
        }
        if (s_abort && w == 64 && issued_v > 0)   // the latest v load may still be in flight
            mbar_wait(bar(B_VFULL), (issued_v - 1) & 1u, kCleanupLimitNs);
        if (s_abort && w == 64 && issued_o) {
            mma_commit(bar(B_DRAINO));
            mbar_wait(bar(B_DRAINO), 0u, kCleanupLimitNs);
        }
    } else {
        // ================================================================ copy
        const int lane = tid & 31;
        uint32_t issued[NSTAGE] = {0, 0, 0};
        auto issue_tma = [&](int n) {     // lane 0 only
            const int st = n % NSTAGE;
            const uint32_t b = bar(B_FULL0 + st);
            const uint32_t kq = sbase + OFF_KQ + st * KQ_BYTES;
            mbar_arrive_expect_tx(b, KQ_BYTES);
            tma_load_3d(kq + 0, &tm_k, b, 0, sv.tz + n * C, sv.z);
            tma_load_3d(kq + 8192, &tm_q, b, 0, sv.tz + n * C, sv.z);
            tma_load_3d(kq + 16384, &tm_k, b, 64, sv.tz + n * C, sv.z);
            tma_load_3d(kq + 24576, &tm_q, b, 64, sv.tz + n * C, sv.z);
            ++issued[st];
        };
        // Pull the inputs of chunk n into L2 ahead of use (v is read from L2 by the chain).
        auto prefetch_l2 = [&](int n) {   // lane 0 only
            if (n >= NC) return;
            tma_prefetch_3d(&tm_k, 0, sv.tz + n * C, sv.z);
            tma_prefetch_3d(&tm_k, 64, sv.tz + n * C, sv.z);
            tma_prefetch_3d(&tm_q, 0, sv.tz + n * C, sv.z);
            tma_prefetch_3d(&tm_q, 64, sv.tz + n * C, sv.z);
            tma_prefetch_3d(&tm_v, j0, sv.tz + n * C, sv.z);
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
        if (lane == 0)
            for (int n = 0; n < NSTAGE + kL2Ahead; ++n) prefetch_l2(n);
        for (int n = 0; n < NSTAGE && n < NC; ++n) {
            load_gb(n, gv, bv);
            if (lane == 0) issue_tma(n);
            decay(n, gv, bv);
        }
        if (NC > NSTAGE) load_gb(NSTAGE, gv, bv);
        for (int n = 0; n + NSTAGE < NC; ++n) {   // refill a stage once chunk n is done with it
            const int st = n % NSTAGE;
            bool ok = (lane != 0) || role_wait(bar(B_KQFREE0 + st), (uint32_t)(n / NSTAGE) & 1u,
                                               a.limit_ns, &s_abort);
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
    // neither CTA leaves while the other may still write into its shared memory
    cluster_sync();
}

}  // namespace

cudaError_t launch_fused_pair(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, float a_min, const float *init, void *out,
                              float *final_state, int BH, int T, const int *cu_seqlens, int H,
                              int total_T, cudaStream_t s) {
    if (BH == 0 || (cu_seqlens ? total_T : T) == 0) return cudaSuccess;   // callers copy the state
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 15)
        return cudaErrorMisalignedAddress;
    CUtensorMap mq, mk, mv;
    const bool ok = cu_seqlens ? (make_map_packed(&mq, q, H, total_T) &&
                                  make_map_packed(&mk, k, H, total_T) &&
                                  make_map_packed(&mv, v, H, total_T))
                               : (make_map(&mq, q, BH, T) && make_map(&mk, k, BH, T) &&
                                  make_map(&mv, v, BH, T));
    if (!ok) return cudaErrorInvalidValue;
    FusedArgs a{g, beta, init, static_cast<__nv_bfloat16 *>(out), final_state, a_min, T,
                wait_limit_ns(), static_cast<const __nv_bfloat16 *>(v)};
    a.cu_seqlens = cu_seqlens;
    a.H = H;
    a.total_T = total_T;
    cudaError_t e = cudaFuncSetAttribute(fused_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    fused_pair_kernel<<<2 * BH, NT, SMEM_ALLOC, s>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

// Clusters of the pair kernel that can be resident at once on the current device.
int fused_pair_max_clusters() {
    static int cached = -1;
    if (cached >= 0) return cached;
    if (cudaFuncSetAttribute(fused_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_ALLOC) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fused_pair_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cached = n;
    return n;
}

cudaError_t take_pair_error_word(unsigned *value) { return take_error_word(value); }

}  // namespace gdr
