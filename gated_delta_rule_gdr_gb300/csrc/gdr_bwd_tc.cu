// gdr_bwd_tc.cu -- the per-chunk gradients of the backward (bf16, dk = dv = 128, chunk
// 64) on the 5th-generation tensor cores.
//
// The backward takes the chunk algebra of "What a Trillion-Parameter MoE Model Reveals
// About the Next Stage of LLM Scaling" (sections 3.1-3.3) in reverse.  Given, per
// chunk, q, k, v, dO, the fp32 dR = T^T dW of the reverse chain, the state at the
// chunk's start S = M^T and the state gradient after it dS' = dM'^T (value-major bf16
// tiles) and W^T (bf16), with D[r][s] = gamma_r / gamma_s:
//   dP = dO W^T,  dA = -strict_lower(dR W^T),  Q K^T,  K K^T
//   X1 = dO M^T,  X2 = dR M^T,  X3 = W dM'^T
//   FP = lower_incl(dP o D),  FA = strict_lower(dA o diag(beta) D)
//   dQ = diag(gamma) X1 + FP K
//   dK = diag(gamma_C / gamma) X3 - diag(gamma beta) X2 + FA K + FA^T K + FP^T Q
//   dv = diag(beta) dR
// and the row reductions the decay and beta gradients need (the same algebra as the
// warp-MMA kernel bwd_chunk_mma_kernel).
//
// Products (tcgen05 kind::f16, bf16 operands from shared memory, fp32 accumulators in
// all 512 TMEM columns; accumulator rows 0-63 are the "lower" lanes L, 64-127 the
// "upper" lanes U, and each stacking puts every quantity a row's epilogue needs in one
// of the two):
//   D1 [0,64)    [dR; dO] W^T          L: dR W^T   U: dP
//   D2 [64,128)  [K; Q] K^T            L: K K^T    U: Q K^T
//   D3 [128,256) [dR; dO] M^T          L: X2       U: X1
//   D4 [256,384) [W; -] dM'^T          L: X3       (U unused)
//   D5 [384,512) [FA; FP] K            L: FA K     U: FP K
//   D6 [0,128)   [FP^T; -] Q + [FA^T; -] K   L: FP^T Q + FA^T K   (after the pair
//                                      epilogue read D1, D2)
// so dK rows come from L lanes and dQ rows from U lanes.  FP^T and FA^T need no
// transposed copy: the K-major FP and FA tiles, read as MN-major operands, are them.
//
// Warps (384 threads, one CTA per SM, persistent over (head, chunk) tasks):
//   0      loads: TMA tiles of k, q (a [K; Q] slab pair), dO, S, dS', W^T; the fp32 dR
//          rows by a bulk copy.  Each region is refilled for the next task as soon
//          as its last reader is done with it.
//   1      TMEM allocation and the MMA issue (one thread).
//   2, 3   conversion: dR -> bf16 operand rows, dv = beta dR, v.dR; gamma, beta;
//          <M, dM'> from the S and dS' tiles.
//   4-11   epilogues: warp w reads TMEM lane quadrant w % 4, column half (w - 4) / 4.
// Every wait is bounded in time; a timeout sets the device error word and every role
// leaves its loop (the epilogue warps decide together with bar.red.and).

#include "gdr_fused_common.cuh"

namespace gdr {
namespace {

namespace bt {
constexpr int NT = 384;                      // threads
constexpr uint32_t OFF_KQ = 0;               // 2 slabs x [k 64 rows | q 64 rows] x 128 B
constexpr uint32_t OFF_RO = 32768;           // 2 slabs x [dR 64 rows | dO 64 rows]
constexpr uint32_t OFF_S = 65536;            // S [j 128 rows][i], 2 slabs of 64 i
constexpr uint32_t OFF_WT = 98304;           // W^T [j 128 rows][s 64]
constexpr uint32_t OFF_DS = 114688;          // dS' [j][i], 2 slabs (also D4's unused half)
constexpr uint32_t OFF_A5 = 147456;          // [FA rows 0-63 | FP rows 64-127] (K = s)
constexpr uint32_t OFF_V = 163840;           // bf16 v rows [64][128] (plain rows)
constexpr uint32_t OFF_DR = 180224;          // fp32 dR rows [64][128]
constexpr uint32_t OFF_SC = 212992;          // per-parity scalars
// scalars of one task parity: gamma, 1/gamma, beta, d log(alpha)/dg (one 1 KB block,
// copied in as the preparation wrote it), v.dR, <M, dM'> (two warps' shares), the row
// sums of the epilogue (two column halves each), the column sums (the partial sums of
// the four 32-row lane quadrants)
constexpr int SC_GAM = 0, SC_IG = 64, SC_BET = 128, SC_DLA = 192, SC_VDR = 256, SC_RED = 320,
              SC_REU = 384, SC_REL = 512, SC_RT = 640, SC_RQ = 768, SC_RK = 896, SC_RZ = 1024,
              SC_COL = 1152, SC_N = 1408;
constexpr uint32_t SMEM_USED = OFF_SC + 2 * SC_N * 4;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 232448, "exceeds 227 KB of shared memory per CTA");
static_assert(OFF_A5 + 16384 == OFF_V && OFF_WT + 16384 == OFF_DS && OFF_V + 16384 == OFF_DR,
              "the unused halves of D4 and D6 read the tile that follows their operand");
static_assert((OFF_SC % 16) == 0 && (SC_N * 4) % 16 == 0, "bulk copies of the scalar blocks");
constexpr uint32_t TM_D1 = 0, TM_D2 = 64, TM_D3 = 128, TM_D4 = 256, TM_D5 = 384, TM_D6 = 0;

enum : int {
    F_KQ = 0, F_WT, F_S, F_DS, F_DO, F_DR, F_V,     // tiles landed (TMA transaction bytes)
    F_SC0, F_SC1,                                   // the scalar block of an even / odd task
    E_KQ, E_WT, E_S, E_DS, E_RO, E_DR, E_V,         // regions free for the next task
                                                    //   (E_KQ: the MMA + the 8 epilogue warps;
                                                    //   E_DR, E_V: the two converter warps)
    B_CONV0,      // converter: dR operand rows, scalars and v.dR of an even / odd task
    B_CONV1,      //   written (2 each; per parity, as B_SFREE)
    B_E1,         // MMA: D1, D2 (and D4) complete
    B_X,          // MMA: D3 complete
    B_A5,         // epilogue: FA and FP written, D1 and D2 read (8)
    B_D56,        // MMA: D5, D6 complete
    B_TFREE,      // epilogue: every accumulator of the task read (8)
    B_SFREE0,     // epilogue: the scalars of an even / odd task used (1 each; one barrier
    B_SFREE1,     //   per parity, so that a wait two tasks back never meets a later phase)
    B_DRAIN,      // MMA: drain on the error path
    NUM_BARS
};
constexpr uint32_t BAR_EPI = 6;   // named barrier of the 256 epilogue threads
constexpr uint32_t BAR_CONV = 7;  // named barrier of the 64 converter threads
}  // namespace bt

// 32 lanes x 16 consecutive 32-bit columns (thread t: lane quadrant base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// byte offset of bf16 element (row, col) of a 128-byte-swizzled K-major tile
__device__ __forceinline__ uint32_t swz_el(uint32_t row, uint32_t col) {
    return row * 128u + ((((col >> 3) ^ (row & 7u)) << 4) | ((col & 7u) << 1));
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

struct BwdTcArgs {
    const __nv_bfloat16 *v;
    const float *tsc, *dR;
    __nv_bfloat16 *dq, *dk, *dv;
    float *dg, *dbeta;
    int T, BH;
    uint64_t limit_ns;
};

__global__ void __launch_bounds__(bt::NT, 1)
bwd_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_s,
                    const __grid_constant__ CUtensorMap tm_ds, const __grid_constant__ CUtensorMap tm_w,
                    const BwdTcArgs a) {
    using namespace bt;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    __shared__ __align__(8) uint64_t s_bar[NUM_BARS];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T, NC = (T + C - 1) / C;
    const int ntask = NC * a.BH;
    auto bar = [&](int i) { return smem_u32(&s_bar[i]); };
    auto scal = [&](int par) { return reinterpret_cast<float *>(sm + OFF_SC) + par * SC_N; };

    if (tid == 0) {
        for (int i = 0; i < NUM_BARS; ++i) {
            uint32_t count = 1;
            if (i == B_CONV0 || i == B_CONV1 || i == E_DR || i == E_V) count = 2;   // converter warps
            if (i == E_S || i == E_DS) count = 9;       // the MMA commit + the 8 epilogue warps
            if (i == B_A5 || i == B_TFREE) count = 8;
            if (i == E_KQ) count = 9;
            mbar_init(bar(i), count);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&s_tmem), 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_o);
        tma_prefetch_desc(&tm_s);
        tma_prefetch_desc(&tm_ds);
        tma_prefetch_desc(&tm_w);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ================================================================ loads
        // Lane 0: the products' operands; lane 1: the converter's rows and the scalar blocks.
        // Each lane waits for its own regions, so a late scalar block never holds back a
        // tile the tensor cores wait for.
        if (lane < 2) {
            int last[F_SC1 + 1];   // the last task whose load each barrier tracks (-1: none)
            for (int b = 0; b <= F_SC1; ++b) last[b] = -1;
            for (int task = blockIdx.x, it = 0; task < ntask; task += gridDim.x, ++it) {
                const int n = task % NC, bh = task / NC, c = min(C, T - n * C);
                const int row0 = n * C;
                const int64_t grow0 = (int64_t)bh * T + row0;
                const uint32_t pe = (uint32_t)(it - 1) & 1u;
                auto free_of = [&](int b) { return it == 0 || role_wait(bar(b), pe, a.limit_ns, &s_abort); };
                if (lane == 0) {
                    if (!free_of(E_WT)) break;
                    mbar_arrive_expect_tx(bar(F_WT), 16384);
                    tma_load_3d(sbase + OFF_WT, &tm_w, bar(F_WT), 0, 0, task);
                    last[F_WT] = it;
                    if (!free_of(E_DS)) break;
                    mbar_arrive_expect_tx(bar(F_DS), 32768);
                    tma_load_3d(sbase + OFF_DS, &tm_ds, bar(F_DS), 0, 0, task);
                    tma_load_3d(sbase + OFF_DS + 16384, &tm_ds, bar(F_DS), 64, 0, task);
                    last[F_DS] = it;
                    if (!free_of(E_RO)) break;
                    mbar_arrive_expect_tx(bar(F_DO), 16384);
                    tma_load_3d(sbase + OFF_RO + 8192, &tm_o, bar(F_DO), 0, row0, bh);
                    tma_load_3d(sbase + OFF_RO + 24576, &tm_o, bar(F_DO), 64, row0, bh);
                    last[F_DO] = it;
                    if (!free_of(E_S)) break;
                    mbar_arrive_expect_tx(bar(F_S), 32768);
                    tma_load_3d(sbase + OFF_S, &tm_s, bar(F_S), 0, 0, task);
                    tma_load_3d(sbase + OFF_S + 16384, &tm_s, bar(F_S), 64, 0, task);
                    last[F_S] = it;
                    if (!free_of(E_KQ)) break;
                    mbar_arrive_expect_tx(bar(F_KQ), 32768);
                    tma_load_3d(sbase + OFF_KQ, &tm_k, bar(F_KQ), 0, row0, bh);
                    tma_load_3d(sbase + OFF_KQ + 8192, &tm_q, bar(F_KQ), 0, row0, bh);
                    tma_load_3d(sbase + OFF_KQ + 16384, &tm_k, bar(F_KQ), 64, row0, bh);
                    tma_load_3d(sbase + OFF_KQ + 24576, &tm_q, bar(F_KQ), 64, row0, bh);
                    last[F_KQ] = it;
                } else {
                    if (!free_of(E_DR)) break;
                    mbar_arrive_expect_tx(bar(F_DR), (uint32_t)c * 512u);
                    bulk_load(sbase + OFF_DR, a.dR + grow0 * D, (uint32_t)c * 512u, bar(F_DR));
                    last[F_DR] = it;
                    if (!free_of(E_V)) break;
                    mbar_arrive_expect_tx(bar(F_V), (uint32_t)c * 256u);
                    bulk_load(sbase + OFF_V, a.v + grow0 * D, (uint32_t)c * 256u, bar(F_V));
                    last[F_V] = it;
                    // the scalar block of this parity: free once the task two back has used it
                    if (it > 1 && !role_wait(bar(B_SFREE0 + (it & 1)), (uint32_t)((it - 2) >> 1) & 1u,
                                             a.limit_ns, &s_abort))
                        break;
                    mbar_arrive_expect_tx(bar(F_SC0 + (it & 1)), 4 * C * 4);
                    bulk_load(sbase + OFF_SC + (uint32_t)(it & 1) * SC_N * 4, a.tsc + (int64_t)task * 4 * C,
                              4 * C * 4, bar(F_SC0 + (it & 1)));
                    last[F_SC0 + (it & 1)] = it;
                }
            }
            // on the error path: wait (bounded) for every load this lane issued, so none
            // lands after the CTA has left
            if (s_abort) {
                for (int b = 0; b <= F_SC1; ++b) {
                    if (last[b] < 0) continue;
                    const int ph = (b == F_SC0 || b == F_SC1) ? (last[b] >> 1) : last[b];
                    mbar_wait(bar(b), (uint32_t)ph & 1u, kCleanupLimitNs);
                }
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issue
        if (lane == 0) {
            constexpr uint32_t id_n64k = idesc_bf16(128, 64, false, false);    // K-major A, B
            constexpr uint32_t id_n64m = idesc_bf16(128, 64, false, true);     // B MN-major
            constexpr uint32_t id_n128m = idesc_bf16(128, 128, false, true);
            constexpr uint32_t id_n128mm = idesc_bf16(128, 128, true, true);   // A and B MN-major
            bool issued = false;
            for (int task = blockIdx.x, it = 0; task < ntask; task += gridDim.x, ++it) {
                const uint32_t pf = (uint32_t)it & 1u;
                bool ok = it == 0 || role_wait(bar(B_TFREE), (uint32_t)(it - 1) & 1u, a.limit_ns, &s_abort);
                ok = ok && role_wait(bar(F_WT), pf, a.limit_ns, &s_abort);
                ok = ok && role_wait(bar(F_DS), pf, a.limit_ns, &s_abort);
                if (!ok) break;
                tc_fence_after();
                // D4 = [W; -] dM'^T: A = W (M = s) MN-major from W^T [j][s], its second M slab
                // the dS' tile that follows; B = dS' (N = i) MN-major; K = j
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + TM_D4, sdesc_sw128(sbase + OFF_WT + kk * 2048, 16384, 1024),
                             sdesc_sw128(sbase + OFF_DS + kk * 2048, 16384, 1024), id_n128mm, kk > 0);
                mma_commit(bar(E_DS));
                issued = true;
                ok = role_wait(bar(B_CONV0 + (it & 1)), (uint32_t)(it >> 1) & 1u, a.limit_ns, &s_abort);
                ok = ok && role_wait(bar(F_DO), pf, a.limit_ns, &s_abort);
                if (!ok) break;
                tc_fence_after();
                // D1 = [dR; dO] W^T: A K-major (K = j, two 64-column slabs), B = W (N = s) MN-major
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + TM_D1, sdesc_sw128(sbase + OFF_RO + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_WT + kk * 2048, 16384, 1024), id_n64m, kk > 0);
                mma_commit(bar(E_WT));
                if (!role_wait(bar(F_KQ), pf, a.limit_ns, &s_abort)) break;
                tc_fence_after();
                // D2 = [K; Q] K^T: both K-major (K = i)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t dkq = sdesc_sw128(sbase + OFF_KQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    mma_bf16(tmem + TM_D2, dkq, dkq, id_n64k, kk > 0);
                }
                mma_commit(bar(B_E1));
                if (!role_wait(bar(F_S), pf, a.limit_ns, &s_abort)) break;
                tc_fence_after();
                // D3 = [dR; dO] M^T: B = S (N = i) MN-major, K = j
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + TM_D3, sdesc_sw128(sbase + OFF_RO + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_S + kk * 2048, 16384, 1024), id_n128m, kk > 0);
                mma_commit(bar(B_X));
                mma_commit(bar(E_S));
                mma_commit(bar(E_RO));
                if (!role_wait(bar(B_A5), pf, a.limit_ns, &s_abort)) break;
                tc_fence_after();
                // D5 = [FA; FP] K: A K-major (K = s), B = K (N = i) MN-major
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_D5, sdesc_sw128(sbase + OFF_A5 + kk * 32, 16, 1024),
                             sdesc_sw128(sbase + OFF_KQ + kk * 2048, 16384, 1024), id_n128m, kk > 0);
                // D6 = [FP^T; -] Q + [FA^T; -] K: the FP and FA tiles read MN-major (M = r, K
                // = s: row s of the tile holds the 64 values of FP^T[., s]); the unused second
                // M slab is the tile that follows each
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_D6, sdesc_sw128(sbase + OFF_A5 + 8192 + kk * 2048, 8192, 1024),
                             sdesc_sw128(sbase + OFF_KQ + 8192 + kk * 2048, 16384, 1024), id_n128mm, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + TM_D6, sdesc_sw128(sbase + OFF_A5 + kk * 2048, 8192, 1024),
                             sdesc_sw128(sbase + OFF_KQ + kk * 2048, 16384, 1024), id_n128mm, 1);
                mma_commit(bar(B_D56));
                mma_commit(bar(E_KQ));
            }
            if (s_abort && issued) {   // let this thread's products land before TMEM goes away
                mma_commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0u, kCleanupLimitNs);
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // ================================================================ conversion
        // The dR rows in (row, 16-byte piece) units: thread t takes piece t % 16 of rows
        // t / 16 + 4 k (k < 16), so that a warp reads and writes two whole rows per
        // instruction (no bank conflicts, coalesced dv).  Everything it reads arrived by
        // bulk copies: plain loads would queue behind every SM's tensor loads.
        const int t = tid - 64, pc = t & 15, rb = t >> 4;
        for (int task = blockIdx.x, it = 0; task < ntask; task += gridDim.x, ++it) {
            const int n = task % NC, bh = task / NC, c = min(C, T - n * C);
            const int64_t row0 = (int64_t)bh * T + n * C;   // global row of chunk row 0
            const uint32_t pf = (uint32_t)it & 1u;
            float *sc = scal(it & 1);
            bool ok = true;
            if (lane == 0) {
                ok = role_wait(bar(F_DR), pf, a.limit_ns, &s_abort);
                if (ok) ok = role_wait(bar(F_V), pf, a.limit_ns, &s_abort);
                if (ok) ok = role_wait(bar(F_SC0 + (it & 1)), (uint32_t)(it >> 1) & 1u, a.limit_ns, &s_abort);
                // the dR operand rows of the last task are read
                if (ok && it > 0) ok = role_wait(bar(E_RO), (uint32_t)(it - 1) & 1u, a.limit_ns, &s_abort);
            }
            // both converter warps decide together (they meet at a barrier below)
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!named_and(BAR_CONV, 64, ok && !s_abort)) break;
            const float *dr = reinterpret_cast<const float *>(sm + OFF_DR);
            float vdk[16];   // this thread's piece of v_r . dR_r for its 16 rows
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int rr = rb + 4 * k;
                const bool in = rr < c;
                float x[8];
                uint4 vv = make_uint4(0u, 0u, 0u, 0u);
                if (in) {
                    const float4 x0 = *reinterpret_cast<const float4 *>(dr + rr * D + 8 * pc);
                    const float4 x1 = *reinterpret_cast<const float4 *>(dr + rr * D + 8 * pc + 4);
                    x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
                    x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
                    vv = *reinterpret_cast<const uint4 *>(sm + OFF_V + (uint32_t)rr * 256u + (uint32_t)pc * 16u);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = 0.f;
                }
                const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
                float vd = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    vd = fmaf(bf_lo(vw[e]), x[2 * e], fmaf(bf_hi(vw[e]), x[2 * e + 1], vd));
                vdk[k] = vd;
                // the operand row: slab pc / 8, 16-byte chunk pc % 8 of row rr
                *reinterpret_cast<uint4 *>(sm + OFF_RO + (uint32_t)(pc >> 3) * 16384u + (uint32_t)rr * 128u +
                                           ((((uint32_t)pc & 7u) ^ ((uint32_t)rr & 7u)) << 4)) =
                    make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                               pack_bf16x2(x[6], x[7]));
                // dv = beta dR over the v piece just read (its own unit: no other thread reads it)
                const float b = sc[SC_BET + rr];
                *reinterpret_cast<uint4 *>(sm + OFF_V + (uint32_t)rr * 256u + (uint32_t)pc * 16u) =
                    make_uint4(pack_bf16x2(b * x[0], b * x[1]), pack_bf16x2(b * x[2], b * x[3]),
                               pack_bf16x2(b * x[4], b * x[5]), pack_bf16x2(b * x[6], b * x[7]));
            }
            // v_r . dR_r: the 16 pieces of a row sit in 16 lanes of one warp; they meet in
            // shared memory (the epilogue's row-sum arrays of this parity, [64 rows][16], are
            // free until the task's epilogue starts), then lane l sums one of the warp's rows
            // (warp shuffles here cost far more than these stores)
            {
                float *part = sc + SC_REU;
#pragma unroll
                for (int k = 0; k < 16; ++k) part[(rb + 4 * k) * 16 + pc] = vdk[k];
                __syncwarp();
                const int row = 4 * (lane >> 1) + 2 * (warp - 2) + (lane & 1);
                float vs = 0.f;
#pragma unroll
                for (int q = 0; q < 16; ++q) vs += part[row * 16 + ((q + lane) & 15)];
                sc[SC_VDR + row] = vs;
            }
            fence_proxy_async_smem();   // the operand rows are read by the tensor cores, dv by a copy
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(B_CONV0 + (it & 1)));
                mbar_arrive(bar(E_DR));   // the dR rows are read: the next task's may land
            }
            // dv: the rows of both converter warps, out by one bulk copy; the v area is free
            // once the copy has read it
            named_sync(BAR_CONV, 64);
            if (t == 0) {
                bulk_store(a.dv + row0 * D, sbase + OFF_V, (uint32_t)c * 256u);
                bulk_commit();
                bulk_wait_read_all();
                mbar_arrive(bar(E_V));
                mbar_arrive(bar(E_V));
            }
        }
    } else {
        // ================================================================ epilogues
        const int qd = warp & 3, h = (warp - 4) >> 2;
        const int lrow = qd * 32 + lane;            // accumulator row (TMEM lane)
        const bool upper = lrow >= 64;
        const int r = lrow & 63;                    // chunk row
        const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
        for (int task = blockIdx.x, it = 0; task < ntask; task += gridDim.x, ++it) {
            const int n = task % NC, bh = task / NC, c = min(C, T - n * C);
            const int64_t grow = (int64_t)bh * T + n * C + r;
            const uint32_t pf = (uint32_t)it & 1u;
            float *sc = scal(it & 1);
            bool ok = true;
            // <M, dM'> over the bf16 state tiles (same layout, so element by element) while
            // the task's first products run; then the two tiles may be refilled
            if (lane == 0) {
                ok = role_wait(bar(F_S), pf, a.limit_ns, &s_abort);
                if (ok) ok = role_wait(bar(F_DS), pf, a.limit_ns, &s_abort);
            }
            if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                const int et = tid - 128;
                float md[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int u = 0; u < 8; ++u) {   // 2048 16-byte pieces of each tile, 256 threads
                    const uint32_t off = (uint32_t)(u * 256 + et) * 16u;
                    const uint4 s4 = *reinterpret_cast<const uint4 *>(sm + OFF_S + off);
                    const uint4 d4 = *reinterpret_cast<const uint4 *>(sm + OFF_DS + off);
                    const uint32_t sw[4] = {s4.x, s4.y, s4.z, s4.w}, dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        md[e] = fmaf(bf_lo(sw[e]), bf_lo(dw[e]), fmaf(bf_hi(sw[e]), bf_hi(dw[e]), md[e]));
                }
                float mds = (md[0] + md[1]) + (md[2] + md[3]);
                for (int off = 16; off > 0; off >>= 1) mds += __shfl_xor_sync(0xffffffffu, mds, off);
                if (lane == 0) {
                    sc[SC_RED + (warp - 4)] = mds;
                    mbar_arrive(bar(E_S));
                    mbar_arrive(bar(E_DS));
                }
            }
            if (lane == 0 && ok) {
                ok = role_wait(bar(B_CONV0 + (it & 1)), (uint32_t)(it >> 1) & 1u, a.limit_ns, &s_abort);
                if (ok) ok = role_wait(bar(F_SC0 + (it & 1)), (uint32_t)(it >> 1) & 1u, a.limit_ns, &s_abort);
                if (ok) ok = role_wait(bar(B_E1), pf, a.limit_ns, &s_abort);
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!named_and(BAR_EPI, 256, ok && !s_abort)) break;
            tc_fence_after();
            const float gr = sc[SC_GAM + r], br = sc[SC_BET + r];
            const bool rin = r < c;
            // ---- pair terms, columns s = 32 h .. 32 h + 31
            float ee[32];
            {
                float p[32], x[32];
                tmem_ld32(tl + TM_D1 + 32 * h, p);   // L: dR W^T   U: dP
                tmem_ld32(tl + TM_D2 + 32 * h, x);   // L: K K^T    U: Q K^T
                tmem_wait_ld();
                float rsum = 0.f, rt = 0.f;
                if (upper) {
                    // FP = lower_incl(dP o D) -> A5 row 64 + r
#pragma unroll
                    for (int s2 = 0; s2 < 32; s2 += 2) {
                        float fp[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int s = 32 * h + s2 + e;
                            const float Dv = gr * sc[SC_IG + s];
                            fp[e] = (rin && s <= r) ? p[s2 + e] * Dv : 0.f;
                            ee[s2 + e] = fp[e] * x[s2 + e];
                            rsum += ee[s2 + e];
                        }
                        *reinterpret_cast<uint32_t *>(sm + OFF_A5 + swz_el((uint32_t)(64 + r), (uint32_t)(32 * h + s2))) =
                            pack_bf16x2(fp[0], fp[1]);
                    }
                    sc[SC_REU + 64 * h + r] = rsum;
                } else {
                    // FA = strict_lower(dA o beta D), dA = -dR W^T -> A5 row r
#pragma unroll
                    for (int s2 = 0; s2 < 32; s2 += 2) {
                        float fa[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int s = 32 * h + s2 + e;
                            const float Dv = gr * sc[SC_IG + s];
                            const bool lo = rin && s < r;
                            const float dA = -p[s2 + e], dkk = Dv * x[s2 + e];
                            fa[e] = lo ? dA * br * Dv : 0.f;
                            ee[s2 + e] = lo ? dA * br * dkk : 0.f;
                            rt += lo ? dA * dkk : 0.f;
                            rsum += ee[s2 + e];
                        }
                        *reinterpret_cast<uint32_t *>(sm + OFF_A5 + swz_el((uint32_t)r, (uint32_t)(32 * h + s2))) =
                            pack_bf16x2(fa[0], fa[1]);
                    }
                    sc[SC_REL + 64 * h + r] = rsum;
                    sc[SC_RT + 64 * h + r] = rt;
                }
            }
            // the operand tiles are complete, D1 and D2 are read: the in-chunk products may run
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_A5));
            // column sums of ee over this warp's 32 rows: a butterfly over the lanes that halves
            // the columns a lane keeps at every step, so that lane l ends with column 32 h + l
            // (the four lane quadrants' partial sums are added in the row phase)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const bool hi = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < o; ++i) {
                    const float send = hi ? ee[i] : ee[i + o];
                    const float keep = hi ? ee[i + o] : ee[i];
                    ee[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            sc[SC_COL + 64 * qd + 32 * h + lane] = ee[0];

            // ---- the state and in-chunk terms: dK rows (L), dQ rows (U), columns 64 h ..
            ok = true;
            if (lane == 0) {
                ok = role_wait(bar(B_X), pf, a.limit_ns, &s_abort);
                if (ok) ok = role_wait(bar(B_D56), pf, a.limit_ns, &s_abort);
                if (ok) ok = role_wait(bar(F_KQ), pf, a.limit_ns, &s_abort);   // the tile's bytes
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!named_and(BAR_EPI, 256, ok && !s_abort)) break;
            tc_fence_after();
            // this row's q (U) or k (L) values, columns 64 h .. 64 h + 63: slab h of the
            // [K; Q] tile, row r (+ 64 for q); then the tile may be refilled
            uint4 rowv[8];
            {
                const uint8_t *rowp = sm + OFF_KQ + (uint32_t)h * 16384u + (uint32_t)(upper ? 64 + r : r) * 128u;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    rowv[u] = *reinterpret_cast<const uint4 *>(rowp + (((uint32_t)u ^ ((uint32_t)r & 7u)) << 4));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(E_KQ));
            uint32_t outv[32];
            float d1 = 0.f, d2 = 0.f;
            const float gC = sc[SC_GAM + c - 1];
            const float sr = __fdividef(gC, gr), gb = gr * br;
#pragma unroll
            for (int g4 = 0; g4 < 4; ++g4) {   // 16 columns i = 64 h + 16 g4 ..
                const uint32_t col = (uint32_t)(64 * h + 16 * g4);
                const uint32_t rw[8] = {rowv[2 * g4].x, rowv[2 * g4].y, rowv[2 * g4].z, rowv[2 * g4].w,
                                        rowv[2 * g4 + 1].x, rowv[2 * g4 + 1].y, rowv[2 * g4 + 1].z,
                                        rowv[2 * g4 + 1].w};
                if (upper) {
                    float x1[16], fk[16];
                    tmem_ld16(tl + TM_D3 + col, x1);
                    tmem_ld16(tl + TM_D5 + col, fk);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        d1 = fmaf(bf_lo(rw[e]), x1[2 * e], fmaf(bf_hi(rw[e]), x1[2 * e + 1], d1));
                        outv[8 * g4 + e] = pack_bf16x2(fmaf(gr, x1[2 * e], fk[2 * e]),
                                                       fmaf(gr, x1[2 * e + 1], fk[2 * e + 1]));
                    }
                } else {
                    float x2[16], x3[16], gk[16], fq[16];
                    tmem_ld16(tl + TM_D3 + col, x2);
                    tmem_ld16(tl + TM_D4 + col, x3);
                    tmem_ld16(tl + TM_D5 + col, gk);
                    tmem_ld16(tl + TM_D6 + col, fq);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        d1 = fmaf(bf_lo(rw[e]), x2[2 * e], fmaf(bf_hi(rw[e]), x2[2 * e + 1], d1));
                        d2 = fmaf(bf_lo(rw[e]), x3[2 * e], fmaf(bf_hi(rw[e]), x3[2 * e + 1], d2));
                        const float o0 = fmaf(sr, x3[2 * e], fmaf(-gb, x2[2 * e], gk[2 * e] + fq[2 * e]));
                        const float o1 =
                            fmaf(sr, x3[2 * e + 1], fmaf(-gb, x2[2 * e + 1], gk[2 * e + 1] + fq[2 * e + 1]));
                        outv[8 * g4 + e] = pack_bf16x2(o0, o1);
                    }
                }
            }
            // every accumulator of the task is read: the next task's products may start
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_TFREE));
            if (rin) {
                uint4 *dst = reinterpret_cast<uint4 *>((upper ? a.dq : a.dk) + grow * D + 64 * h);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    dst[u] = make_uint4(outv[4 * u], outv[4 * u + 1], outv[4 * u + 2], outv[4 * u + 3]);
            }
            if (upper) {
                sc[SC_RQ + 64 * h + r] = d1;
            } else {
                sc[SC_RK + 64 * h + r] = d1;
                sc[SC_RZ + 64 * h + r] = d2;
            }
            named_sync(BAR_EPI, 256);
            // ---- per row: dbeta, db, then dlog(alpha) as the reverse cumulative sum and dg
            if (warp == 4) {
                float red = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) red += sc[SC_RED + w];
                float zsum = 0.f;
                float db[2] = {0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int x = 2 * lane + e;
                    if (x < c) {
                        const float gx = sc[SC_GAM + x], bx = sc[SC_BET + x];
                        const float rk = sc[SC_RK + x] + sc[SC_RK + 64 + x];
                        const float rq = sc[SC_RQ + x] + sc[SC_RQ + 64 + x];
                        const float rz = sc[SC_RZ + x] + sc[SC_RZ + 64 + x];
                        const float dbt = sc[SC_RT + x] + sc[SC_RT + 64 + x];
                        const float col = (sc[SC_COL + x] + sc[SC_COL + 64 + x]) +
                                          (sc[SC_COL + 128 + x] + sc[SC_COL + 192 + x]);
                        const float dbp = sc[SC_REU + x] + sc[SC_REU + 64 + x] + sc[SC_REL + x] +
                                          sc[SC_REL + 64 + x] - col;
                        const int64_t gx_row = (int64_t)bh * T + n * C + x;
                        a.dbeta[gx_row] = dbt + sc[SC_VDR + x] - gx * rk;
                        const float z = gC / gx * rz;
                        zsum += z;
                        db[e] = dbp + gx * rq - gx * bx * rk - z;
                    }
                }
                for (int off = 16; off > 0; off >>= 1) zsum += __shfl_xor_sync(0xffffffffu, zsum, off);
                const float last = zsum + gC * red;   // the chunk's last row, through gamma_C
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
                    const int x = 2 * lane + e;
                    if (x < c) {
                        const int64_t gx_row = (int64_t)bh * T + n * C + x;
                        a.dg[gx_row] = dl[e] * sc[SC_DLA + x];
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_SFREE0 + (it & 1)));
            }
        }
    }

    if (tid == 64) bulk_wait_all();   // the converter's dv copies are complete
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// [X][rows][inner] bf16 tiles as a 3-D tensor: boxes of 64 columns x `rows` rows of one
// tile, 128-byte swizzle
bool make_map_tiles(CUtensorMap *m, const void *ptr, int inner, int rows, int64_t X) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)X};
    cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * rows * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_bwd_chunk_tc(const void *q, const void *k, const void *v, const float *tsc,
                                const void *Wt, const void *Sb, const void *dout, const float *dR,
                                const void *dSb, void *dq, void *dk, void *dv, float *dg,
                                float *dbeta, int BH, int T, cudaStream_t s) {
    if (BH == 0 || T == 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(Wt) | reinterpret_cast<uintptr_t>(Sb) |
         reinterpret_cast<uintptr_t>(dSb) | reinterpret_cast<uintptr_t>(dR) | reinterpret_cast<uintptr_t>(tsc) |
         reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 15)
        return cudaErrorMisalignedAddress;
    const int64_t X = (int64_t)BH * ((T + C - 1) / C);
    if (X > 0x7fffffff) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mo, ms, mds, mw;
    if (!make_map(&mq, q, BH, T) || !make_map(&mk, k, BH, T) || !make_map(&mo, dout, BH, T) ||
        !make_map_tiles(&ms, Sb, D, D, X) || !make_map_tiles(&mds, dSb, D, D, X) ||
        !make_map_tiles(&mw, Wt, C, D, X))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(bwd_chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bt::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int grid = (int)(X < nsm ? X : nsm);
    BwdTcArgs a{static_cast<const __nv_bfloat16 *>(v), tsc, dR,
                static_cast<__nv_bfloat16 *>(dq), static_cast<__nv_bfloat16 *>(dk),
                static_cast<__nv_bfloat16 *>(dv), dg, dbeta, T, BH, wait_limit_ns()};
    bwd_chunk_tc_kernel<<<grid, bt::NT, bt::SMEM_ALLOC, s>>>(mq, mk, mo, ms, mds, mw, a);
    return cudaGetLastError();
}

cudaError_t take_bwd_tc_error_word(unsigned *value) { return take_error_word(value); }

bool make_rows_map(CUtensorMap *m, const void *ptr, int BH, int T) { return make_map(m, ptr, BH, T); }

// The reverse chain's tensor stores: dR (fp32 [BH][T][128]) in boxes of 16 columns x 64
// rows, no swizzle, clipped at T; dM' (bf16 [X][128 j][128 i]) in boxes of 64 i x 16 j with
// the 128-byte swizzle.
bool make_dr_store_map(CUtensorMap *m, void *ptr, int BH, int T) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)T * D * 4};
    cuuint32_t box[3] = {16, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_ds_store_map(CUtensorMap *m, void *ptr, int64_t X) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)D, (cuuint64_t)X};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * D * 2};
    cuuint32_t box[3] = {64, 16, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gdr
