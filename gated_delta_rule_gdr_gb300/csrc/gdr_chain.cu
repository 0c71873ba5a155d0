// gdr_chain.cu -- the sequential half of the two-kernel prefill path: the
// state chain of every (sequence, head) and the chunk outputs, reading the
// [Lb | P] tiles that gdr_prep.cu wrote for every chunk.
//
// Chunk algebra (sections 3.1-3.3 of "What a Trillion-Parameter MoE Model
// Reveals About the Next Stage of LLM Scaling"):
//   E = V - diag(gamma) K M_n,   W = diag(beta) E + Lb E,   Wt = diag(gamma_C/gamma) W,
//   O = diag(gamma) Q M_n + P W,   M_{n+1} = gamma_C M_n + K^T Wt,
// with P = lower_incl(D o Q K^T), D[r][s] = e^(b_r - b_s), from the preparation.
// Every factor here is at most 1 (gamma, gamma_C / gamma, D), so the chain
// holds however far the decay falls over a chunk; where gamma underflows, the
// state's share of the row is below fp32's range anyway.
//
// Work split.  A CTA owns DVH value columns J of one head (DVH = 64: two CTAs
// per head, independent of each other; DVH = 128: one).  The recurrence never
// mixes value columns, so each chain warp c owns 16 columns j = 16 c .. 16 c +
// 15 of J and runs their chain alone, with warp-level MMAs (mma.sync m16n8k16,
// bf16 operands, fp32 accumulators) whose accumulator layout is the A-operand
// layout of the next product: S_J = M_J^T (16 x 128 fp32, rows j) stays in
// registers and feeds X^T = S_J K^T, E^T feeds E^T Lb^T and Wt^T feeds
// S_J = gamma_C S_J + Wt^T K directly.  No chain step waits for another warp
// or for a tensor-memory round trip.
//
// The output leaves the chain: [K;Q] MS_n and [Lb;P] W_n run on the 5th-
// generation tensor cores (tcgen05, M = 128, N = DVH, two accumulators in
// TMEM), issued by an output thread once the chain warps have published MS_n =
// bf16(S_J) and W_n; rows 64-127 of the accumulators are Q M_n and P W_n, which
// the two output warps combine as gamma Q M_n + P W_n into the Q slabs of the
// chunk's stage (Q is
// dead once the products completed) and write out with tensor stores, so the
// output leaves by the TMA engine instead of 32-row scattered stores that
// would share the load/store pipe with the chain warps' ldmatrix traffic.
//
// Warps: chain 0 .. NCH-1 (NCH = DVH / 16), copy NCH (TMA of K, Q, v, the
// [Lb | P] tile by a plain bulk copy, the decay of each stage, L2 prefetch),
// NCH + 1 output products (one thread), output rows NCH + 2 and NCH + 3 (TMEM
// lane quadrants 2 and 3).
// Every mbarrier wait is bounded in time; a timeout sets the device error
// word and makes every role of the CTA leave its loop.
//
// Shared memory: NST stages of [K | Q (two 64-column slabs each) | v[s][J]
// (64-column slabs) | Lb | P], MS ([slab i/64][j][64 i]), the W tiles [2]
// ([j][r]; a chain warp's rows hold E^T first where E is not kept in
// registers), the stage scalars.  Every bf16 tile has
// 128-byte rows with the 16-byte chunks XOR-swizzled by row (the TMA and UMMA
// 128-byte swizzle).

#include "gdr_fused_common.cuh"

namespace gdr {
namespace {

template <int DVH> struct ChainCfg {
    static constexpr int NCH = DVH / 16;                   // chain warps
    static constexpr int NT = 32 * (NCH + 4);
    static constexpr int NST = DVH == 64 ? 3 : 2;          // input stages
    static constexpr uint32_t ST_K = 0, ST_Q = 8192;       // + 16384 per 64-column slab
    static constexpr uint32_t ST_V = 32768;                // DVH / 64 slabs of 8 KB
    static constexpr uint32_t ST_LP = ST_V + DVH * 128;    // [Lb | P]
    static constexpr uint32_t ST_BYTES = ST_LP + TILE_BYTES;
    static constexpr int MSB = DVH == 64 ? 2 : 1;           // MS buffers (as shared memory allows)
    // E^T stays in registers as the A operand of E^T Lb^T where registers allow (the
    // 256-thread CTA); else it goes through the warp's rows of the Wt tile
    static constexpr bool E_REGS = DVH == 64;
    static constexpr uint32_t OFF_MS = NST * ST_BYTES;     // MSB x 2 slabs of DVH x 128 B
    static constexpr uint32_t MS_SLAB = DVH * 128;
    static constexpr uint32_t OFF_WT = OFF_MS + MSB * 2 * MS_SLAB;
    static constexpr uint32_t WT_BYTES = DVH * 128;
    static constexpr uint32_t OFF_SC = OFF_WT + 2 * WT_BYTES;   // a 5 x 64 fp32 slot per stage
    static constexpr uint32_t SMEM_USED = OFF_SC + NST * 5 * 64 * 4;
    static constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
    // accumulators Q M_n and P W_n, each for two chunks in flight
    static constexpr uint32_t TM_COLS = 4 * DVH;
    static constexpr uint32_t TM_PW = 2 * DVH;   // first column of the P W_n pair
    static_assert(SMEM_ALLOC <= 232448, "exceeds 227 KB of shared memory per CTA");
    static_assert(ST_BYTES % 1024 == 0 && OFF_MS % 1024 == 0 && OFF_WT % 1024 == 0 &&
                      ST_LP % 1024 == 0 && MS_SLAB % 1024 == 0,
                  "swizzled tiles must be 1024-byte aligned");
};

// mbarriers (index into s_bar)
enum : int {
    B_FULL0 = 0,          // stage landed (TMA, bulk copy) and its scalars written (x3, count 2)
    B_FREE0 = 3,          // chain warps + output warps done with a stage (x3, count NCH + 1)
    B_MSREADY0 = 6,       // chain warps: MS_m and W_{m-1} published, phase of m on buffer m % 2
                          //   (x2, count NCH)
    B_QMS = 8,            // issue commit: [K;Q] MS_n done (single MS buffer: may be overwritten)
    B_SAFE0 = 9,          // issue commit after [K;Q] MS_{n-1} and [Lb;P] W_{n-2}: chunk n may
                          //   overwrite W[n % 2] and MS[(n + 1) % 2] (x2)
    B_OFULL0 = 11,        // issue commit: accumulator buffer b complete (x2)
    B_OFREE0 = 13,        // output warps: accumulator buffer b read out (x2)
    B_DRAIN = 15,         // commit of the error path
    NUM_BARS = 16
};
constexpr uint32_t BAR_OUT = 5;   // named barrier of the two output warps

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t c8) {
    return row * 128u + ((c8 ^ (row & 7u)) << 4);
}
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}

// Output row r (< 64) of a chunk with c valid rows, NCOL columns from the TMEM
// accumulators at columns x (Q M_n) and y (P W_n), this thread's lane = 64 + r:
// out[r][:] = gamma_r X[64 + r][:] + Y[64 + r][:].
template <int NCOL>
__device__ __noinline__ void emit_rows(uint32_t x, uint32_t y, int r, int c, const float *gam,
                                       __nv_bfloat16 *out0, int64_t orow) {
    const float gr = gam[r];
#pragma unroll 1
    for (int cb = 0; cb < NCOL / 32; ++cb) {
        float v[32], w[32];
        tmem_ld32(x + cb * 32, v);
        tmem_ld32(y + cb * 32, w);
        tmem_wait_ld();
        if (r < c) {
            uint4 *dst = reinterpret_cast<uint4 *>(out0 + (int64_t)r * orow + cb * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint4 u;
                u.x = pack_bf16x2(fmaf(gr, v[q4 * 8 + 0], w[q4 * 8 + 0]), fmaf(gr, v[q4 * 8 + 1], w[q4 * 8 + 1]));
                u.y = pack_bf16x2(fmaf(gr, v[q4 * 8 + 2], w[q4 * 8 + 2]), fmaf(gr, v[q4 * 8 + 3], w[q4 * 8 + 3]));
                u.z = pack_bf16x2(fmaf(gr, v[q4 * 8 + 4], w[q4 * 8 + 4]), fmaf(gr, v[q4 * 8 + 5], w[q4 * 8 + 5]));
                u.w = pack_bf16x2(fmaf(gr, v[q4 * 8 + 6], w[q4 * 8 + 6]), fmaf(gr, v[q4 * 8 + 7], w[q4 * 8 + 7]));
                __stcs(dst + q4, u);
            }
        }
    }
}

// Output row r of a chunk into a 128-byte-swizzled staging tile (64-column slabs
// SLAB bytes apart) for a tensor store: row r = gamma_r X[64 + r][:] + Y[64 + r][:], bf16.
template <int NCOL>
__device__ __noinline__ void stage_rows(uint32_t x, uint32_t y, int r, const float *gam, uint32_t dst,
                                        uint32_t slab) {
    const float gr = gam[r];
#pragma unroll 1
    for (int cb = 0; cb < NCOL / 32; ++cb) {
        float v[32], w[32];
        tmem_ld32(x + cb * 32, v);
        tmem_ld32(y + cb * 32, w);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const uint32_t u0 = pack_bf16x2(fmaf(gr, v[q4 * 8 + 0], w[q4 * 8 + 0]), fmaf(gr, v[q4 * 8 + 1], w[q4 * 8 + 1]));
            const uint32_t u1 = pack_bf16x2(fmaf(gr, v[q4 * 8 + 2], w[q4 * 8 + 2]), fmaf(gr, v[q4 * 8 + 3], w[q4 * 8 + 3]));
            const uint32_t u2 = pack_bf16x2(fmaf(gr, v[q4 * 8 + 4], w[q4 * 8 + 4]), fmaf(gr, v[q4 * 8 + 5], w[q4 * 8 + 5]));
            const uint32_t u3 = pack_bf16x2(fmaf(gr, v[q4 * 8 + 6], w[q4 * 8 + 6]), fmaf(gr, v[q4 * 8 + 7], w[q4 * 8 + 7]));
            const uint32_t addr = dst + (uint32_t)(cb >> 1) * slab + swz((uint32_t)r, (uint32_t)((cb & 1) * 4 + q4));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(u0), "r"(u1), "r"(u2), "r"(u3)
                         : "memory");
        }
    }
}

// SO (states only, with saving): the chain without the output products -- the
// backward's recomputation of the states and W tiles, which needs no output; the
// output thread only stores the published tiles, the copy warp loads no Q or P.
template <int DVH, bool SO>
__global__ void __launch_bounds__(ChainCfg<DVH>::NT, 1)
chain_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
             const __grid_constant__ CUtensorMap tm_sm, const __grid_constant__ CUtensorMap tm_sw,
             const FusedArgs a, const uint8_t *ws,
             int64_t nslot) {
    using Cfg = ChainCfg<DVH>;
    constexpr int NCH = Cfg::NCH, NST = Cfg::NST, SPLIT = 128 / DVH;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the __shared__ array by pointer
    // arithmetic so that every access through it stays a shared-memory access
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    __shared__ __align__(8) uint64_t s_bar[NUM_BARS];
    __shared__ uint32_t s_tmem;
    __shared__ float s_gC[NST];
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x / SPLIT, rho = blockIdx.x % SPLIT;
    const int j0 = rho * DVH;                  // first value column of this CTA
    const SeqView sv = seq_view(a, bh);        // dense [B][H][T] or packed sequences
    const int T = sv.T;
    const int NC = (T + C - 1) / C;
    __nv_bfloat16 *const out0 = a.out + sv.gbase * D + j0;   // out row of token 0, columns J
    const int64_t orow = (int64_t)sv.stride * D;             // elements between token rows
    const uint8_t *tiles = ws + ((int64_t)sv.z * nslot + tile_slot0(a, bh, sv)) * TILE_BYTES;
    auto bar = [&](int i) { return smem_u32(&s_bar[i]); };
    auto stage = [&](int n) { return sbase + (uint32_t)(n % NST) * Cfg::ST_BYTES; };
    auto scal = [&](int n) { return scal_at(reinterpret_cast<float *>(sm + Cfg::OFF_SC) + (n % NST) * 5 * 64); };

    if (tid == 0) {
        for (int i = 0; i < NUM_BARS; ++i) {
            uint32_t count = 1;
            if (i >= B_FULL0 && i < B_FULL0 + 3) count = 2;
            if (i >= B_FREE0 && i < B_FREE0 + 3) count = SO ? NCH : NCH + 1;   // + the output warps
            if (i == B_MSREADY0 || i == B_MSREADY0 + 1) count = NCH;
            mbar_init(bar(i), count);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == NCH) {
        if (!SO) {
            tmem_alloc(smem_u32(&s_tmem), Cfg::TM_COLS);
            tmem_relinquish();
        }
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_o);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = SO ? 0u : s_tmem;

    if (warp < NCH) {
        // ================================================================ chain
        // Warp c: value columns jw .. jw + 15 of J (S_J rows); lane 4g + t holds rows
        // jw + g, jw + g + 8 and the column pairs 8 q + 2 t, +1 of each 8-column tile q.
        const int cw = warp, g = lane >> 2, t4 = lane & 3;
        const int jw = 16 * cw;
        // ldmatrix lane roles for B fragments: from [n][k] rows (non-transposed) ...
        const uint32_t bn_r = (uint32_t)((lane & 7) + (lane >> 4) * 8);
        const uint32_t bn_c = (uint32_t)((lane >> 3) & 1);
        // ... and from [k][n] rows (transposed), which is also the A-fragment
        // pattern of a non-transposed [m][k] load
        const uint32_t bt_r = (uint32_t)((lane & 7) + ((lane >> 3) & 1) * 8);
        const uint32_t bt_c = (uint32_t)(lane >> 4);
        // stmatrix lane roles: matrices (rows 0-7 | 8-15) x (columns 0-7 | 8-15), in the
        // accumulator register order (row g, row g + 8) of one 8-column tile, then the next
        const uint32_t st_r = (uint32_t)((lane & 7) + ((lane >> 3) & 1) * 8);
        const uint32_t st_c = (uint32_t)(lane >> 4);
        float s[16][4];   // S_J: rows jw + g (+ 8), columns i = 8 q + 2 t4 (+ 1)
        float *const fin_view = view_final(a, bh);
        {
            // a segment's initial state comes from the scan kernel just before this one
            if (a.nseg > 1) grid_dependency_wait();
            const float *v0 = view_init(a, bh);
            const float *src = v0 ? v0 + j0 + jw : nullptr;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int i = 8 * q + 2 * t4;
                s[q][0] = src ? src[(int64_t)i * D + g] : 0.f;
                s[q][1] = src ? src[(int64_t)(i + 1) * D + g] : 0.f;
                s[q][2] = src ? src[(int64_t)i * D + g + 8] : 0.f;
                s[q][3] = src ? src[(int64_t)(i + 1) * D + g + 8] : 0.f;
            }
        }
        auto store_state = [&]() {   // S_J^T into the fp32 [dk][dv] final state
            float *fin = fin_view + j0 + jw;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int i = 8 * q + 2 * t4;
                fin[(int64_t)i * D + g] = s[q][0];
                fin[(int64_t)(i + 1) * D + g] = s[q][1];
                fin[(int64_t)i * D + g + 8] = s[q][2];
                fin[(int64_t)(i + 1) * D + g + 8] = s[q][3];
            }
        };
        // Publication m, for the output products: MS_m = bf16(S_J) into buffer m % MSB
        // (rows j, K-major; m < NC) and the W_{m-1} tile stored earlier, behind one
        // fence (the products read them through the async proxy)
        auto publish = [&](int m) {
            if (m < NC) {
                const uint32_t ms = sbase + Cfg::OFF_MS + (uint32_t)(m % Cfg::MSB) * 2 * Cfg::MS_SLAB;
#pragma unroll
                for (int qp = 0; qp < 8; ++qp) {   // columns i = 16 qp .. 16 qp + 15
                    const int q = 2 * qp;
                    stsm_x4(ms + (uint32_t)(q >> 3) * Cfg::MS_SLAB + swz((uint32_t)jw + st_r, (uint32_t)(q & 7) + st_c),
                            pack_bf16x2(s[q][0], s[q][1]), pack_bf16x2(s[q][2], s[q][3]),
                            pack_bf16x2(s[q + 1][0], s[q + 1][1]), pack_bf16x2(s[q + 1][2], s[q + 1][3]));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_MSREADY0 + (m & 1)));
        };
        // one lane waits; the warp learns the result
        auto warp_wait = [&](int b, uint32_t parity) -> bool {
            bool ok = true;
            if (lane == 0) ok = role_wait(bar(b), parity, a.limit_ns, &s_abort);
            return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        };
        // the start of chunk n: its stage, and (n > 0) the buffers it overwrites
        auto chunk_wait = [&](int n) -> bool {   // lanes 0 and 1 test one barrier each
            bool ok = true;
            if (lane == 0)
                ok = role_wait(bar(B_FULL0 + n % NST), (uint32_t)(n / NST) & 1u, a.limit_ns, &s_abort);
            else if (lane == 1 && n > 0)
                ok = role_wait(bar(B_SAFE0 + (n & 1)), (uint32_t)((n - 1) >> 1) & 1u, a.limit_ns,
                               &s_abort);
            return __all_sync(0xffffffffu, ok);
        };
        if (NC == 0 && fin_view) store_state();   // an empty sequence: final = initial
        if (NC > 0) publish(0);

        bool ready = false;   // chunk n's barriers were found complete during chunk n - 1
        for (int n = 0; n < NC; ++n) {
            const int wb = n & 1;
            const uint32_t st_a = stage(n);
            // ---- K, Q, v, [Lb | P] and the scalars of chunk n are in place, and the
            // Wt and MS buffers this chunk writes are free
            if (!ready && !chunk_wait(n)) break;
            const Scal S = scal(n);

            // ---- X^T = S_J K^T (16 x 64, K = 128): A = bf16(S_J), B = K[s][i] rows
            float x[8][4];
#pragma unroll
            for (int p = 0; p < 8; ++p) x[p][0] = x[p][1] = x[p][2] = x[p][3] = 0.f;
            // operands of the E step, loaded while the X^T products run: the v fragments
            // (matrices (s 16sp+0..7 | 8..15) x (j jw+0..7 | jw+8..15), transposed: vfa[sp][0]
            // s 16sp+2t.., j g;  [1] s 16sp+2t.., j g+8;  [2] s 16sp+8+2t.., j g;  [3] s
            // 16sp+8+2t.., j g+8), gamma and beta at s = 8p + 2t4 (+1)
            uint32_t vfa[4][4];
            float2 gaa[8], bea[8];
            const float gC = s_gC[n % NST];
            {
                // B fragments of one k-step (16 i x 64 s), loaded two k-steps ahead
                auto load_k = [&](uint32_t (&bf)[4][4], int kt) {
                    const uint32_t kb = st_a + Cfg::ST_K + (uint32_t)(kt >> 2) * 16384u;
#pragma unroll
                    for (int sp = 0; sp < 4; ++sp)
                        ldsm_x4(bf[sp], kb + swz((uint32_t)(16 * sp) + bn_r, (uint32_t)((kt & 3) * 2) + bn_c));
                };
                uint32_t bq[3][4][4];
                load_k(bq[0], 0);
                load_k(bq[1], 1);
#pragma unroll
                for (int kt = 0; kt < 8; ++kt) {   // i = 16 kt .. 16 kt + 15
                    if (kt + 2 < 8) load_k(bq[(kt + 2) % 3], kt + 2);
                    if (kt == 1) {
                        // v[s][J] (TMA, 64-column slabs; zero-filled past the end of a dense tensor)
                        const uint32_t vt = st_a + Cfg::ST_V + (uint32_t)(jw >> 6) * 8192u;
                        const uint32_t vc = (uint32_t)((jw >> 3) & 7);
#pragma unroll
                        for (int sp = 0; sp < 4; ++sp)
                            ldsm_x4_t(vfa[sp], vt + swz((uint32_t)(16 * sp) + (uint32_t)(lane & 7) + (uint32_t)((lane >> 4) * 8),
                                                        vc + (uint32_t)((lane >> 3) & 1)));
#pragma unroll
                        for (int p = 0; p < 8; ++p) {
                            gaa[p] = *reinterpret_cast<const float2 *>(&S.gam[8 * p + 2 * t4]);
                            bea[p] = *reinterpret_cast<const float2 *>(&S.bs[8 * p + 2 * t4]);
                        }
                    }
                    uint32_t af[4];
                    af[0] = pack_bf16x2(s[2 * kt][0], s[2 * kt][1]);
                    af[1] = pack_bf16x2(s[2 * kt][2], s[2 * kt][3]);
                    af[2] = pack_bf16x2(s[2 * kt + 1][0], s[2 * kt + 1][1]);
                    af[3] = pack_bf16x2(s[2 * kt + 1][2], s[2 * kt + 1][3]);
#pragma unroll
                    for (int sp = 0; sp < 4; ++sp) {   // s = 16 sp .. 16 sp + 15
                        mma16816(x[2 * sp], af, bq[kt % 3][sp][0], bq[kt % 3][sp][1]);
                        mma16816(x[2 * sp + 1], af, bq[kt % 3][sp][2], bq[kt % 3][sp][3]);
                    }
                }
            }

            // ---- E^T = V^T - X^T diag(gamma) -> bf16 into this warp's rows of the Wt
            // tile of this chunk (buffer n % 2);  X^T <- E^T diag(beta) (fp32: the
            // identity part of T)
            uint8_t *wt = sm + Cfg::OFF_WT + wb * Cfg::WT_BYTES;
            uint32_t ea[4][4];   // E^T A fragments, 16-column steps (E_REGS)
            {
#pragma unroll
                for (int sp = 0; sp < 4; ++sp) {
                    const uint32_t (&vf)[4] = vfa[sp];
                    uint32_t eb[4];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int p = 2 * sp + h;
                        const float2 ga = gaa[p];
                        const float2 be = bea[p];
                        const float2 vlo = bf16x2_to_float2(vf[2 * h]);
                        const float2 vhi = bf16x2_to_float2(vf[2 * h + 1]);
                        const float e0 = fmaf(-ga.x, x[p][0], vlo.x), e1 = fmaf(-ga.y, x[p][1], vlo.y);
                        const float e2 = fmaf(-ga.x, x[p][2], vhi.x), e3 = fmaf(-ga.y, x[p][3], vhi.y);
                        eb[2 * h] = pack_bf16x2(e0, e1);
                        eb[2 * h + 1] = pack_bf16x2(e2, e3);
                        x[p][0] = be.x * e0;
                        x[p][1] = be.y * e1;
                        x[p][2] = be.x * e2;
                        x[p][3] = be.y * e3;
                    }
                    if constexpr (Cfg::E_REGS) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) ea[sp][e] = eb[e];
                    } else {
                        stsm_x4(smem_u32(wt) + swz((uint32_t)jw + st_r, (uint32_t)(2 * sp) + st_c), eb[0],
                                eb[1], eb[2], eb[3]);
                    }
                }
            }
            __syncwarp();

            // ---- W^T = X^T + E^T Lb^T: A = E^T (this warp's rows), B = Lb[r][s] rows.
            // Lb is strictly lower triangular (exact zeros for s >= r), so the 16 x 16
            // blocks with s-block ks above r-block rp add nothing and are skipped: 20 of the
            // 32 products remain.
            float2 sca[8];   // gamma_C / gamma at r = 8p + 2t4 (+1), loaded during the products
            {
                const uint32_t lb_a = st_a + Cfg::ST_LP;
                auto load_l = [&](uint32_t (&af)[4], uint32_t (&bf)[4][4], int ks) {
                    if constexpr (!Cfg::E_REGS)
                        ldsm_x4(af, smem_u32(wt) + swz((uint32_t)jw + bt_r, (uint32_t)(2 * ks) + bt_c));
#pragma unroll
                    for (int rp = 0; rp < 4; ++rp)
                        if (rp >= ks)
                            ldsm_x4(bf[rp], lb_a + swz((uint32_t)(16 * rp) + bn_r, (uint32_t)(2 * ks) + bn_c));
                };
                uint32_t aq[2][4], bq[2][4][4];
                load_l(aq[0], bq[0], 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {   // s = 16 ks .. 16 ks + 15
                    if (ks + 1 < 4) load_l(aq[(ks + 1) & 1], bq[(ks + 1) & 1], ks + 1);
                    if (ks == 1) {
#pragma unroll
                        for (int p = 0; p < 8; ++p) sca[p] = *reinterpret_cast<const float2 *>(&S.sc[8 * p + 2 * t4]);
                    }
                    const uint32_t (&af)[4] = Cfg::E_REGS ? ea[ks] : aq[ks & 1];
#pragma unroll
                    for (int rp = ks; rp < 4; ++rp) {   // r = 16 rp .. 16 rp + 15
                        mma16816(x[2 * rp], af, bq[ks & 1][rp][0], bq[ks & 1][rp][1]);
                        mma16816(x[2 * rp + 1], af, bq[ks & 1][rp][2], bq[ks & 1][rp][3]);
                    }
                }
            }
            __syncwarp();   // every lane has read E^T: Wt may overwrite it

            // ---- W^T -> bf16 into the W tile ([j][r], K-major) that the output product
            // P W reads;  Wt^T = W^T diag(gamma_C / gamma) -> bf16 A fragments of the
            // state update
            uint32_t ef[4][4];
            {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    stsm_x4(smem_u32(wt) + swz((uint32_t)jw + st_r, (uint32_t)(2 * ks) + st_c),
                            pack_bf16x2(x[2 * ks][0], x[2 * ks][1]), pack_bf16x2(x[2 * ks][2], x[2 * ks][3]),
                            pack_bf16x2(x[2 * ks + 1][0], x[2 * ks + 1][1]),
                            pack_bf16x2(x[2 * ks + 1][2], x[2 * ks + 1][3]));
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    const float2 sc = sca[p];
                    ef[p >> 1][2 * (p & 1) + 0] = pack_bf16x2(sc.x * x[p][0], sc.y * x[p][1]);
                    ef[p >> 1][2 * (p & 1) + 1] = pack_bf16x2(sc.x * x[p][2], sc.y * x[p][3]);
                }
            }

            // ---- S_J = gamma_C S_J + Wt^T K: B = K[r][i] rows (transposed)
            {
#pragma unroll
                for (int q = 0; q < 16; ++q)
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[q][e] *= gC;
                // B fragments of a quarter step (16 r x 64 i), loaded two quarters ahead
                auto load_kt = [&](uint32_t (&bf)[4][4], int qq) {
                    const int ks = qq >> 1, slab = qq & 1;
#pragma unroll
                    for (int ip = 0; ip < 4; ++ip)
                        ldsm_x4_t(bf[ip], st_a + Cfg::ST_K + (uint32_t)slab * 16384u +
                                              swz((uint32_t)(16 * ks) + bt_r, (uint32_t)(ip * 2) + bt_c));
                };
                uint32_t bq[3][4][4];
                load_kt(bq[0], 0);
                load_kt(bq[1], 1);
#pragma unroll
                for (int qq = 0; qq < 8; ++qq) {   // r = 16 (qq / 2) .., i = 64 (qq % 2) ..
                    if (qq + 2 < 8) load_kt(bq[(qq + 2) % 3], qq + 2);
                    const int ks = qq >> 1, slab = qq & 1;
#pragma unroll
                    for (int ip = 0; ip < 4; ++ip) {   // i = 64 slab + 16 ip ..
                        mma16816(s[8 * slab + 2 * ip], ef[ks], bq[qq % 3][ip][0], bq[qq % 3][ip][1]);
                        mma16816(s[8 * slab + 2 * ip + 1], ef[ks], bq[qq % 3][ip][2], bq[qq % 3][ip][3]);
                    }
                }
            }
            // while the state update's MMAs run: are chunk n + 1's barriers already
            // complete (then its start needs no wait)?  Lanes 0 and 1 test one each.  Only
            // with four chain warps: with eight (two per SM sub-partition) the tests cost
            // more issue slots than the waits they save (measured: 2.010 -> 2.091 ms on the
            // long workload, against 0.1686 -> 0.1645 ms on the prefill with four).
            if constexpr (DVH == 64) {
                bool t = n + 1 < NC;
                if (t && lane == 0)
                    t = mbar_test_wait(bar(B_FULL0 + (n + 1) % NST), (uint32_t)((n + 1) / NST) & 1u);
                else if (t && lane == 1)
                    t = mbar_test_wait(bar(B_SAFE0 + ((n + 1) & 1)), (uint32_t)(n >> 1) & 1u);
                ready = __all_sync(0xffffffffu, t);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_FREE0 + n % NST));   // this warp is done with stage n
            // a single MS buffer is free once the output's [K;Q] MS_n has completed
            if (Cfg::MSB == 1 && n + 1 < NC && !warp_wait(B_QMS, (uint32_t)n & 1u)) break;
            publish(n + 1);   // MS_{n+1} (if any) and W_n
            if (n + 1 == NC && fin_view) store_state();
        }
    } else if (SO && warp == NCH + 1) {
        // ================================================================ saves only
        // Iteration m: once MS_m and W_{m-1} are published, their tiles leave by tensor
        // stores; once the stores have read them, the chain may overwrite the buffers.
        if (lane == 0) {
            const int64_t x0 = (int64_t)sv.z * ((a.T + C - 1) / C) + sv.tz / C;
            for (int m = 0; m <= NC && NC > 0; ++m) {
                if (!role_wait(bar(B_MSREADY0 + (m & 1)), (uint32_t)(m >> 1) & 1u, a.limit_ns, &s_abort)) break;
                if (m < NC) {
                    const uint32_t ms = sbase + Cfg::OFF_MS + (uint32_t)(m % Cfg::MSB) * 2 * Cfg::MS_SLAB;
                    tma_store_3d(&tm_sm, ms, 0, j0, (int)(x0 + m));
                    tma_store_3d(&tm_sm, ms + Cfg::MS_SLAB, 64, j0, (int)(x0 + m));
                }
                if (m > 0)
                    tma_store_3d(&tm_sw, sbase + Cfg::OFF_WT + (uint32_t)((m - 1) & 1) * Cfg::WT_BYTES, 0, j0,
                                 (int)(x0 + m - 1));
                bulk_commit();
                bulk_wait_read_all();
                if (m < NC) {
                    mbar_arrive(bar(B_QMS));
                    if (m + 1 < NC) mbar_arrive(bar(B_SAFE0 + ((m + 1) & 1)));
                }
            }
            bulk_wait_all();   // the saved tiles are written before the CTA leaves
        }
        __syncwarp();
    } else if (warp == NCH + 1) {
        // ================================================================ output products
        if (lane == 0) {
            const uint32_t idesc_o = idesc_bf16(128, DVH, false, false);   // K-major A and B
            bool issued = false;
            // saving: chunk n's tiles go to row x(n) of the saved tensors (value columns J)
            const int64_t x0 = (int64_t)sv.z * ((a.T + C - 1) / C) + sv.tz / C;
            auto save_ms = [&](int n) {   // M_n^T: 2 slabs of 64 key columns, DVH value rows
                const uint32_t ms = sbase + Cfg::OFF_MS + (uint32_t)(n % Cfg::MSB) * 2 * Cfg::MS_SLAB;
                tma_store_3d(&tm_sm, ms, 0, j0, (int)(x0 + n));
                tma_store_3d(&tm_sm, ms + Cfg::MS_SLAB, 64, j0, (int)(x0 + n));
            };
            auto save_w = [&](int n) {    // W_n^T: DVH value rows of 64 tokens
                tma_store_3d(&tm_sw, sbase + Cfg::OFF_WT + (uint32_t)(n & 1) * Cfg::WT_BYTES, 0, j0, (int)(x0 + n));
            };
            // Iteration m: [Lb;P] W_{m-1} fills chunk m-1's second accumulator (rows
            // 64-127: P W), then [K;Q] MS_m chunk m's first (rows 64-127: Q M_m)
            for (int m = 0; m <= NC && NC > 0; ++m) {
                if (!role_wait(bar(B_MSREADY0 + (m & 1)), (uint32_t)(m >> 1) & 1u, a.limit_ns, &s_abort)) break;
                if (m > 0) {
                    const int n = m - 1;
                    tc_fence_after();
                    const uint64_t dl = sdesc_sw128(stage(n) + Cfg::ST_LP, 16, 1024);
                    const uint64_t dw = sdesc_sw128(sbase + Cfg::OFF_WT + (uint32_t)(n & 1) * Cfg::WT_BYTES, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + Cfg::TM_PW + (uint32_t)(n & 1) * DVH, sdesc_add(dl, kk * 32),
                                 sdesc_add(dw, kk * 32), idesc_o, kk > 0);
                    mma_commit(bar(B_OFULL0 + (n & 1)));
                }
                if (m == NC) {
                    if (a.save) {
                        save_w(m - 1);
                        bulk_commit();
                    }
                    break;
                }
                // O(m) = [K;Q] MS_m, once the accumulator buffer has been read out (chunk m-2)
                bool ok = role_wait(bar(B_FULL0 + m % NST), (uint32_t)(m / NST) & 1u, a.limit_ns, &s_abort);
                if (ok && m > 1)
                    ok = role_wait(bar(B_OFREE0 + (m & 1)), (uint32_t)((m - 2) >> 1) & 1u, a.limit_ns, &s_abort);
                if (!ok) break;
                tc_fence_after();
                {
                    const uint64_t da = sdesc_sw128(stage(m) + Cfg::ST_K, 16, 1024);
                    const uint64_t db = sdesc_sw128(sbase + Cfg::OFF_MS + (uint32_t)(m % Cfg::MSB) * 2 * Cfg::MS_SLAB,
                                                    16, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16(tmem + (uint32_t)(m & 1) * DVH, sdesc_add(da, (kk >> 2) * 16384 + (kk & 3) * 32),
                                 sdesc_add(db, (kk >> 2) * Cfg::MS_SLAB + (kk & 3) * 32), idesc_o, kk > 0);
                }
                if (a.save) {
                    // the tiles the two products just read, before their buffers are released:
                    // the stores must have read them before the commits below
                    save_ms(m);
                    if (m > 0) save_w(m - 1);
                    bulk_commit();
                    bulk_wait_read_all();
                }
                mma_commit(bar(B_QMS));
                // chunk m+1 may overwrite W[(m+1) % 2] (read by W_{m-1}'s product) and
                // MS[m % 2] once both products issued so far are done
                if (m + 1 < NC) mma_commit(bar(B_SAFE0 + ((m + 1) & 1)));
                issued = true;
            }
            if (s_abort && issued) {   // let this thread's MMAs land before TMEM goes away
                mma_commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0u, kCleanupLimitNs);
            }
            if (a.save) bulk_wait_all();   // the saved tiles are written before the CTA leaves
        }
        __syncwarp();
    } else if (SO && warp >= NCH + 2) {
        // no outputs
    } else if (warp >= NCH + 2) {
        // ================================================================ output rows
        // thread r: accumulator row 64 + r (TMEM lane 64 + r) = output row r of a chunk
        const int r = tid - 32 * (NCH + 2);
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const bool packed = a.cu_seqlens != nullptr;
        for (int m = 0; m < NC; ++m) {
            bool ok = (r != 0) ||
                      role_wait(bar(B_OFULL0 + (m & 1)), (uint32_t)(m >> 1) & 1u, a.limit_ns, &s_abort);
            if (!named_and(BAR_OUT, 64, ok)) break;
            tc_fence_after();
            const int c = min(C, T - m * C);
            // A whole chunk, or the clipped tail of a dense sequence: staged in the Q slabs
            // of its stage (the products that read Q_m are complete) and written by tensor
            // stores; the tail of a packed sequence by plain stores.
            const bool tiled = !packed || c == C;
            const uint32_t stg = stage(m) + Cfg::ST_Q;
            if (tiled) {
                fence_proxy_async_smem();
                stage_rows<DVH>(tl + (uint32_t)(m & 1) * DVH, tl + Cfg::TM_PW + (uint32_t)(m & 1) * DVH, r,
                                scal(m).gam, stg, 16384u);
                fence_proxy_async_smem();
            } else {
                emit_rows<DVH>(tl + (uint32_t)(m & 1) * DVH, tl + Cfg::TM_PW + (uint32_t)(m & 1) * DVH, r, c,
                               scal(m).gam, out0 + (int64_t)m * C * orow, orow);
            }
            tc_fence_before();
            named_sync(BAR_OUT, 64);
            if (r == 0) {
                mbar_arrive(bar(B_OFREE0 + (m & 1)));   // the accumulator buffer is read out
                if (tiled) {
#pragma unroll
                    for (int vs = 0; vs < DVH / 64; ++vs)
                        tma_store_3d(&tm_o, stg + (uint32_t)vs * 16384u, j0 + 64 * vs, sv.tz + m * C, sv.z);
                    bulk_commit();
                    bulk_wait_read_all();   // the stage may be refilled once the store has read it
                }
                mbar_arrive(bar(B_FREE0 + m % NST));    // the products of chunk m are done
            }
        }
        if (r == 0) bulk_wait_all();
    } else {
        // ================================================================ copy (warp NCH)
        // Stage n % NST of chunk n: K and Q (two slabs each) and v[., J] by TMA, the
        // [Lb | P] tile by a bulk copy, and the chunk's decay scalars; two arrivals
        // (the expect_tx and the decay) and the bytes complete it.
        uint32_t issued[3] = {0, 0, 0};
        // without outputs the chain reads K, v and Lb only
        constexpr uint32_t STAGE_TX = SO ? 16384 + DVH * 128 + TILE_BYTES / 2 : 32768 + DVH * 128 + TILE_BYTES;
        auto issue = [&](int n) {     // lane 0 only
            const int st = n % NST;
            const uint32_t b = bar(B_FULL0 + st);
            const uint32_t kq = stage(n);
            const int row = sv.tz + n * C;
            mbar_arrive_expect_tx(b, STAGE_TX);
            tma_load_3d(kq + Cfg::ST_K, &tm_k, b, 0, row, sv.z);
            if (!SO) tma_load_3d(kq + Cfg::ST_Q, &tm_q, b, 0, row, sv.z);
            tma_load_3d(kq + Cfg::ST_K + 16384, &tm_k, b, 64, row, sv.z);
            if (!SO) tma_load_3d(kq + Cfg::ST_Q + 16384, &tm_q, b, 64, row, sv.z);
#pragma unroll
            for (int vs = 0; vs < DVH / 64; ++vs)
                tma_load_3d(kq + Cfg::ST_V + vs * 8192, &tm_v, b, j0 + 64 * vs, row, sv.z);
            bulk_load(kq + Cfg::ST_LP, tiles + (int64_t)n * TILE_BYTES, SO ? TILE_BYTES / 2 : TILE_BYTES, b);
            ++issued[st];
        };
        // Pull the inputs of chunk n into L2 ahead of their shared-memory loads.
        auto prefetch_l2 = [&](int n) {   // lane 0 only
            if (n >= NC) return;
            const int row = sv.tz + n * C;
            tma_prefetch_3d(&tm_k, 0, row, sv.z);
            tma_prefetch_3d(&tm_k, 64, row, sv.z);
            if (!SO) {
                tma_prefetch_3d(&tm_q, 0, row, sv.z);
                tma_prefetch_3d(&tm_q, 64, row, sv.z);
            }
#pragma unroll
            for (int vs = 0; vs < DVH / 64; ++vs) tma_prefetch_3d(&tm_v, j0 + 64 * vs, row, sv.z);
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
            const int st = n % NST;
            warp_decay(lane, gv, bv, min(C, T - n * C), a.a_min, scal(n), &s_gC[st]);
            if (lane == 0) mbar_arrive(bar(B_FULL0 + st));
        };
        constexpr int kAhead = 3;   // chunks prefetched into L2 beyond the staged ones
        float gv[2], bv[2];
        if (lane == 0)
            for (int n = 0; n < NST + kAhead; ++n) prefetch_l2(n);
        grid_dependency_wait();   // the preparation kernel's tiles are complete and visible
        for (int n = 0; n < NST && n < NC; ++n) {
            load_gb(n, gv, bv);
            if (lane == 0) issue(n);
            decay(n, gv, bv);
        }
        if (NC > NST) load_gb(NST, gv, bv);
        for (int n = 0; n + NST < NC; ++n) {   // refill a stage once chunk n is done with it
            const int st = n % NST;
            bool ok = (lane != 0) ||
                      role_wait(bar(B_FREE0 + st), (uint32_t)(n / NST) & 1u, a.limit_ns, &s_abort);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) {
                issue(n + NST);
                prefetch_l2(n + NST + kAhead);
            }
            decay(n + NST, gv, bv);
            if (n + NST + 1 < NC) load_gb(n + NST + 1, gv, bv);
        }
        if (s_abort && lane == 0) {
            // at most the latest load of each stage can still be in flight (its decay
            // arrival was made with it): wait for its bytes
            for (int st = 0; st < NST; ++st)
                if (issued[st] > 0)
                    mbar_wait(bar(B_FULL0 + st), (issued[st] - 1) & 1u, kCleanupLimitNs);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (!SO && warp == NCH) {
        __syncwarp();
        tmem_dealloc(tmem, Cfg::TM_COLS);
    }
}

template <int DVH, bool SO>
cudaError_t launch_chain_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                           const CUtensorMap &mo, const CUtensorMap &msm, const CUtensorMap &msw,
                           const FusedArgs &a, const void *ws, int64_t nslot, int BH, cudaStream_t s) {
    using Cfg = ChainCfg<DVH>;
    cudaError_t e = cudaFuncSetAttribute(chain_kernel<DVH, SO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Cfg::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    // launched as a programmatic dependent of the preparation kernel before it: the CTAs
    // set up (barriers, tensor memory, the initial state, L2 prefetch) while its last
    // CTAs finish, and the copy warp waits for its tiles before the first read
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(BH * (128 / DVH)));
    cfg.blockDim = dim3(Cfg::NT);
    cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chain_kernel<DVH, SO>, mq, mk, mv, mo, msm, msw, a,
                              static_cast<const uint8_t *>(ws), nslot);
}

}  // namespace

// Value columns per CTA: two CTAs per head while every CTA has an SM of its
// own, one CTA per head beyond that.  The GDR_OPT_CHAIN_SPLIT option forces
// one (the tests cover both on small shapes).
int chain_split(int BH) {
    const int forced = opt_chain_split();
    if (forced == 1 || forced == 2) return forced;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return 2 * BH <= sms ? 2 : 1;
}

// A bf16 [rows][n][inner] tensor viewed as 3-D for 64 x box_rows tensor stores with the
// 128-byte swizzle (the smem tile's layout), so that the global copy is row-major.
bool make_map_saved(CUtensorMap *m, void *ptr, int inner, int n, int64_t rows, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)n, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * n * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_chain(const void *q, const void *k, const void *v, const float *g, const float *beta,
                         float a_min, const float *init, void *out, float *final_state, const void *ws,
                         int BH, int T, const int *cu_seqlens, int H, int total_T, cudaStream_t s,
                         int nseg, const float *seg_init, void *saved, bool states_only) {
    if (BH == 0 || (cu_seqlens ? total_T : T) == 0) return cudaSuccess;   // callers copy the state
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(ws)) & 15)
        return cudaErrorMisalignedAddress;
    CUtensorMap mq, mk, mv, mo;
    const bool ok = cu_seqlens ? (make_map_packed(&mq, q, H, total_T) && make_map_packed(&mk, k, H, total_T) &&
                                  make_map_packed(&mv, v, H, total_T) && make_map_packed(&mo, out, H, total_T))
                               : (make_map(&mq, q, BH, T) && make_map(&mk, k, BH, T) && make_map(&mv, v, BH, T) &&
                                  make_map(&mo, out, BH, T));
    if (!ok) return cudaErrorInvalidValue;
    FusedArgs a{g, beta, init, static_cast<__nv_bfloat16 *>(out), final_state, a_min, T, wait_limit_ns(),
                static_cast<const __nv_bfloat16 *>(v)};
    a.cu_seqlens = cu_seqlens;
    a.H = H;
    a.total_T = total_T;
    const int64_t nslot = tile_slots(a, BH);
    if (!cu_seqlens && nseg > 1) {   // one view per (head, segment)
        a.nseg = nseg;
        a.seg_chunks = segment_chunks(T, nseg);
        a.seg_init = seg_init;
    }
    const int views = BH * a.nseg;
    const int split = chain_split(views);
    CUtensorMap msm = mo, msw = mo;   // placeholders when nothing is saved
    if (saved) {
        if (cu_seqlens || (reinterpret_cast<uintptr_t>(saved) & 15)) return cudaErrorInvalidValue;
        const int64_t xs = (int64_t)BH * ((T + C - 1) / C);   // (head, chunk) tiles
        uint8_t *sb = static_cast<uint8_t *>(saved);
        if (!make_map_saved(&msm, sb, D, D, xs, 128 / split) ||
            !make_map_saved(&msw, sb + saved_state_bytes(BH, T), C, D, xs, 128 / split))
            return cudaErrorInvalidValue;
        a.save = 1;
    }
    if (states_only && saved)   // the states and W tiles only, no outputs
        return split == 2 ? launch_chain_t<64, true>(mq, mk, mv, mo, msm, msw, a, ws, nslot, views, s)
                          : launch_chain_t<128, true>(mq, mk, mv, mo, msm, msw, a, ws, nslot, views, s);
    return split == 2 ? launch_chain_t<64, false>(mq, mk, mv, mo, msm, msw, a, ws, nslot, views, s)
                      : launch_chain_t<128, false>(mq, mk, mv, mo, msm, msw, a, ws, nslot, views, s);
}

cudaError_t take_chain_error_word(unsigned *value) { return take_error_word(value); }

}  // namespace gdr
