// gdr_segment.cu -- exact sequence parallelism for the two-kernel prefill path:
// the chunks of every (sequence, head) are split into S segments whose chains
// run at the same time.
//
// The chunk step of the state is affine in the state ("What a Trillion-
// Parameter MoE Model Reveals About the Next Stage of LLM Scaling", sections
// 3.1-3.3: between tiles the computation proceeds through the recurrent state):
//   M_{n+1} = gamma_C M_n + K^T diag(gamma_C / gamma) T diag(beta) (V - diag(gamma) K M_n)
//           = F_n M_n + G_n,
// with F_n = gamma_C I - K^T diag(gamma_C/gamma) T diag(beta gamma) K (dk x dk) and
// G_n the step from a zero state.  So a segment s of consecutive chunks maps its
// initial state M_s to its final state by M_{s+1} = Phi_s M_s + Delta_s, where
// Phi_s = F_last ... F_first and Delta_s is the segment's chain run from a zero
// state.  Both come from the same chain arithmetic as the state itself:
//   Delta_s: the chain over the segment from M = 0 with the segment's v;
//   Phi_s:   the chain from M = I (dk "value" columns) with v = 0, since then
//            E = -diag(gamma) K Phi and every step applies F_n to the columns.
// The prefill then runs in three steps after the chunk preparation:
//   1. seg_pass1_kernel: Delta_s for s = 0 .. S-2 (segment 0 from the initial
//      state, so that Delta_0 = M_1) and Phi_s for s = 1 .. S-2, every segment
//      at once;
//   2. seg_scan_kernel: M_0 = init, M_1 = Delta_0, M_{s+1} = Phi_s M_s + Delta_s
//      (S - 2 fp32 products of dk x dk by dk x dv per head);
//   3. the chain kernel over all S segments at once, each from its M_s, writing
//      the outputs (and the last segment the final state).
// Nothing is approximated: the segment maps compose exactly, and each is
// computed with the chain's own operand roundings.
//
// seg_pass1_kernel: one CTA = 128 columns of one segment's chain (the Delta
// columns = the value columns of the head, or the Phi columns = the key
// columns), 8 chain warps of 16 columns each and one copy warp.  A chain warp
// runs the same warp-level MMA steps as the chain kernel (S_J = M_J^T in
// registers, X^T = S_J K^T, E^T, W^T = X^T + E^T Lb^T, S_J = gamma_C S_J + Wt^T
// K), without outputs.

#include "gdr_fused_common.cuh"

#include <algorithm>

namespace gdr {
namespace {

namespace sp {
constexpr int NCH = 8;                    // chain warps: 128 columns
constexpr int NT = 32 * (NCH + 1);        // + the copy warp
constexpr int NST = 3;                    // input stages
constexpr uint32_t ST_K = 0;              // K: two 64-column slabs of 8 KB
constexpr uint32_t ST_V = 16384;          // v: two 64-column slabs of 8 KB (Delta CTAs)
constexpr uint32_t ST_LB = 32768;         // Lb: the first 8 KB of the chunk's tile
constexpr uint32_t ST_BYTES = 40960;
constexpr uint32_t OFF_SC = NST * ST_BYTES;   // a 5 x 64 fp32 slot per stage
constexpr uint32_t SMEM_USED = OFF_SC + NST * 5 * 64 * 4;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(ST_BYTES % 1024 == 0 && ST_V % 1024 == 0 && ST_LB % 1024 == 0,
              "swizzled tiles must be 1024-byte aligned");
static_assert(SMEM_ALLOC <= 232448, "exceeds 227 KB of shared memory per CTA");
enum : int { B_FULL0 = 0, B_FREE0 = 3, NUM_BARS = 6 };
}  // namespace sp

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t c8) {
    return row * 128u + ((c8 ^ (row & 7u)) << 4);
}
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}

struct SegArgs {
    const float *g, *beta, *init;   // init: [BH][D][D] or nullptr (zeros)
    float *delta, *phi;             // [BH][S - 1][D][D] each
    float a_min;
    int T, S, L;                    // tokens per head, segments, chunks per segment
    uint64_t limit_ns;
};

// CTA c of a head: c = 0 the Delta columns of segment 0; c = 1 + 2 (s - 1) + r for
// s = 1 .. S-2 with r = 0 the Delta columns, r = 1 the Phi columns.
__global__ void __launch_bounds__(sp::NT, 1)
seg_pass1_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const SegArgs a, const uint8_t *tiles_all, int64_t nslot) {
    using namespace sp;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    __shared__ __align__(8) uint64_t s_bar[NUM_BARS];
    __shared__ float s_gC[NST];
    __shared__ volatile int s_abort;

    const int per_head = 2 * a.S - 3;
    const int bh = blockIdx.x / per_head, c = blockIdx.x % per_head;
    const int s = c == 0 ? 0 : 1 + (c - 1) / 2;
    const bool is_phi = c > 0 && ((c - 1) & 1) == 1;
    const int NC = a.L;                           // segments 0 .. S-2 are whole
    const int t0 = s * a.L * C;                   // first token of the segment
    const int Tv = a.T - t0 < a.L * C ? a.T - t0 : a.L * C;
    const uint8_t *tiles = tiles_all + ((int64_t)bh * nslot + (int64_t)s * a.L) * TILE_BYTES;
    float *dst = (is_phi ? a.phi : a.delta) + ((int64_t)bh * (a.S - 1) + s) * D * D;
    auto bar = [&](int i) { return smem_u32(&s_bar[i]); };
    auto stage = [&](int n) { return sbase + (uint32_t)(n % NST) * ST_BYTES; };
    auto scal = [&](int n) { return scal_at(reinterpret_cast<float *>(sm + OFF_SC) + (n % NST) * 5 * 64); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(bar(B_FULL0 + i), 2);     // expect_tx arrival + the decay
            mbar_init(bar(B_FREE0 + i), NCH);
        }
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == NCH && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    __syncthreads();

    if (warp < NCH) {
        // ================================================================ chain
        const int g = lane >> 2, t4 = lane & 3;
        const int jw = 16 * warp;
        const uint32_t bn_r = (uint32_t)((lane & 7) + (lane >> 4) * 8);
        const uint32_t bn_c = (uint32_t)((lane >> 3) & 1);
        const uint32_t bt_r = (uint32_t)((lane & 7) + ((lane >> 3) & 1) * 8);
        const uint32_t bt_c = (uint32_t)(lane >> 4);
        float st[16][4];   // S_J: rows jw + g (+ 8), columns i = 8 q + 2 t4 (+ 1)
        {
            const float *src = (!is_phi && s == 0 && a.init) ? a.init + (int64_t)bh * D * D + jw : nullptr;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int i = 8 * q + 2 * t4;
                if (is_phi) {   // M = I: column j of Phi starts as e_j
                    st[q][0] = (i == jw + g) ? 1.f : 0.f;
                    st[q][1] = (i + 1 == jw + g) ? 1.f : 0.f;
                    st[q][2] = (i == jw + g + 8) ? 1.f : 0.f;
                    st[q][3] = (i + 1 == jw + g + 8) ? 1.f : 0.f;
                } else {
                    st[q][0] = src ? src[(int64_t)i * D + g] : 0.f;
                    st[q][1] = src ? src[(int64_t)(i + 1) * D + g] : 0.f;
                    st[q][2] = src ? src[(int64_t)i * D + g + 8] : 0.f;
                    st[q][3] = src ? src[(int64_t)(i + 1) * D + g + 8] : 0.f;
                }
            }
        }
        bool ok = true;
        for (int n = 0; n < NC; ++n) {
            const uint32_t st_a = stage(n);
            {
                bool w_ok = true;
                if (lane == 0)
                    w_ok = role_wait(bar(B_FULL0 + n % NST), (uint32_t)(n / NST) & 1u, a.limit_ns, &s_abort);
                if (__shfl_sync(0xffffffffu, w_ok ? 1 : 0, 0) == 0) {
                    ok = false;
                    break;
                }
            }
            const Scal S = scal(n);
            const float gC = s_gC[n % NST];

            // ---- X^T = S_J K^T (16 x 64, K = 128)
            float x[8][4];
#pragma unroll
            for (int p = 0; p < 8; ++p) x[p][0] = x[p][1] = x[p][2] = x[p][3] = 0.f;
            uint32_t vfa[4][4];
            float2 gaa[8], bea[8];
            {
                auto load_k = [&](uint32_t (&bf)[4][4], int kt) {
                    const uint32_t kb = st_a + ST_K + (uint32_t)(kt >> 2) * 8192u;
#pragma unroll
                    for (int sp4 = 0; sp4 < 4; ++sp4)
                        ldsm_x4(bf[sp4], kb + swz((uint32_t)(16 * sp4) + bn_r, (uint32_t)((kt & 3) * 2) + bn_c));
                };
                uint32_t bq[3][4][4];
                load_k(bq[0], 0);
                load_k(bq[1], 1);
#pragma unroll
                for (int kt = 0; kt < 8; ++kt) {
                    if (kt + 2 < 8) load_k(bq[(kt + 2) % 3], kt + 2);
                    if (kt == 1) {
                        if (!is_phi) {
                            const uint32_t vt = st_a + ST_V + (uint32_t)(jw >> 6) * 8192u;
                            const uint32_t vc = (uint32_t)((jw >> 3) & 7);
#pragma unroll
                            for (int sp4 = 0; sp4 < 4; ++sp4)
                                ldsm_x4_t(vfa[sp4], vt + swz((uint32_t)(16 * sp4) + (uint32_t)(lane & 7) +
                                                                 (uint32_t)((lane >> 4) * 8),
                                                             vc + (uint32_t)((lane >> 3) & 1)));
                        } else {
#pragma unroll
                            for (int sp4 = 0; sp4 < 4; ++sp4)
                                vfa[sp4][0] = vfa[sp4][1] = vfa[sp4][2] = vfa[sp4][3] = 0u;
                        }
#pragma unroll
                        for (int p = 0; p < 8; ++p) {
                            gaa[p] = *reinterpret_cast<const float2 *>(&S.gam[8 * p + 2 * t4]);
                            bea[p] = *reinterpret_cast<const float2 *>(&S.bs[8 * p + 2 * t4]);
                        }
                    }
                    uint32_t af[4];
                    af[0] = pack_bf16x2(st[2 * kt][0], st[2 * kt][1]);
                    af[1] = pack_bf16x2(st[2 * kt][2], st[2 * kt][3]);
                    af[2] = pack_bf16x2(st[2 * kt + 1][0], st[2 * kt + 1][1]);
                    af[3] = pack_bf16x2(st[2 * kt + 1][2], st[2 * kt + 1][3]);
#pragma unroll
                    for (int sp4 = 0; sp4 < 4; ++sp4) {
                        mma16816(x[2 * sp4], af, bq[kt % 3][sp4][0], bq[kt % 3][sp4][1]);
                        mma16816(x[2 * sp4 + 1], af, bq[kt % 3][sp4][2], bq[kt % 3][sp4][3]);
                    }
                }
            }

            // ---- E^T = V^T - X^T diag(gamma) (bf16 A fragments); X^T <- E^T diag(beta)
            uint32_t ea[4][4];
#pragma unroll
            for (int sp4 = 0; sp4 < 4; ++sp4) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int p = 2 * sp4 + h;
                    const float2 ga = gaa[p], be = bea[p];
                    const float2 vlo = bf16x2_to_float2(vfa[sp4][2 * h]);
                    const float2 vhi = bf16x2_to_float2(vfa[sp4][2 * h + 1]);
                    const float e0 = fmaf(-ga.x, x[p][0], vlo.x), e1 = fmaf(-ga.y, x[p][1], vlo.y);
                    const float e2 = fmaf(-ga.x, x[p][2], vhi.x), e3 = fmaf(-ga.y, x[p][3], vhi.y);
                    ea[sp4][2 * h] = pack_bf16x2(e0, e1);
                    ea[sp4][2 * h + 1] = pack_bf16x2(e2, e3);
                    x[p][0] = be.x * e0;
                    x[p][1] = be.y * e1;
                    x[p][2] = be.x * e2;
                    x[p][3] = be.y * e3;
                }
            }

            // ---- W^T = X^T + E^T Lb^T: B = Lb[r][s] rows (strictly lower triangular: the
            // blocks with ks > rp are zero and skipped)
            float2 sca[8];
            {
                const uint32_t lb_a = st_a + ST_LB;
                auto load_l = [&](uint32_t (&bf)[4][4], int ks) {
#pragma unroll
                    for (int rp = 0; rp < 4; ++rp)
                        if (rp >= ks)
                            ldsm_x4(bf[rp], lb_a + swz((uint32_t)(16 * rp) + bn_r, (uint32_t)(2 * ks) + bn_c));
                };
                uint32_t bq[2][4][4];
                load_l(bq[0], 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    if (ks + 1 < 4) load_l(bq[(ks + 1) & 1], ks + 1);
                    if (ks == 1) {
#pragma unroll
                        for (int p = 0; p < 8; ++p) sca[p] = *reinterpret_cast<const float2 *>(&S.sc[8 * p + 2 * t4]);
                    }
#pragma unroll
                    for (int rp = ks; rp < 4; ++rp) {
                        mma16816(x[2 * rp], ea[ks], bq[ks & 1][rp][0], bq[ks & 1][rp][1]);
                        mma16816(x[2 * rp + 1], ea[ks], bq[ks & 1][rp][2], bq[ks & 1][rp][3]);
                    }
                }
            }

            // ---- Wt^T = W^T diag(gamma_C / gamma) -> bf16 A fragments
            uint32_t ef[4][4];
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const float2 sc = sca[p];
                ef[p >> 1][2 * (p & 1) + 0] = pack_bf16x2(sc.x * x[p][0], sc.y * x[p][1]);
                ef[p >> 1][2 * (p & 1) + 1] = pack_bf16x2(sc.x * x[p][2], sc.y * x[p][3]);
            }

            // ---- S_J = gamma_C S_J + Wt^T K: B = K[r][i] rows (transposed)
            {
#pragma unroll
                for (int q = 0; q < 16; ++q)
#pragma unroll
                    for (int e = 0; e < 4; ++e) st[q][e] *= gC;
                auto load_kt = [&](uint32_t (&bf)[4][4], int qq) {
                    const int ks = qq >> 1, slab = qq & 1;
#pragma unroll
                    for (int ip = 0; ip < 4; ++ip)
                        ldsm_x4_t(bf[ip], st_a + ST_K + (uint32_t)slab * 8192u +
                                              swz((uint32_t)(16 * ks) + bt_r, (uint32_t)(ip * 2) + bt_c));
                };
                uint32_t bq[3][4][4];
                load_kt(bq[0], 0);
                load_kt(bq[1], 1);
#pragma unroll
                for (int qq = 0; qq < 8; ++qq) {
                    if (qq + 2 < 8) load_kt(bq[(qq + 2) % 3], qq + 2);
                    const int ks = qq >> 1, slab = qq & 1;
#pragma unroll
                    for (int ip = 0; ip < 4; ++ip) {
                        mma16816(st[8 * slab + 2 * ip], ef[ks], bq[qq % 3][ip][0], bq[qq % 3][ip][1]);
                        mma16816(st[8 * slab + 2 * ip + 1], ef[ks], bq[qq % 3][ip][2], bq[qq % 3][ip][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_FREE0 + n % NST));   // this warp is done with stage n
        }
        if (ok) {   // S_J^T into the segment's [dk][128] fp32 map
            float *d0 = dst + jw;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int i = 8 * q + 2 * t4;
                d0[(int64_t)i * D + g] = st[q][0];
                d0[(int64_t)(i + 1) * D + g] = st[q][1];
                d0[(int64_t)i * D + g + 8] = st[q][2];
                d0[(int64_t)(i + 1) * D + g + 8] = st[q][3];
            }
        }
    } else {
        // ================================================================ copy (warp NCH)
        uint32_t issued[NST] = {0, 0, 0};
        const uint32_t tx = 16384u + (is_phi ? 0u : 16384u) + 8192u;
        auto issue = [&](int n) {   // lane 0 only
            const int stn = n % NST;
            const uint32_t b = bar(B_FULL0 + stn);
            const uint32_t kq = stage(n);
            const int row = t0 + n * C;
            mbar_arrive_expect_tx(b, tx);
            tma_load_3d(kq + ST_K, &tm_k, b, 0, row, bh);
            tma_load_3d(kq + ST_K + 8192, &tm_k, b, 64, row, bh);
            if (!is_phi) {
                tma_load_3d(kq + ST_V, &tm_v, b, 0, row, bh);
                tma_load_3d(kq + ST_V + 8192, &tm_v, b, 64, row, bh);
            }
            bulk_load(kq + ST_LB, tiles + (int64_t)n * TILE_BYTES, 8192u, b);
            ++issued[stn];
        };
        const int64_t gb = (int64_t)bh * a.T + t0;
        auto load_gb = [&](int n, float (&gv)[2], float (&bv)[2]) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = n * C + 2 * lane + e;
                gv[e] = (t < Tv) ? a.g[gb + t] : 0.f;
                bv[e] = (t < Tv) ? a.beta[gb + t] : 0.f;
            }
        };
        auto decay = [&](int n, const float (&gv)[2], const float (&bv)[2]) {
            const int stn = n % NST;
            warp_decay(lane, gv, bv, min(C, Tv - n * C), a.a_min, scal(n), &s_gC[stn]);
            if (lane == 0) mbar_arrive(bar(B_FULL0 + stn));
        };
        float gv[2], bv[2];
        grid_dependency_wait();   // the preparation kernel's tiles are complete and visible
        for (int n = 0; n < NST && n < NC; ++n) {
            load_gb(n, gv, bv);
            if (lane == 0) issue(n);
            decay(n, gv, bv);
        }
        if (NC > NST) load_gb(NST, gv, bv);
        for (int n = 0; n + NST < NC; ++n) {
            const int stn = n % NST;
            bool ok = (lane != 0) ||
                      role_wait(bar(B_FREE0 + stn), (uint32_t)(n / NST) & 1u, a.limit_ns, &s_abort);
            if (!__all_sync(0xffffffffu, ok)) break;
            if (lane == 0) issue(n + NST);
            decay(n + NST, gv, bv);
            if (n + NST + 1 < NC) load_gb(n + NST + 1, gv, bv);
        }
        if (s_abort && lane == 0) {
            for (int i = 0; i < NST; ++i)
                if (issued[i] > 0) mbar_wait(bar(B_FULL0 + i), (issued[i] - 1) & 1u, kCleanupLimitNs);
        }
    }
    __syncthreads();
}

// M_0 = init (or zeros), M_1 = Delta_0, M_{s+1} = Phi_s M_s + Delta_s for
// s = 1 .. S-2, all fp32.  One CTA per (16 value columns J, head): M_s[:, J] stays
// in shared memory, Phi_s is staged whole (64 KB) for each step.
constexpr int kScanCols = 16;
__global__ void __launch_bounds__(256)
seg_scan_kernel(const float *__restrict__ init, const float *__restrict__ delta,
                const float *__restrict__ phi, float *__restrict__ mseg, int S) {
    extern __shared__ float sm_scan[];
    float *Ph = sm_scan;              // [D][D]
    float *Ms = Ph + D * D;           // [D][kScanCols]
    const int j0 = blockIdx.x * kScanCols;
    const int64_t bh = blockIdx.y;
    const int tid = threadIdx.x;
    const int i = tid >> 1, jh = (tid & 1) * 8;   // output row i, columns jh .. jh + 7 of J
    auto at = [&](const float *base, int64_t m) { return base + m * D * D; };
    float *out0 = mseg + bh * S * D * D;
    // M_0
    for (int x = tid; x < D * kScanCols; x += 256) {
        const int r = x / kScanCols, j = x % kScanCols;
        out0[(int64_t)r * D + j0 + j] = init ? init[(bh * D + r) * D + j0 + j] : 0.f;
    }
    if (S < 2) return;
    // M_1 = Delta_0
    const float *d0 = at(delta, bh * (S - 1));
    for (int x = tid; x < D * kScanCols; x += 256) {
        const int r = x / kScanCols, j = x % kScanCols;
        const float m = d0[(int64_t)r * D + j0 + j];
        Ms[x] = m;
        out0[(int64_t)1 * D * D + (int64_t)r * D + j0 + j] = m;
    }
    for (int s = 1; s + 1 < S; ++s) {
        const float4 *p4 = reinterpret_cast<const float4 *>(at(phi, bh * (S - 1) + s));
        __syncthreads();   // Ms holds M_s; the previous step is done with Ph
        for (int x = tid; x < D * D / 4; x += 256) reinterpret_cast<float4 *>(Ph)[x] = p4[x];
        __syncthreads();
        const float *ds = at(delta, bh * (S - 1) + s) + (int64_t)i * D + j0 + jh;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = ds[e];
        for (int m = 0; m < D; ++m) {
            const float ph = Ph[i * D + m];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(ph, Ms[m * kScanCols + jh + e], acc[e]);
        }
        __syncthreads();   // every thread has read M_s
        float *o = out0 + (int64_t)(s + 1) * D * D + (int64_t)i * D + j0 + jh;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            Ms[i * kScanCols + jh + e] = acc[e];
            o[e] = acc[e];
        }
    }
}

}  // namespace

int segment_count(int BH, int T) {
    const int NC = (T + C - 1) / C;
    if (BH <= 0 || NC <= 0) return 1;
    int S = opt_segments();
    if (S <= 0) {
        // Automatic: the count (3 or more, every segment keeping at least 8 chunks) that
        // minimises a wave-quantised cost of the two sequential kernels, each running
        // ceil(CTAs / SMs) waves of L = ceil(NC / S) dependent chunks plus a fixed ramp of
        // ~9 chunk times per wave: pass 1 with 2 S - 3 CTAs per head at ~0.65 of a
        // one-CTA-per-view chain chunk's time, the chain with S views per head at 1 (one
        // CTA per view) or 0.6 (two); no segments unless that saves 10 % against one
        // chain per head.  The weights are fitted to measured counts: long prefill B1 H32
        // T65536 takes 2.05, 2.12, 2.09, 1.95, 2.17, 2.10, 2.19 ms with 3, 4, 6, 8, 10, 12,
        // 16 segments (this picks 8); million-token B1 H16 15.85, 16.37, 14.87, 18.45,
        // 18.39, 16.39, 14.32 ms with 6, 8, 9, 10, 12, 16, 19 (this picks 19).
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 1;
        }
        if (sms <= 0) return 1;
        constexpr double kRamp = 9.0, kPass1 = 0.65, kSplit2 = 0.6;
        auto waves = [&](int64_t ctas) { return (double)((ctas + sms - 1) / sms); };
        auto chain = [&](int views, int L) {
            const int sp = chain_split(views);
            const double w = waves((int64_t)views * sp);
            return w * (L * (sp == 2 ? kSplit2 : 1.0) + kRamp);
        };
        const double base = chain(BH, NC);
        const int top = (int)std::min<int64_t>((int64_t)NC / 8, 4LL * sms / BH);
        double best = 0.9 * base;
        S = 1;
        for (int s = 3; s <= top; ++s) {
            const int L = (NC + s - 1) / s;
            const double w1 = waves((int64_t)BH * (2 * s - 3));
            const double c = w1 * (L * kPass1 + kRamp) + chain(BH * s, L);
            if (c < best) {
                best = c;
                S = s;
            }
        }
        if (S < 3) return 1;
    }
    if (S > NC) S = NC;
    const int L = (NC + S - 1) / S;
    return (NC + L - 1) / L;   // no empty segment
}

int segment_chunks(int T, int S) {
    const int NC = (T + C - 1) / C;
    return (NC + S - 1) / S;
}

size_t segment_workspace_bytes(int BH, int S) {
    if (S <= 1) return 0;
    // Delta and Phi for S - 1 segments, M_s for S segments
    return sizeof(float) * (size_t)BH * (size_t)(3 * S - 2) * D * D;
}

cudaError_t launch_segment_states(const void *k, const void *v, const float *g, const float *beta,
                                  float a_min, const float *init, const void *ws_tiles,
                                  float *seg_ws, int BH, int T, int S, cudaStream_t s) {
    if (S <= 1) return cudaSuccess;
    const int L = segment_chunks(T, S);
    float *delta = seg_ws;
    float *phi = delta + (size_t)BH * (S - 1) * D * D;
    float *mseg = phi + (size_t)BH * (S - 1) * D * D;
    CUtensorMap mk, mv;
    if (!make_map(&mk, k, BH, T) || !make_map(&mv, v, BH, T)) return cudaErrorInvalidValue;
    SegArgs a{g, beta, init, delta, phi, a_min, T, S, L, wait_limit_ns()};
    cudaError_t e = cudaFuncSetAttribute(seg_pass1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sp::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    // a programmatic dependent of the preparation kernel: set-up overlaps its tail, the
    // copy warp waits for its tiles
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(BH * (2 * S - 3)));
    cfg.blockDim = dim3(sp::NT);
    cfg.dynamicSmemBytes = sp::SMEM_ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int64_t nslot = (T + C - 1) / C;
    e = cudaLaunchKernelEx(&cfg, seg_pass1_kernel, mk, mv, a, static_cast<const uint8_t *>(ws_tiles), nslot);
    if (e != cudaSuccess) return e;
    const size_t smem = sizeof(float) * ((size_t)D * D + (size_t)D * kScanCols);
    e = cudaFuncSetAttribute(seg_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    seg_scan_kernel<<<dim3(D / kScanCols, (unsigned)BH), 256, smem, s>>>(init, delta, phi, mseg, S);
    return cudaGetLastError();
}

cudaError_t take_segment_error_word(unsigned *value) { return take_error_word(value); }

}  // namespace gdr
