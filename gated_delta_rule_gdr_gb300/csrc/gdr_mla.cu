// gdr_mla.cu -- one decode step of gated multi-head latent attention: the
// exact-attention layer interleaved with the incremental linear attention
// ("Trillion-Parameter MoE Multimodal LLMs: How to Evaluate the New
// Generation", section 2.1; "How to Think About Trillion-Parameter Sparse
// Multimodal LLMs", section 2.3).  The key/value projections are compressed
// into a latent space, so the cache holds one latent c_t (dc = 512 values) per
// token; the key up-projection is absorbed into the query (q_abs), so
//   score_{t,h} = scale q_abs_h . c_t,   o_h = W_uv,h sum_t softmax_t(score) c_t,
//   y_h = sigmoid(z_h) o_h.
//
// Kernel 1, mla_attn_kernel: one CTA per (split of the cache, group of 64
// heads, sequence) streams its share of the latent cache in 64-token tiles by
// TMA and runs both products on the 5th-generation tensor cores:
//   S^T = C Q^T      (M = 64 tokens, N = 64 heads, K = 512; C K-major)
//   O^T += C^T P^T   (four M = 128 blocks of the latent, N = 64 heads, K = 64
//                     tokens; C read MN-major from the same tile, P^T MN-major)
// Tokens sit on the accumulator rows of S^T, heads on its columns; O^T (256
// TMEM columns) keeps every head's 512 latent sums.  Four softmax warps read
// S^T from TMEM, take each head's maximum over the tile (a 16-lane shuffle
// reduction, then across the four warps), keep a running maximum per head and
// rescale O^T only when a head's maximum grows by more than e^8 (otherwise the
// stale maximum stays the reference and the exponentials stay below e^8),
// and write P^T in bf16 for the second product.  The partial result of the
// split -- O (unnormalised), the reference maximum and the sum of the weights
// per head -- goes to the workspace.
// Kernel 2, mla_combine_kernel: one CTA per (head, sequence) merges the splits
// (weights e^(m_s - M)), normalises, applies W_uv,h (dh x 512) and the gate.
//
// Warps of kernel 1: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2-5 softmax
// (TMEM lane quadrants 2, 3, 0, 1).  Every wait is bounded in time.

#include "gdr_fused_common.cuh"

namespace gdr {
namespace {

namespace ml {
constexpr int DC = 512;          // latent width
constexpr int HG = 64;           // heads per CTA
constexpr int TT = 64;           // tokens per tile
constexpr int NT = 192;          // 6 warps
constexpr uint32_t SLAB = 8192;  // 64 rows x 128 B
constexpr uint32_t OFF_Q = 0;                    // 8 slabs: heads x 64 latent values
constexpr uint32_t OFF_C = 8 * SLAB;             // 2 stages x 8 slabs: tokens x 64 latent values
constexpr uint32_t OFF_P = OFF_C + 2 * 8 * SLAB; // 2 buffers of P^T: tokens x 64 heads
constexpr uint32_t OFF_RED = OFF_P + 2 * SLAB;   // fp32 scratch of the softmax warps
constexpr uint32_t RED_FLOATS = 4 * 64 + 64 + 64 + 4 * 64;   // tile maxima, running max, alpha, sums
constexpr uint32_t SMEM_USED = OFF_RED + RED_FLOATS * 4;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 232448, "exceeds 227 KB of shared memory per CTA");
constexpr uint32_t TM_S = 0;     // two S^T buffers (M = 64 layout), 64 columns each
constexpr uint32_t TM_O = 128;   // four O^T blocks (M = 128), 64 columns each
constexpr uint32_t TM_COLS = 512;
constexpr float TAU = 8.0f;      // rescale O when a head's maximum grows by more than this
enum : int {
    B_Q = 0, B_CFULL0 = 1, B_CREADY0 = 3, B_CFREE0 = 5, B_SFULL0 = 7, B_PREADY0 = 9,
    B_PVDONE0 = 11, B_DRAIN = 13, NUM_BARS = 14
};
constexpr uint32_t BAR_SOFT = 1;   // named barrier of the four softmax warps
}  // namespace ml

struct MlaArgs {
    const int *seqlens;
    float *o_part;    // [N][HGn][S][64 heads][512] fp32
    float *ml_part;   // [N][HGn][S][64 heads][2] fp32: reference maximum, weight sum
    float scale;
    int Lmax, HGn, S;
    uint64_t limit_ns;
};

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t c16) {
    return row * 128u + ((c16 ^ (row & 7u)) << 4);
}

__global__ void __launch_bounds__(ml::NT, 1)
mla_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
                const MlaArgs a) {
    using namespace ml;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    __shared__ __align__(8) uint64_t s_bar[NUM_BARS];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    float *red = reinterpret_cast<float *>(sm + OFF_RED);
    float *s_tmax = red;              // [4][64]
    float *s_m = red + 256;           // [64]
    float *s_alpha = red + 320;       // [64]
    float *s_l = red + 384;           // [4][64]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, hg = blockIdx.y, n = blockIdx.z;
    int len = a.seqlens[n];
    len = len < 0 ? 0 : (len > a.Lmax ? a.Lmax : len);
    const int ntiles = (len + TT - 1) / TT;
    const int tps = (ntiles + a.S - 1) / a.S;
    const int j0 = split * tps;
    const int nt = max(0, min(ntiles, j0 + tps) - j0);
    const int tok0 = j0 * TT;
    const int64_t part = ((int64_t)n * a.HGn + hg) * a.S + split;
    auto bar = [&](int i) { return smem_u32(&s_bar[i]); };
    auto cstage = [&](int st) { return sbase + OFF_C + (uint32_t)st * 8 * SLAB; };
    auto partial = [&](int j) { return tok0 + (j + 1) * TT > len; };

    if (tid == 0) {
        mbar_init(bar(B_Q), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_CFULL0 + i), 1);
            mbar_init(bar(B_CREADY0 + i), 1);
            mbar_init(bar(B_CFREE0 + i), 1);
            mbar_init(bar(B_SFULL0 + i), 1);
            mbar_init(bar(B_PREADY0 + i), 4);
            mbar_init(bar(B_PVDONE0 + i), 1);
        }
        mbar_init(bar(B_DRAIN), 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&s_tmem), TM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_c);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ================================================================ producer
        uint32_t issued[2] = {0, 0};
        if (nt > 0 && lane == 0) {
            mbar_arrive_expect_tx(bar(B_Q), 8 * SLAB);
            for (int sl = 0; sl < 8; ++sl)
                tma_load_3d(sbase + OFF_Q + sl * SLAB, &tm_q, bar(B_Q), 64 * sl, HG * hg, n);
        }
        for (int j = 0; j < nt; ++j) {
            const int st = j & 1;
            bool ok = true;
            if (lane == 0 && j >= 2)
                ok = role_wait(bar(B_CFREE0 + st), (uint32_t)((j - 2) >> 1) & 1u, a.limit_ns, &s_abort);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(B_CFULL0 + st), 8 * SLAB);
                for (int sl = 0; sl < 8; ++sl)
                    tma_load_3d(cstage(st) + sl * SLAB, &tm_c, bar(B_CFULL0 + st), 64 * sl, tok0 + TT * j, n);
                ++issued[st];
            }
            if (partial(j)) {
                // rows past the sequence's length hold whatever the cache holds there:
                // zero them so that no stale value meets a zero weight in the products
                if (lane == 0)
                    ok = role_wait(bar(B_CFULL0 + st), (uint32_t)(j >> 1) & 1u, a.limit_ns, &s_abort);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
                const int rem = len - (tok0 + TT * j);   // 1 .. 63 valid rows
                const int nz = (TT - rem) * 8 * 8;       // 16-byte chunks to clear
                for (int x = lane; x < nz; x += 32) {
                    const int row = rem + x / 64, sl = (x / 8) % 8, c16 = x % 8;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(
                                     cstage(st) + sl * SLAB + (uint32_t)row * 128u + (uint32_t)c16 * 16u),
                                 "r"(0u)
                                 : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_CREADY0 + st));
            }
        }
        if (s_abort && lane == 0) {
            if (nt > 0) mbar_wait(bar(B_Q), 0u, kCleanupLimitNs);
            for (int st = 0; st < 2; ++st)
                if (issued[st] > 0) mbar_wait(bar(B_CFULL0 + st), (issued[st] - 1) & 1u, kCleanupLimitNs);
        }
    } else if (warp == 1) {
        // ================================================================ MMA issue
        if (lane == 0 && nt > 0) {
            const uint32_t idesc_s = idesc_bf16(64, HG, false, false);   // S^T: C K-major, Q K-major
            const uint32_t idesc_o = idesc_bf16(128, HG, true, true);    // O^T: C MN-major, P^T MN-major
            bool ok = role_wait(bar(B_Q), 0u, a.limit_ns, &s_abort);
            bool issued = false;
            auto issue_s = [&](int j) {
                const int st = j & 1;
                tc_fence_after();
                const uint64_t da = sdesc_sw128(cstage(st), 16, 1024);
                const uint64_t db = sdesc_sw128(sbase + OFF_Q, 16, 1024);
#pragma unroll 4
                for (int kk = 0; kk < DC / 16; ++kk)
                    mma_bf16(tmem + TM_S + (uint32_t)st * 64u, sdesc_add(da, (kk >> 2) * SLAB + (kk & 3) * 32),
                             sdesc_add(db, (kk >> 2) * SLAB + (kk & 3) * 32), idesc_s, kk > 0);
                mma_commit(bar(B_SFULL0 + st));
                issued = true;
            };
            auto issue_pv = [&](int j) {
                const int st = j & 1;
                tc_fence_after();
                const uint64_t dp = sdesc_sw128(sbase + OFF_P + (uint32_t)st * SLAB, 8192, 1024);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const uint64_t da = sdesc_sw128(cstage(st) + (uint32_t)(2 * b) * SLAB, SLAB, 1024);
#pragma unroll
                    for (int kk = 0; kk < TT / 16; ++kk)
                        mma_bf16(tmem + TM_O + (uint32_t)b * 64u, sdesc_add(da, kk * 2048), sdesc_add(dp, kk * 2048),
                                 idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(B_CFREE0 + st));
                mma_commit(bar(B_PVDONE0 + st));
            };
            // Issue whichever product is ready: S^T of tile js once its tile has landed
            // (and the softmax has read S^T(js - 2) from the same buffer, which it had
            // when it published P(js - 2)), the second product of tile jp once the
            // softmax has published P(jp).  Neither waits for the other's condition.
            int js = 0, jp = 0;
            uint64_t t_idle = 0;
            while (ok && jp < nt) {
                bool progress = false;
                if (js < nt && js <= jp + 1) {
                    const bool ready = partial(js) ? mbar_test_wait(bar(B_CREADY0 + (js & 1)), 0u)
                                                   : mbar_test_wait(bar(B_CFULL0 + (js & 1)), (uint32_t)(js >> 1) & 1u);
                    if (ready) {
                        issue_s(js);
                        ++js;
                        progress = true;
                    }
                }
                if (jp < js && mbar_test_wait(bar(B_PREADY0 + (jp & 1)), (uint32_t)(jp >> 1) & 1u)) {
                    issue_pv(jp);
                    ++jp;
                    progress = true;
                }
                if (progress) {
                    t_idle = 0;
                    continue;
                }
                // nothing ready: a bounded wait, as every other wait
                if (s_abort) break;
                const uint64_t now = global_timer_ns();
                if (t_idle == 0) t_idle = now;
                if (a.limit_ns == 0 || now - t_idle > a.limit_ns) {
                    s_abort = 1;
                    atomicOr(&g_device_error_word, kDevErrTimeout);
                    break;
                }
                __nanosleep(32);
            }
            if (s_abort && issued) {   // let this thread's MMAs land before TMEM goes away
                mma_commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0u, kCleanupLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ================================================================ softmax (warps 2-5)
        const int qd = warp & 3;                 // TMEM lane quadrant
        const int ts = tid - 64;                 // 0 .. 127
        const int r = 16 * qd + (lane & 15);     // token row of the tile (S^T, M = 64 layout)
        const int hf = lane >> 4;                // heads 32 hf .. 32 hf + 31
        const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
        float lp[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) lp[i] = 0.f;
        if (ts < 64) s_m[ts] = -INFINITY;
        named_sync(BAR_SOFT, 128);
        auto warp_wait = [&](int b, uint32_t parity) -> bool {
            bool ok = true;
            if (lane == 0) ok = role_wait(bar(b), parity, a.limit_ns, &s_abort);
            return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        };
        // Every softmax thread passes the same named barriers in an iteration (the votes
        // are reductions over all 128 threads, so all take the same branch); the loop is
        // left only on such a vote, so a failed wait in one warp (raising the abort flag)
        // can never strand the others at a barrier.
        bool ok = true;
        for (int j = 0; j < nt; ++j) {
            const int sb = j & 1;
            ok = ok && warp_wait(B_SFULL0 + sb, (uint32_t)(j >> 1) & 1u);
            float v[32];
            if (ok) {
                tc_fence_after();
                tmem_ld32_m64<32>(tl + TM_S + (uint32_t)sb * 64u, v);
                tmem_wait_ld();
            }
            const bool valid = ok && (tok0 + TT * j + r < len);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = valid ? v[i] * a.scale : -INFINITY;
            // Fast path: no score exceeds its head's reference maximum by more than TAU,
            // so the reference stays and no reduction is needed (one vote).
            bool exceed = j == 0;
            if (j > 0)
#pragma unroll
                for (int i = 0; i < 32; ++i) exceed |= v[i] > s_m[32 * hf + i] + TAU;
            if (!named_and(BAR_SOFT, 128, ok && !s_abort && !exceed)) {
                if (!named_and(BAR_SOFT, 128, ok && !s_abort)) {
                    ok = false;
                    break;
                }
                // the tile's maximum per head: over this warp's 16 rows, then the four warps
                {
                    float mx[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx[i] = v[i];
#pragma unroll
                    for (int off = 1; off < 16; off <<= 1)
#pragma unroll
                        for (int i = 0; i < 32; ++i) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], off));
                    if ((lane & 15) == 0)
#pragma unroll
                        for (int i = 0; i < 32; ++i) s_tmax[qd * 64 + 32 * hf + i] = mx[i];
                }
                named_sync(BAR_SOFT, 128);
                bool need = false;
                if (ts < 64) {
                    const float tm = fmaxf(fmaxf(s_tmax[ts], s_tmax[64 + ts]), fmaxf(s_tmax[128 + ts], s_tmax[192 + ts]));
                    const float mo = s_m[ts];
                    if (j == 0) {
                        s_m[ts] = tm;           // O^T is written fresh by the first product
                        s_alpha[ts] = 1.f;
                    } else if (tm > mo + TAU) {
                        s_m[ts] = tm;
                        s_alpha[ts] = __expf(mo - tm);
                        need = true;
                    } else {
                        s_alpha[ts] = 1.f;
                    }
                }
                const bool rescale = !named_and(BAR_SOFT, 128, !need);
                if (ok && rescale) {
                    // O^T may change only once the product of the previous tile has landed
                    ok = warp_wait(B_PVDONE0 + ((j - 1) & 1), (uint32_t)((j - 1) >> 1) & 1u);
                    if (ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int b = 0; b < 4; ++b)
#pragma unroll 1
                            for (int cb = 0; cb < 2; ++cb) {
                                float o[32];
                                const uint32_t ta = tl + TM_O + (uint32_t)b * 64u + (uint32_t)cb * 32u;
                                tmem_ld32(ta, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 32; ++i) o[i] *= s_alpha[32 * cb + i];
                                tmem_st32(ta, o);
                            }
                        tmem_wait_st();
#pragma unroll
                        for (int i = 0; i < 32; ++i) lp[i] *= s_alpha[32 * hf + i];
                    }
                }
            }
            // P buffer sb was last read by the product of tile j - 2
            if (ok && j >= 2) ok = warp_wait(B_PVDONE0 + sb, (uint32_t)((j - 2) >> 1) & 1u);
            if (ok) {
                float p[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    p[i] = valid ? __expf(v[i] - s_m[32 * hf + i]) : 0.f;
                    lp[i] += p[i];
                }
                const uint32_t pb = sbase + OFF_P + (uint32_t)sb * SLAB;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t addr = pb + swz((uint32_t)r, (uint32_t)(4 * hf + k));
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                 "r"(pack_bf16x2(p[8 * k + 0], p[8 * k + 1])),
                                 "r"(pack_bf16x2(p[8 * k + 2], p[8 * k + 3])),
                                 "r"(pack_bf16x2(p[8 * k + 4], p[8 * k + 5])),
                                 "r"(pack_bf16x2(p[8 * k + 6], p[8 * k + 7]))
                                 : "memory");
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_PREADY0 + sb));
            }
        }
        // ---- the split's partial result
        if (ok && nt > 0 && !warp_wait(B_PVDONE0 + ((nt - 1) & 1), (uint32_t)((nt - 1) >> 1) & 1u)) ok = false;
        if (ok) {
#pragma unroll
            for (int off = 1; off < 16; off <<= 1)
#pragma unroll
                for (int i = 0; i < 32; ++i) lp[i] += __shfl_xor_sync(0xffffffffu, lp[i], off);
            if ((lane & 15) == 0)
#pragma unroll
                for (int i = 0; i < 32; ++i) s_l[qd * 64 + 32 * hf + i] = lp[i];
        }
        named_sync(BAR_SOFT, 128);
        if (ok) {
            float *ml = a.ml_part + part * HG * 2;
            if (ts < 64) {
                ml[2 * ts] = nt > 0 ? s_m[ts] : -INFINITY;
                ml[2 * ts + 1] = nt > 0 ? s_l[ts] + s_l[64 + ts] + s_l[128 + ts] + s_l[192 + ts] : 0.f;
            }
            float *op = a.o_part + part * HG * DC;
            tc_fence_after();
#pragma unroll 1
            for (int b = 0; b < 4; ++b)
#pragma unroll 1
                for (int cb = 0; cb < 2; ++cb) {
                    float o[32];
                    if (nt > 0) {
                        tmem_ld32(tl + TM_O + (uint32_t)b * 64u + (uint32_t)cb * 32u, o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0.f;
                    }
                    const int c = 128 * b + 32 * qd + lane;   // latent index of this thread's row
#pragma unroll
                    for (int i = 0; i < 32; ++i) op[(int64_t)(32 * cb + i) * DC + c] = o[i];
                }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, TM_COLS);
    }
}

// Merge the splits of one (head, sequence), normalise, apply W_uv,h and the gate.
// The splits' maxima and sums are staged first (one thread each), the partial sums
// are read with several splits in flight per thread, and each warp takes four rows
// of W_uv at a time, so that the loads overlap instead of following each other.
__global__ void __launch_bounds__(128)
mla_combine_kernel(const float *__restrict__ o_part, const float *__restrict__ ml_part,
                   const __nv_bfloat16 *__restrict__ w_uv, const float *__restrict__ gate,
                   __nv_bfloat16 *__restrict__ out, int H, int HGn, int S, int dh) {
    constexpr int DC = ml::DC;
    __shared__ float s_o[DC];
    __shared__ float s_w[64];   // e^(m_s - M), then the weight of split s
    __shared__ float s_l[64];
    __shared__ float s_inv;
    const int h = blockIdx.x, n = blockIdx.y, tid = threadIdx.x;
    const int hg = h / ml::HG, hl = h % ml::HG;
    const int64_t p0 = ((int64_t)n * HGn + hg) * S;
    if (tid < S) {
        const float2 ml2 = *reinterpret_cast<const float2 *>(ml_part + ((p0 + tid) * ml::HG + hl) * 2);
        s_w[tid] = ml2.x;
        s_l[tid] = ml2.y;
    }
    __syncthreads();
    if (tid < 32) {   // M, the split weights and 1 / (sum of the weights), one warp
        float M = -INFINITY;
        for (int s = tid; s < S; s += 32) M = fmaxf(M, s_w[s]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float lt = 0.f;
        for (int s = tid; s < S; s += 32) {
            const float w = M == -INFINITY ? 0.f : __expf(s_w[s] - M);
            s_w[s] = w;
            lt = fmaf(w, s_l[s], lt);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(0xffffffffu, lt, off);
        if (tid == 0) s_inv = lt > 0.f ? 1.f / lt : 0.f;   // an empty cache contributes zero
    }
    __syncthreads();
    {
        const float *src = o_part + (p0 * ml::HG + hl) * DC + tid;
        const int64_t stride = (int64_t)ml::HG * DC;   // between splits
        float acc[DC / 128] = {};
        int s = 0;
        for (; s + 4 <= S; s += 4) {
            float x[4][DC / 128];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int e = 0; e < DC / 128; ++e) x[u][e] = src[(s + u) * stride + 128 * e];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int e = 0; e < DC / 128; ++e) acc[e] = fmaf(s_w[s + u], x[u][e], acc[e]);
        }
        for (; s < S; ++s)
#pragma unroll
            for (int e = 0; e < DC / 128; ++e) acc[e] = fmaf(s_w[s], src[s * stride + 128 * e], acc[e]);
        const float inv = s_inv;
#pragma unroll
        for (int e = 0; e < DC / 128; ++e) s_o[tid + 128 * e] = acc[e] * inv;
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    float o16[16];   // this lane's latent values 16 lane .. 16 lane + 15
#pragma unroll
    for (int e = 0; e < 16; ++e) o16[e] = s_o[16 * lane + e];
    for (int j0 = 4 * warp; j0 < dh; j0 += 16) {   // rows j0 .. j0 + 3 of this warp
        uint4 u[4][2];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int j = min(j0 + rr, dh - 1);
            const uint4 *row = reinterpret_cast<const uint4 *>(w_uv + ((int64_t)h * dh + j) * DC) + 2 * lane;
            u[rr][0] = row[0];
            u[rr][1] = row[1];
        }
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const uint32_t w4[4] = {u[rr][e].x, u[rr][e].y, u[rr][e].z, u[rr][e].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[k]));
                    acc = fmaf(f.x, o16[8 * e + 2 * k], fmaf(f.y, o16[8 * e + 2 * k + 1], acc));
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            const int j = j0 + rr;
            if (lane == 0 && j < dh) {
                const int64_t idx = ((int64_t)n * H + h) * dh + j;
                out[idx] = __float2bfloat16_rn(acc / (1.f + __expf(-gate[idx])));
            }
        }
    }
}

bool make_map_mla(CUtensorMap *m, const void *ptr, int rows, int N) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)ml::DC, (cuuint64_t)rows, (cuuint64_t)N};
    cuuint64_t strides[2] = {(cuuint64_t)ml::DC * 2, (cuuint64_t)rows * ml::DC * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool mla_supported(int H, int dc, int dh) {
    return dc == ml::DC && H > 0 && H % ml::HG == 0 && dh > 0 && dh % 4 == 0 && dh <= 1024;
}

int mla_splits(int N, int H, int Lmax) {
    // Splits of each sequence's cache.  One CTA per (split, head group, sequence)
    // fills an SM, so the step takes ceil(CTAs / SMs) rounds of ceil(tiles / S)
    // tiles each; a split's partial result (128 KB written, then read by the merge)
    // moves as many bytes as about four tiles.  The count minimising
    // rounds x (tiles + 4) wins, which favours whole waves.
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        sms = 148;
    }
    const int64_t groups = (int64_t)N * (H / ml::HG);
    const int64_t tiles = (Lmax + ml::TT - 1) / ml::TT;
    int best = 1;
    int64_t best_cost = -1;
    for (int s = 1; s <= 64 && s <= tiles; ++s) {
        const int64_t rounds = (groups * s + sms - 1) / sms;
        const int64_t cost = rounds * ((tiles + s - 1) / s + 4);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

size_t mla_workspace_bytes(int N, int H, int Lmax) {
    const int64_t parts = (int64_t)N * (H / ml::HG) * mla_splits(N, H, Lmax);
    return (size_t)parts * ml::HG * (ml::DC + 2) * sizeof(float);
}

cudaError_t launch_mla_decode(const void *q_abs, const void *ckv, const int *seqlens, const void *w_uv,
                              const float *gate, float scale, void *out, int N, int H, int Lmax, int dh,
                              void *ws, cudaStream_t s) {
    if ((int64_t)N * H == 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(q_abs) | reinterpret_cast<uintptr_t>(ckv) |
         reinterpret_cast<uintptr_t>(w_uv) | reinterpret_cast<uintptr_t>(ws)) & 15)
        return cudaErrorMisalignedAddress;
    const int HGn = H / ml::HG;
    const int S = mla_splits(N, H, Lmax);
    CUtensorMap mq, mc;
    if (!make_map_mla(&mq, q_abs, H, N) || !make_map_mla(&mc, ckv, Lmax, N)) return cudaErrorInvalidValue;
    float *o_part = static_cast<float *>(ws);
    float *ml_part = o_part + (size_t)N * HGn * S * ml::HG * ml::DC;
    MlaArgs a{seqlens, o_part, ml_part, scale, Lmax, HGn, S, wait_limit_ns()};
    cudaError_t e = cudaFuncSetAttribute(mla_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)ml::SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    mla_attn_kernel<<<dim3((unsigned)S, (unsigned)HGn, (unsigned)N), ml::NT, ml::SMEM_ALLOC, s>>>(mq, mc, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mla_combine_kernel<<<dim3((unsigned)H, (unsigned)N), 128, 0, s>>>(
        o_part, ml_part, static_cast<const __nv_bfloat16 *>(w_uv), gate, static_cast<__nv_bfloat16 *>(out), H,
        HGn, S, dh);
    return cudaGetLastError();
}

cudaError_t take_mla_error_word(unsigned *value) { return take_error_word(value); }

}  // namespace gdr
