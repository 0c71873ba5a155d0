// gdr_fused_common.cuh -- pieces shared by the fused tensor-core prefill
// kernels (one CTA per head, and the value-split pair per head): the chunk
// geometry, bf16 tile writes, bounded role waits, the per-chunk decay of one
// warp, the 64 x 64 unit-lower triangular solve and the TMA map of a
// [BH][T][128] bf16 tensor.  Everything here has internal linkage: each
// kernel translation unit gets its own copy, including its own device error
// word, which its host code reads and clears.
#pragma once

#include "gdr_internal.h"
#include "gdr_math.cuh"
#include "gdr_sm100.cuh"

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>

namespace gdr {
namespace {

using namespace sm100;

constexpr int C = 64;      // chunk
constexpr int D = 128;     // dk (and dv of the input tensors)
constexpr int NPREP = 256; // threads of the preparation warps
constexpr uint32_t BAR_PREP = 1, BAR_CHAIN = 2;   // named barriers (0 is __syncthreads)
constexpr uint32_t BAR_EROWS = 3, BAR_OROWS = 4;  // chain warps owning rows 0-63 / 64-127 of X
constexpr int LDA = 68;    // fp32 row stride of the solve matrices
constexpr int LDY = 40;    // row stride of the merge scratch
constexpr uint64_t kCleanupLimitNs = 2000000000ull;

// Sticky device error word of this translation unit's kernels.
__device__ unsigned g_device_error_word = 0;

struct Scal {   // per-stage per-row scalars of one chunk
    float *gam, *ig, *bs, *bg, *sc;   // gamma, 1/gamma, beta, beta gamma, gamma_C / gamma
};

__device__ __forceinline__ Scal scal_at(float *b) {   // 5 x 64 floats
    return {b, b + 64, b + 128, b + 192, b + 256};
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Write 32 fp32 values as half a 128-byte bf16 row (chunks 4h..4h+3).
__device__ __forceinline__ void st_halfrow_bf16(uint8_t *tile, uint32_t row, uint32_t h,
                                                const float *v) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t ch = h * 4 + q4;
        uint4 u;
        u.x = pack_bf16x2(v[q4 * 8 + 0], v[q4 * 8 + 1]);
        u.y = pack_bf16x2(v[q4 * 8 + 2], v[q4 * 8 + 3]);
        u.z = pack_bf16x2(v[q4 * 8 + 4], v[q4 * 8 + 5]);
        u.w = pack_bf16x2(v[q4 * 8 + 6], v[q4 * 8 + 7]);
        *reinterpret_cast<uint4 *>(tile + row * 128u + ((ch ^ (row & 7u)) << 4)) = u;
    }
}

// Bounded wait used by the warp roles: gives up when the CTA-wide abort flag is
// raised or the time limit passes (then raises the flag and the error word).
// Each try suspends the thread until the phase completes or kWaitSliceNs pass,
// so a waiting thread takes no issue slots from the working warps; one thread
// per role waits and a named barrier passes the result on.
constexpr uint32_t kWaitSliceNs = 20000;
__device__ __noinline__ bool role_wait_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                            volatile int *abort, bool cluster_scope) {
    if (limit_ns == 0) {                                // injected timeout: give up at once
        *abort = 1;
        atomicOr(&g_device_error_word, kDevErrTimeout);
        return false;
    }
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (cluster_scope ? mbar_try_wait_cluster_hint(bar, parity, kWaitSliceNs)
                          : mbar_try_wait_hint(bar, parity, kWaitSliceNs))
            return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort = 1;
            atomicOr(&g_device_error_word, kDevErrTimeout);
            return false;
        }
    }
}
// The common case -- the phase has already completed -- stays inline.
__device__ __forceinline__ bool role_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                          volatile int *abort) {
    if (mbar_test_wait(bar, parity)) return true;
    return role_wait_slow(bar, parity, limit_ns, abort, false);
}
// role_wait for barriers that another CTA of the cluster arrives on
// (cluster-scope acquire).
__device__ __forceinline__ bool role_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  volatile int *abort) {
    if (mbar_test_wait_cluster(bar, parity)) return true;
    return role_wait_slow(bar, parity, limit_ns, abort, true);
}

// Cumulative decay of one chunk by one warp (lane l owns rows 2l, 2l+1, whose
// g and beta it already holds): alpha = a_min + (1 - a_min) sigmoid(g) (or, for
// a_min <= 0, the log-domain form log alpha = a_min sigmoid(g)), the
// inclusive scan of log alpha, gamma = exp(scan), 1/gamma, beta, beta gamma,
// gamma_C (the last valid row) and gamma_C / gamma.  Rows past the chunk's end
// get gamma = 1, beta = 0 and gamma_C / gamma = 0 so that they drop out of
// every product.  log alpha = log1p(-(1 - a_min) / (1 + e^g)) keeps alpha
// close to 1 accurate; the exponentials and reciprocals use the hardware
// approximations (relative error below 1e-5 over the range the range rule
// allows, far inside the bf16 tolerance of the fused path).
__device__ __forceinline__ void warp_decay_inl(int lane, float g0, float g1, float be0, float be1, int c,
                                               float a_min, Scal s, float *s_gC) {
    const float gv[2] = {g0, g1}, bv[2] = {be0, be1};
    const int r0 = 2 * lane;
    // a_min > 0: the linear-domain floor; a_min <= 0: log alpha = a_min sigmoid(g)
    const float om = 1.0f - a_min;
    auto la = [&](float gg) {
        return a_min > 0.0f ? log1pf(-__fdividef(om, 1.0f + __expf(gg)))
                            : a_min * __fdividef(1.0f, 1.0f + __expf(-gg));
    };
    const float l0 = (r0 < c) ? la(gv[0]) : 0.f;
    const float l1 = (r0 + 1 < c) ? la(gv[1]) : 0.f;
    float incl = l0 + l1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float b1 = incl, b0 = incl - l1;
    // gamma_C: the scan value of row c - 1, held by lane (c - 1) / 2
    const float bC = __shfl_sync(0xffffffffu, ((c - 1) & 1) ? b1 : b0, (c - 1) >> 1);
    const float gC = __expf(bC);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = r0 + e;
        const bool valid = r < c;
        const float gam = valid ? __expf(e ? b1 : b0) : 1.f;
        const float ig = __frcp_rn(gam);
        const float b = valid ? bv[e] : 0.f;
        s.gam[r] = gam;
        s.ig[r] = ig;
        s.bs[r] = b;
        s.bg[r] = b * gam;
        // gamma_C / gamma as one exponential of the difference (at most 1), so that
        // it stays exact where gamma alone underflows
        s.sc[r] = valid ? __expf(bC - (e ? b1 : b0)) : 0.f;
    }
    if (lane == 0) *s_gC = gC;
    __syncwarp();
}
// Scalars of the preparation's diagonal tile with 16-row reference points.
// The decay over a whole 64-row chunk may span far more than fp32 can hold as
// gamma and 1/gamma (the pages bound it over 16-token tiles only), so the
// position-pair factor e^(b_r - b_s) of row r in block R = r / 16 is split at
// rho_R = b_{16 R}: a row factor e^(b_r - rho_R) in (e^-80, 1] and a column
// factor e^(rho_R - b_s), at most e^80 for s in block R and at most 1 for s in
// an earlier block.  Both stay finite whenever 16 |log alpha| <= 80, and their
// product underflows only where the exact factor is below fp32's range.
// Writes rf[r] = beta_r e^(b_r - rho_R), pf[r] = e^(b_r - rho_R), bs[r] = beta_r
// (zero past the chunk's c rows) and cf[R * 64 + s] = e^(rho_R - b_s) for s <
// min(16 R + 16, c), zero elsewhere.  Warp-wide; lane l holds rows 2l, 2l + 1.
struct TileScal {
    float *rf, *pf, *bs, *cf;   // 64, 64, 64 and 4 x 64 floats
};
__device__ __forceinline__ TileScal tile_scal_at(float *b) {   // 7 x 64 floats
    return {b, b + 64, b + 128, b + 192};
}
__device__ __forceinline__ void warp_decay_tiles(int lane, float g0, float g1, float be0, float be1,
                                                 int c, float a_min, TileScal s) {
    const int r0 = 2 * lane;
    const float om = 1.0f - a_min;
    auto la = [&](float gg) {
        return a_min > 0.0f ? log1pf(-__fdividef(om, 1.0f + __expf(gg)))
                            : a_min * __fdividef(1.0f, 1.0f + __expf(-gg));
    };
    const float l0 = (r0 < c) ? la(g0) : 0.f;
    const float l1 = (r0 + 1 < c) ? la(g1) : 0.f;
    float incl = l0 + l1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float b[2] = {incl - l1, incl};
    float rho[4];   // b at rows 0, 16, 32, 48: the b[0] of lanes 0, 8, 16, 24
#pragma unroll
    for (int R = 0; R < 4; ++R) rho[R] = __shfl_sync(0xffffffffu, b[0], 8 * R);
    const float bt[2] = {be0, be1};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = r0 + e;
        const bool valid = r < c;
        const float f = valid ? __expf(b[e] - rho[r >> 4]) : 0.f;
        s.pf[r] = f;
        s.rf[r] = valid ? bt[e] * f : 0.f;
        s.bs[r] = valid ? bt[e] : 0.f;
#pragma unroll
        for (int R = 0; R < 4; ++R)
            s.cf[R * 64 + r] = (valid && (r >> 4) <= R) ? __expf(rho[R] - b[e]) : 0.f;
    }
    __syncwarp();
}

// The same, not inlined, for the copy warps of the fused and chain kernels: they
// call it at two places, and its code would otherwise crowd the instruction
// cache the other warps share.  (A warp with many live registers inlines it
// instead: a call would save and restore them.)  The values cross the call in
// registers, so loads issued ahead of the call stay in flight until it.
__device__ __noinline__ void warp_decay_v(int lane, float g0, float g1, float be0, float be1, int c,
                                          float a_min, Scal s, float *s_gC) {
    warp_decay_inl(lane, g0, g1, be0, be1, c, a_min, s, s_gC);
}
__device__ __forceinline__ void warp_decay(int lane, const float (&gv)[2], const float (&bv)[2],
                                           int c, float a_min, Scal s, float *s_gC) {
    warp_decay_v(lane, gv[0], gv[1], bv[0], bv[1], c, a_min, s, s_gC);
}

// tf32 warp-level MMA (m16n8k8) for the small merge products of the solve.
// Fragment layouts (g = lane / 4, t = lane % 4): A (16 x 8) a0 (g, t), a1
// (g+8, t), a2 (g, t+4), a3 (g+8, t+4); B (8 x 8) b0 (t, g), b1 (t+4, g);
// C (16 x 8) c0 (g, 2t), c1 (g, 2t+1), c2 (g+8, 2t), c3 (g+8, 2t+1).
// fp32 -> tf32 bit pattern, rounded to nearest with ties away from zero: add
// half of the 13 dropped mantissa bits' weight, then clear them (finite inputs;
// the solve's operands always are).  Two integer operations.
__device__ __forceinline__ uint32_t to_tf32(float x) {
    return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], const float *M, int ld, int r0, int c0,
                                       int lane) {
    const int g = lane >> 2, t = lane & 3;
    a[0] = to_tf32(M[(r0 + g) * ld + c0 + t]);
    a[1] = to_tf32(M[(r0 + g + 8) * ld + c0 + t]);
    a[2] = to_tf32(M[(r0 + g) * ld + c0 + t + 4]);
    a[3] = to_tf32(M[(r0 + g + 8) * ld + c0 + t + 4]);
}
__device__ __forceinline__ void frag_b(uint32_t (&b)[2], const float *M, int ld, int k0, int n0,
                                       int lane) {
    const int g = lane >> 2, t = lane & 3;
    b[0] = to_tf32(M[(k0 + t) * ld + n0 + g]);
    b[1] = to_tf32(M[(k0 + t + 4) * ld + n0 + g]);
}
__device__ __forceinline__ void frag_store(float *M, int ld, int r0, int n0, const float (&d)[4],
                                           float sign, int lane) {
    const int g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2 *>(&M[(r0 + g) * ld + n0 + 2 * t]) = make_float2(sign * d[0], sign * d[1]);
    *reinterpret_cast<float2 *>(&M[(r0 + g + 8) * ld + n0 + 2 * t]) =
        make_float2(sign * d[2], sign * d[3]);
}

// T = (I + A)^-1 for the strictly lower 64 x 64 A in As (fp32), into Ts (which
// may be As itself: every block of A is read before T overwrites it), by
// the prep warps (w = thread index 0..255).  Blocked: four 16 x 16
// diagonal inverses by right-looking forward substitution in fp32 (one column
// per thread), then two merge levels T_ij = -T_ii (A_ij T_jj) on tf32 warp
// MMAs.  On return the lower triangle of Ts holds T; the 16 x 16 blocks right
// of the even diagonal blocks hold zeros (the merges read them).  T feeds
// bf16 tensor-core operands, so the tf32 merges cost no accuracy that matters.
template <int NTH>   // 256 or 128 threads (a multiple of 4 warps)
__device__ __forceinline__ void solve_unit_lower_t(int w, const float *As, float *Ts, float *Ys) {
    static_assert(NTH == 256 || NTH == 128, "the solve runs on 4 or 8 warps");
    const int lane = w & 31, wp = w >> 5;
    if (w < 64) {
        const int b = w >> 4, l = w & 15, o = 16 * b;
        float x[16], acc[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            x[m] = (m == l) ? 1.f : 0.f;
            acc[m] = 0.f;
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            if (m > l) x[m] = -acc[m];          // x[m] is final from here on
#pragma unroll
            for (int r = m + 1; r < 16; ++r) acc[r] = fmaf(As[(o + r) * LDA + o + m], x[m], acc[r]);
        }
        __syncwarp();   // the block's 16 lanes have read it: T may overwrite A (in place)
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            Ts[(o + r) * LDA + o + l] = x[r];
            if ((b & 1) == 0) Ts[(o + r) * LDA + o + 16 + l] = 0.f;
        }
    }
    named_sync(BAR_PREP, NTH);
    {   // level 1: T(1,0) and T(3,2); warps 0-3 -> (pair, 8-column tile)
        const int p = (wp >> 1) & 1, nt = wp & 1;
        const int R = 16 * (2 * p + 1), Cb = 16 * (2 * p);
        if (wp < 4) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t fa[4], fb[2];
                frag_a(fa, As, LDA, R, Cb + 8 * ks, lane);
                frag_b(fb, Ts, LDA, Cb + 8 * ks, Cb + 8 * nt, lane);
                mma_tf32(d, fa, fb);
            }
            frag_store(Ys + p * 16 * LDY, LDY, 0, 8 * nt, d, 1.f, lane);
        }
        named_sync(BAR_PREP, NTH);
        if (wp < 4) {
            float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t fa[4], fb[2];
                frag_a(fa, Ts, LDA, R, R + 8 * ks, lane);          // zero above the diagonal
                frag_b(fb, Ys + p * 16 * LDY, LDY, 8 * ks, 8 * nt, lane);
                mma_tf32(e, fa, fb);
            }
            frag_store(Ts, LDA, R, Cb + 8 * nt, e, -1.f, lane);
        }
    }
    named_sync(BAR_PREP, NTH);
    {   // level 2: T[32:64, 0:32] = -T[32:64, 32:64] (A[32:64, 0:32] T[0:32, 0:32]);
        // task -> (16-row tile, 8-column tile), 8 tasks over the warps
#pragma unroll
        for (int task = wp; task < 8; task += NTH / 32) {
            const int m0 = 16 * (task & 1), n0 = 8 * (task >> 1);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t fb[2], fa[4];
                frag_b(fb, Ts, LDA, 8 * ks, n0, lane);
                frag_a(fa, As, LDA, 32 + m0, 8 * ks, lane);
                mma_tf32(d, fa, fb);
            }
            frag_store(Ys, LDY, m0, n0, d, 1.f, lane);
        }
        named_sync(BAR_PREP, NTH);
#pragma unroll
        for (int task = wp; task < 8; task += NTH / 32) {
            const int m0 = 16 * (task & 1), n0 = 8 * (task >> 1);
            float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t fb[2], fa[4];
                frag_b(fb, Ys, LDY, 8 * ks, n0, lane);
                frag_a(fa, Ts, LDA, 32 + m0, 32 + 8 * ks, lane);
                mma_tf32(e, fa, fb);
            }
            frag_store(Ts, LDA, 32 + m0, n0, e, -1.f, lane);
        }
    }
    named_sync(BAR_PREP, NTH);
}
__device__ __forceinline__ void solve_unit_lower(int w, const float *As, float *Ts, float *Ys) {
    solve_unit_lower_t<NPREP>(w, As, Ts, Ys);
}

struct FusedArgs {
    const float *g, *beta, *init;
    __nv_bfloat16 *out;
    float *final_state;
    float a_min;
    int T;
    uint64_t limit_ns;
    const __nv_bfloat16 *v = nullptr;   // read directly by kernels that load v rows themselves
    // Packed variable-length sequences: q, k, v, out [total_T][H][d], g, beta
    // [total_T][H], sequence s = tokens cu_seqlens[s] .. cu_seqlens[s+1]; the
    // state index is s H + h.  nullptr = the dense [B][H][T] layout.
    const int *cu_seqlens = nullptr;
    int H = 0, total_T = 0;
    // Sequence segments of the dense layout (nseg > 1, the two-kernel path only):
    // view v = bh nseg + s covers chunks s seg_chunks .. of head bh, starts from
    // seg_init[v] ([dk][dv] fp32, written by the segment scan) and, for the last
    // segment only, writes the head's final state.
    int nseg = 1, seg_chunks = 0;
    const float *seg_init = nullptr;
    // Saving for the backward (the two-kernel chain, dense layout): every chunk's state
    // M_n^T and W_n^T leave as value-major bf16 tiles through two tensor maps.
    int save = 0;
};

// Where the tokens of the (sequence, head) with state index bh live.  Token t
// (0 <= t < T) of it: g / beta index gbase + t * stride, out row (d elements)
// obase + t * stride, TMA coordinates (x, tz + t, z).
struct SeqView {
    int T, tz, z, stride;
    int64_t gbase;
};
__device__ __forceinline__ SeqView seq_view(const FusedArgs &a, int bh) {
    SeqView v;
    if (!a.cu_seqlens && a.nseg > 1) {   // segment bh % nseg of head bh / nseg
        const int h = bh / a.nseg, sg = bh % a.nseg;
        const int t0 = sg * a.seg_chunks * C;
        v.T = max(0, min(a.seg_chunks * C, a.T - t0));
        v.tz = t0;
        v.z = h;
        v.stride = 1;
        v.gbase = (int64_t)h * a.T + t0;
    } else if (!a.cu_seqlens) {
        v.T = a.T;
        v.tz = 0;
        v.z = bh;
        v.stride = 1;
        v.gbase = (int64_t)bh * a.T;
    } else {
        // clamped into [0, total_T] so that a malformed offset array cannot take
        // a CTA out of the tensors
        const int s = bh / a.H, h = bh % a.H;
        const int t0 = min(max(a.cu_seqlens[s], 0), a.total_T);
        const int t1 = min(max(a.cu_seqlens[s + 1], t0), a.total_T);
        v.T = t1 - t0;
        v.tz = t0;
        v.z = h;
        v.stride = a.H;
        v.gbase = (int64_t)t0 * a.H + h;
    }
    return v;
}

// Tiles of the two-kernel path: the preparation writes the [Lb | P] tile of
// chunk n of a (sequence, head) view to tile index z * nslot + slot0 + n of
// the workspace, and the chain kernel reads it there.
//   dense [B][H][T]:  z = bh, nslot = ceil(T / C), slot0 = 0
//   packed sequences: z = h,  nslot = total_T / C + S + 1, slot0 = t0 / C + s
// (t0 the sequence's first token).  Packed slots never overlap: sequence s
// ends below t1 / C + s + 1 <= slot0 of s + 1, and every slot of a malformed
// offset array still falls inside [0, nslot).
constexpr uint32_t TILE_BYTES = 16384;   // [Lb rows | P rows] bf16, 128-byte swizzled rows

__host__ __device__ __forceinline__ int64_t tile_slots(const FusedArgs &a, int BH) {
    return a.cu_seqlens ? (int64_t)(a.total_T / C + BH / a.H + 1) : (int64_t)((a.T + C - 1) / C);
}
__device__ __forceinline__ int tile_slot0(const FusedArgs &a, int bh, const SeqView &v) {
    return a.cu_seqlens ? v.tz / C + bh / a.H : v.tz / C;
}
// Initial state of view bh ([dk][dv] fp32, or nullptr = zeros) and its final state
// (nullptr = not written).  Segment views start from the scan's states and only the
// last segment of a head writes the final state.
__device__ __forceinline__ const float *view_init(const FusedArgs &a, int bh) {
    if (a.nseg > 1) return a.seg_init + (int64_t)bh * D * D;
    return a.init ? a.init + (int64_t)bh * D * D : nullptr;
}
__device__ __forceinline__ float *view_final(const FusedArgs &a, int bh) {
    if (!a.final_state) return nullptr;
    if (a.nseg > 1)
        return bh % a.nseg == a.nseg - 1 ? a.final_state + (int64_t)(bh / a.nseg) * D * D : nullptr;
    return a.final_state + (int64_t)bh * D * D;
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

// Packed [total_T][H][128] bf16 as a 3-D tensor (d, t, h): 64 x 64 boxes of
// consecutive tokens of one head, 128-byte swizzle, zero fill beyond total_T.
bool make_map_packed(CUtensorMap *m, const void *ptr, int H, int total_T) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)total_T, (cuuint64_t)H};
    cuuint64_t strides[2] = {(cuuint64_t)H * D * 2, (cuuint64_t)D * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bound of every device-side wait: 2 s unless gdr_set_option changed it (0
// makes every wait give up at once, which drives the error path in tests
// without any GPU fault).
uint64_t wait_limit_ns() { return opt_wait_limit_ns(); }

// Reads and clears this translation unit's device error word (synchronous).
cudaError_t take_error_word(unsigned *value) {
    unsigned word = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&word, g_device_error_word, sizeof(word));
    if (e != cudaSuccess) return e;
    *value = word;
    if (word != 0) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace
}  // namespace gdr
