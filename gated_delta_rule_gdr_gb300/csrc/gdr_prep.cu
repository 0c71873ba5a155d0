// gdr_prep.cu -- the state-independent preparation of every chunk of a
// prefill, as one fully parallel kernel (the first half of the two-kernel
// path; gdr_chain.cu is the second).
//
// Per chunk (sections 3.1-3.3 of "What a Trillion-Parameter MoE Model Reveals
// About the Next Stage of LLM Scaling": with the lower-bounded decay the
// reciprocal decay stays finite over a 16-token tile, and the causal tile is a
// dense product with diagonal scalings):
//   [K;Q] K^T                                  (tcgen05, M = 128, N = 64, K = 128)
//   A  = strict_lower(diag(beta) D o K K^T),  T = (I + A)^-1
//   Lb = bf16(strict_lower(T) diag(beta)),  P = bf16(lower_incl(D o Q K^T))
// with D[r][s] = e^(b_r - b_s) the decay between positions s <= r, applied as
// the diagonal scalings of the pages' 16-token tiles: row r of 16-row block R
// takes e^(b_r - b_{16R}), column s takes e^(b_{16R} - b_s) for that block, so
// no factor leaves fp32's range however far the decay falls over the chunk.
// and the [Lb | P] tile (16 KB, the 128-byte-swizzled shared-memory image the
// chain kernel loads verbatim) goes to the workspace.  Nothing here depends on
// the state, so every (sequence, head, chunk) is an independent work item; a
// persistent grid walks them, each CTA loading its next item's K and Q while it
// prepares the current one.
//
// For training (tpb, tsc given) it also writes what the backward's tiles and
// decay kernels would recompute: T and P as bf16 [64][64] tiles with the 128-byte
// swizzle (P is the tile's half as it is), and the chunk's row scalars gamma, 1/gamma, beta,
// d log(alpha)/dg (rows past the chunk's end 1, 1, 0, 0).
//
// CTA: 128 threads, three per SM.  Thread 0 issues the TMA loads, the
// tensor-core product and the bulk store of each tile; warp 3 computes the
// decay (away from the warp that issues the product, whose later instructions
// wait behind it) and loads the next item's g and beta; the four warps read the
// accumulator (TMEM lane quadrant = warp), solve and convert.  Shared memory:
// the input buffer (K and Q in two 64-column slabs; the next item's load goes
// in as soon as the product has consumed them), the tile buffer, the fp32
// solve space, the chunk scalars.

#include "gdr_fused_common.cuh"

namespace gdr {
namespace {

constexpr int NT = 128;
constexpr int CTAS_PER_SM = 3;
constexpr uint32_t IN_BYTES = 32768;                    // [slab i/64][K rows | Q rows][128 B]
constexpr uint32_t OFF_IN = 0;
constexpr uint32_t OFF_OUT = OFF_IN + IN_BYTES;         // the [Lb | P] tile (16 KB)
constexpr uint32_t LP_TILE_P = 8192;                    // P within the tile
constexpr uint32_t OFF_AS = OFF_OUT + TILE_BYTES;       // 64 x 68 fp32: A, then T in place
constexpr uint32_t OFF_YS = OFF_AS + 64 * LDA * 4;      // 32 x 40 fp32 merge scratch
constexpr uint32_t OFF_SC = OFF_YS + 32 * LDY * 4;      // 7 x 64 fp32 tile scalars
constexpr uint32_t SMEM_USED = OFF_SC + 7 * 64 * 4;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;       // alignment slack
static_assert(IN_BYTES % 1024 == 0 && OFF_OUT % 1024 == 0, "swizzled tiles must be 1024-byte aligned");
static_assert(CTAS_PER_SM * SMEM_ALLOC <= 232448, "CTAs per SM");
constexpr uint32_t TM_COLS = 64;

enum : int { B_FULL = 0, B_KQK = 1, B_DRAIN = 2, NUM_BARS = 3 };


__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t c8) {
    return row * 128u + ((c8 ^ (row & 7u)) << 4);
}

// Work item -> (bh, n) of a chunk, false for a padding slot of the packed layout.
__device__ bool item_chunk(const FusedArgs &a, int BH, int nslot, int item, int &bh, int &n,
                           SeqView &v) {
    const int z = item / nslot, u = item - z * nslot;
    if (!a.cu_seqlens) {
        bh = z;
        n = u;
        v = seq_view(a, bh);
        return true;
    }
    // the last sequence s whose first slot t0(s) / C + s is at most u
    const int S = BH / a.H;
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const int t0 = min(max(a.cu_seqlens[mid], 0), a.total_T);
        if (t0 / C + mid <= u) lo = mid;
        else hi = mid - 1;
    }
    bh = lo * a.H + z;
    v = seq_view(a, bh);
    n = u - tile_slot0(a, bh, v);
    return n >= 0 && n * C < v.T;
}

// The chunk's row scalars for the backward (training): gamma_r = e^(b_r) with b the
// chunk-local cumulative log-decay, 1 / gamma_r, beta_r and d log(alpha_r) / dg_r, in
// the full-precision functions of the backward's own decay; rows past the chunk's c
// rows 1, 1, 0, 0.  Warp-wide: lane l holds rows 2 l, 2 l + 1.
__device__ __noinline__ void chunk_row_scalars(int lane, const float (&gv)[2], const float (&bv)[2], int c,
                                               float d, float *blk) {
    const int r0 = 2 * lane;
    const float l0 = (r0 < c) ? log_alpha(gv[0], d) : 0.f;
    const float l1 = (r0 + 1 < c) ? log_alpha(gv[1], d) : 0.f;
    float incl = l0 + l1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float b[2] = {incl - l1, incl};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int r = r0 + e;
        const bool valid = r < c;
        const float ga = valid ? expf(b[e]) : 1.f;
        blk[r] = ga;
        blk[C + r] = 1.0f / ga;
        blk[2 * C + r] = valid ? bv[e] : 0.f;
        blk[3 * C + r] = valid ? decay_dlog_dg(gv[e], d) : 0.f;
    }
}

template <bool kTrain>
__global__ void __launch_bounds__(NT, CTAS_PER_SM)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const FusedArgs a, uint8_t *ws, int BH, int nslot, int items, __nv_bfloat16 *tpb,
                  float *tsc) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    __shared__ __align__(8) uint64_t s_bar[NUM_BARS];
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto bar = [&](int i) { return smem_u32(&s_bar[i]); };
    if (tid == 0) {
        for (int i = 0; i < NUM_BARS; ++i) mbar_init(bar(i), 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), TM_COLS);
        tmem_relinquish();
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_launch_dependents();   // the chain kernel after this one may start its set-up
    const uint32_t tmem = s_tmem;
    const uint32_t idesc_kqk = idesc_bf16(128, 64, false, false);
    float *As = reinterpret_cast<float *>(sm + OFF_AS);
    float *Ys = reinterpret_cast<float *>(sm + OFF_YS);
    uint8_t *tile = sm + OFF_OUT;
    const TileScal S = tile_scal_at(reinterpret_cast<float *>(sm + OFF_SC));
    const int lrow = warp * 32 + lane;           // TMEM lane (quadrant = warp) = accumulator row
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);

    // the CTA's valid items, in order
    auto next_valid = [&](int it, int &bh, int &n, SeqView &v) -> int {
        for (; it < items; it += (int)gridDim.x)
            if (item_chunk(a, BH, nslot, it, bh, n, v)) return it;
        return items;
    };
    // g, beta of a chunk, two rows per lane of warp 3 (loaded an item ahead of their use)
    auto load_gb = [&](int n, const SeqView &v, float (&gv)[2], float (&bv)[2]) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = n * C + 2 * lane + e;
            gv[e] = (t < v.T) ? a.g[v.gbase + (int64_t)t * v.stride] : 0.f;
            bv[e] = (t < v.T) ? a.beta[v.gbase + (int64_t)t * v.stride] : 0.f;
        }
    };
    auto issue = [&](int n, const SeqView &v) {   // thread 0
        const uint32_t buf = sbase + OFF_IN;
        mbar_arrive_expect_tx(bar(B_FULL), IN_BYTES);
        tma_load_3d(buf + 0, &tm_k, bar(B_FULL), 0, v.tz + n * C, v.z);
        tma_load_3d(buf + 8192, &tm_q, bar(B_FULL), 0, v.tz + n * C, v.z);
        tma_load_3d(buf + 16384, &tm_k, bar(B_FULL), 64, v.tz + n * C, v.z);
        tma_load_3d(buf + 24576, &tm_q, bar(B_FULL), 64, v.tz + n * C, v.z);
    };

    int bh, n;
    SeqView v;
    int it = next_valid((int)blockIdx.x, bh, n, v);
    uint32_t loads = 0, products = 0;   // thread 0: TMA loads issued, products issued
    float gv[2] = {0.f, 0.f}, bv[2] = {0.f, 0.f};
    if (tid == 0 && it < items) {
        issue(n, v);
        ++loads;
    }
    if (warp == 3 && it < items) load_gb(n, v, gv, bv);
    for (int cnt = 0; it < items; ++cnt) {
        bool ok = true;
        if (tid == 0) {
            ok = role_wait(bar(B_FULL), (uint32_t)cnt & 1u, a.limit_ns, &s_abort);
            if (ok) {   // [K;Q] K^T: rows 0-63 K K^T, rows 64-127 Q K^T
                tc_fence_after();
                const uint64_t dkq = sdesc_sw128(sbase + OFF_IN, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t d = sdesc_add(dkq, (kk >> 2) * 16384 + (kk & 3) * 32);
                    mma_bf16(tmem, d, d, idesc_kqk, kk > 0);
                }
                mma_commit(bar(B_KQK));
                ++products;
            }
        }
        int bh2, n2;   // the next item, looked up while the product runs
        SeqView v2;
        const int nx = next_valid(it + (int)gridDim.x, bh2, n2, v2);
        if (warp == 3) {   // the chunk's decay (away from the warp that issued the product),
                           // then the next item's g, beta
            warp_decay_tiles(lane, gv[0], gv[1], bv[0], bv[1], min(C, v.T - n * C), a.a_min, S);
            if (kTrain) chunk_row_scalars(lane, gv, bv, min(C, v.T - n * C), a.a_min,
                                       tsc + ((int64_t)bh * (int64_t)nslot + n) * 4 * C);
            if (nx < items) load_gb(n2, v2, gv, bv);
        }
        if (tid == 0 && ok) {
            ok = role_wait(bar(B_KQK), (uint32_t)cnt & 1u, a.limit_ns, &s_abort);
            bulk_wait_read_all();   // the previous tile's store has read the tile buffer
        }
        if (!__syncthreads_and(ok)) break;
        if (tid == 0 && nx < items) {   // K and Q are consumed: the next item's load goes in
            issue(n2, v2);
            ++loads;
        }
        tc_fence_after();
        const int c = min(C, v.T - n * C);
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            // A (rows 0-63) into the solve space, P (rows 64-127) into the tile's second
            // half; this thread: accumulator row lrow, columns 32 half .. 32 half + 31
            float x[32];
            tmem_ld32(tl + half * 32, x);
            tmem_wait_ld();
            if (lrow < 64) {
                const int r = lrow;
                const float br = S.rf[r];                  // zero past the chunk's rows
                const float *cf = S.cf + (r >> 4) * 64;    // this row block's column factors
#pragma unroll
                for (int s4 = 0; s4 < 32; s4 += 4) {
                    const int s0 = half * 32 + s4;
                    const float4 f4 = *reinterpret_cast<const float4 *>(&cf[s0]);
                    float4 o;
                    o.x = (s0 + 0 < r) ? br * x[s4 + 0] * f4.x : 0.f;
                    o.y = (s0 + 1 < r) ? br * x[s4 + 1] * f4.y : 0.f;
                    o.z = (s0 + 2 < r) ? br * x[s4 + 2] * f4.z : 0.f;
                    o.w = (s0 + 3 < r) ? br * x[s4 + 3] * f4.w : 0.f;
                    *reinterpret_cast<float4 *>(&As[r * LDA + s0]) = o;
                }
            } else {
                const int r = lrow - 64;
                const float pr = S.pf[r];                  // zero past the chunk's rows
                const float *cf = S.cf + (r >> 4) * 64;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    float p8[8];
                    const int sb = half * 32 + q4 * 8;
                    const float4 fa = *reinterpret_cast<const float4 *>(&cf[sb]);
                    const float4 fb = *reinterpret_cast<const float4 *>(&cf[sb + 4]);
                    const float f8[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = sb + e;
                        p8[e] = (s <= r) ? pr * x[q4 * 8 + e] * f8[e] : 0.f;
                    }
                    uint4 u;
                    u.x = pack_bf16x2(p8[0], p8[1]);
                    u.y = pack_bf16x2(p8[2], p8[3]);
                    u.z = pack_bf16x2(p8[4], p8[5]);
                    u.w = pack_bf16x2(p8[6], p8[7]);
                    *reinterpret_cast<uint4 *>(tile + LP_TILE_P + swz((uint32_t)r, (uint32_t)(half * 4 + q4))) = u;
                }
            }
        }
        tc_fence_before();
        named_sync(BAR_PREP, NT);
        solve_unit_lower_t<NT>(tid, As, As, Ys);   // T = (I + A)^-1, in place
#pragma unroll 1
        for (int q4 = tid >> 6; q4 < 4; q4 += NT / 64) {
            // Lb = strict_lower(T) diag(beta): row tid % 64, columns 16 q4 + 0..15
            const int r = tid & 63;
            float x[16];
#pragma unroll
            for (int s4 = 0; s4 < 16; s4 += 4) {
                const int s0 = q4 * 16 + s4;
                const float4 t = *reinterpret_cast<const float4 *>(&As[r * LDA + s0]);
                const float4 f = *reinterpret_cast<const float4 *>(&S.bs[s0]);
                x[s4 + 0] = (s0 + 0 < r) ? t.x * f.x : 0.f;
                x[s4 + 1] = (s0 + 1 < r) ? t.y * f.y : 0.f;
                x[s4 + 2] = (s0 + 2 < r) ? t.z * f.z : 0.f;
                x[s4 + 3] = (s0 + 3 < r) ? t.w * f.w : 0.f;
            }
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint4 u;
                u.x = pack_bf16x2(x[h2 * 8 + 0], x[h2 * 8 + 1]);
                u.y = pack_bf16x2(x[h2 * 8 + 2], x[h2 * 8 + 3]);
                u.z = pack_bf16x2(x[h2 * 8 + 4], x[h2 * 8 + 5]);
                u.w = pack_bf16x2(x[h2 * 8 + 6], x[h2 * 8 + 7]);
                *reinterpret_cast<uint4 *>(tile + swz((uint32_t)r, (uint32_t)(q4 * 2 + h2))) = u;
            }
        }
        if (kTrain) {
            // training: T (the unit lower triangle) as bf16 rows with the tile's 128-byte
            // swizzle, each warp store covering four whole rows
            __nv_bfloat16 *tdst = tpb + ((int64_t)bh * nslot + n) * 2 * C * C;
#pragma unroll 1
            for (int x = tid; x < C * 8; x += NT) {
                const int r = x >> 3, c8 = x & 7;
                const float4 t0 = *reinterpret_cast<const float4 *>(&As[r * LDA + 8 * c8]);
                const float4 t1 = *reinterpret_cast<const float4 *>(&As[r * LDA + 8 * c8 + 4]);
                const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
                float m[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) m[e] = (8 * c8 + e <= r) ? tv[e] : 0.f;
                *reinterpret_cast<uint4 *>(tdst + r * C + ((c8 ^ (r & 7)) << 3)) =
                    make_uint4(pack_bf16x2(m[0], m[1]), pack_bf16x2(m[2], m[3]), pack_bf16x2(m[4], m[5]),
                               pack_bf16x2(m[6], m[7]));
            }
        }
        fence_proxy_async_smem();   // the tile leaves by a bulk copy (async proxy)
        __syncthreads();            // every thread is also done with the scalars and A
        if (tid == 0) {
            bulk_store(ws + ((int64_t)v.z * nslot + tile_slot0(a, bh, v) + n) * TILE_BYTES,
                       smem_u32(tile), TILE_BYTES);
            // training: the P half as it is (128-byte rows, 16-byte chunks swizzled by row)
            if (kTrain)
                bulk_store(tpb + (((int64_t)bh * nslot + n) * 2 + 1) * C * C, smem_u32(tile) + LP_TILE_P, 8192);
            bulk_commit();
        }
        it = nx;
        bh = bh2;
        n = n2;
        v = v2;
    }
    if (tid == 0) {
        if (s_abort) {   // let this thread's load and products land before leaving
            if (loads > 0) mbar_wait(bar(B_FULL), (loads - 1) & 1u, kCleanupLimitNs);
            if (products > 0) {
                mma_commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0u, kCleanupLimitNs);
            }
        }
        bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace

// Bytes of workspace the two-kernel path needs: one tile per chunk slot.
size_t prep_workspace_bytes(int BH, int T, const int *cu_seqlens, int H, int total_T) {
    FusedArgs a{};
    a.T = T;
    a.cu_seqlens = cu_seqlens;
    a.H = H;
    a.total_T = total_T;
    if (BH == 0 || (cu_seqlens ? total_T : T) == 0) return 0;
    const int64_t zs = cu_seqlens ? H : BH;
    return (size_t)(zs * tile_slots(a, BH)) * TILE_BYTES;
}

cudaError_t launch_prep(const void *q, const void *k, const float *g, const float *beta, float a_min,
                        void *ws, int BH, int T, const int *cu_seqlens, int H, int total_T,
                        cudaStream_t s, void *tpb, float *tsc) {
    if ((tpb || tsc) && (cu_seqlens || !tpb || !tsc ||
                         ((reinterpret_cast<uintptr_t>(tpb) | reinterpret_cast<uintptr_t>(tsc)) & 15)))
        return cudaErrorInvalidValue;   // the training outputs: dense layout, both, aligned
    if (BH == 0 || (cu_seqlens ? total_T : T) == 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(ws)) & 15)
        return cudaErrorMisalignedAddress;
    CUtensorMap mq, mk;
    const bool ok = cu_seqlens ? (make_map_packed(&mq, q, H, total_T) && make_map_packed(&mk, k, H, total_T))
                               : (make_map(&mq, q, BH, T) && make_map(&mk, k, BH, T));
    if (!ok) return cudaErrorInvalidValue;
    FusedArgs a{g, beta, nullptr, nullptr, nullptr, a_min, T, wait_limit_ns()};
    a.cu_seqlens = cu_seqlens;
    a.H = H;
    a.total_T = total_T;
    const int64_t nslot = tile_slots(a, BH);
    const int64_t items = (cu_seqlens ? (int64_t)H : (int64_t)BH) * nslot;
    if (items > 0x7fffffff) return cudaErrorInvalidValue;   // work items are counted in 32 bits
    const auto kern = tpb ? chunk_prep_kernel<true> : chunk_prep_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(items, (int64_t)sms * CTAS_PER_SM);
    kern<<<(unsigned)grid, NT, SMEM_ALLOC, s>>>(mq, mk, a, static_cast<uint8_t *>(ws), BH, (int)nslot,
                                                (int)items, static_cast<__nv_bfloat16 *>(tpb), tsc);
    return cudaGetLastError();
}

cudaError_t take_prep_error_word(unsigned *value) { return take_error_word(value); }

}  // namespace gdr
