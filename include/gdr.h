/*
 * gdr.h -- C ABI of the GB300 gated delta rule library (libgdr.so).
 *
 * The layer: incremental (delta-rule) linear attention with a lower-bounded
 * decay gate.  For every sequence b and head h the library carries a fixed
 * size state S (dv x dk) through the tokens t = 0..T-1:
 *
 *     alpha_t = a_min + (1 - a_min) * sigmoid(g_t)                 (decay)
 *     S_t     = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t     = S_t q_t
 *
 * Sources.  The update is the "correct-on-write" incremental rule with a
 * position-dependent decay gate of "How to Think About Trillion-Parameter
 * Sparse Multimodal LLMs", section 2.2 (Incremental Linear Attention), whose
 * state is fixed-size so that inference cost does not grow with the context
 * ("Trillion-Parameter MoE Multimodal LLMs: How to Evaluate the New
 * Generation", section 2.1).  The decay floor is the lower-bounded decay of
 * the same page, section 3.1 (and "What a Trillion-Parameter MoE Model Reveals
 * About the Next Stage of LLM Scaling", section 3.2), read in the linear
 * domain: alpha in (a_min, 1], so inside a chunk of C tokens the cumulative
 * decay gamma stays >= a_min^C and its reciprocal <= a_min^-C.  That bound is
 * what lets every causal tile of the chunked form -- the diagonal (intra-
 * chunk) one included -- run as one dense tensor-core product ("Architecture
 * Evolution and Training Engineering for Trillion-Scale Sparse Multimodal
 * Models", section 3.2).
 *
 * Conventions for every entry point below
 *   - All array pointers are caller-owned DEVICE memory, contiguous,
 *     row-major, in the layouts given.  The library keeps no pointer after a
 *     call returns.
 *   - The state is fp32 [.., dk, dv] and holds M = S^T (M[i][j] = S[j][i]),
 *     the same layout for prefill and decode, so a prefill's final state
 *     feeds decode directly.
 *   - g, beta are fp32.  q, k, v and out are all of `dtype`.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued asynchronously on it; no call synchronises except
 *     gdr_last_device_error.
 *   - Argument errors are reported synchronously, before anything is
 *     enqueued.  A failed launch returns GDR_ERR_CUDA.  Kernels never trap:
 *     a bounded wait that runs out records GDR_ERR_TIMEOUT in a device error
 *     word, read by gdr_last_device_error.  No C++ exception crosses this ABI.
 *   - Supported shapes: dk, dv in {16, 32, 64, 128}; chunk in {16, 32, 64};
 *     any T >= 0 (a ragged last chunk is masked).  Others: GDR_ERR_UNSUPPORTED.
 *   - Range rule: chunk * (-ln a_min) must not exceed 80, the worst in-tile
 *     cumulative log-decay the pages' range argument allows (section 3.1 of
 *     the first page above); otherwise GDR_ERR_RANGE.  The two-kernel
 *     workspace path below applies it over a 16-token tile instead of the
 *     chunk: 16 * (-ln a_min) <= 80.  a_min must lie in (0, 1]:
 *     GDR_ERR_INVALID_ARG otherwise.
 */
#ifndef GDR_H
#define GDR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDR_OK = 0,
    GDR_ERR_INVALID_ARG = 1,  /* null pointer, negative size, a_min out of (0,1] */
    GDR_ERR_UNSUPPORTED = 2,  /* shape or dtype this build does not implement   */
    GDR_ERR_RANGE = 3,        /* chunk (or tile) * (-ln a_min) > 80              */
    GDR_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed            */
    GDR_ERR_TIMEOUT = 5       /* a device-side bounded wait gave up              */
} gdr_status_t;

typedef enum {
    GDR_DTYPE_F32 = 0,        /* q, k, v, out are float                          */
    GDR_DTYPE_BF16 = 1        /* q, k, v, out are bfloat16 (round-to-nearest-even
                                 on the output store)                            */
} gdr_dtype_t;

/*
 * Chunked prefill over B sequences x H heads x T tokens.
 *   q, k        [B,H,T,dk]  dtype
 *   v           [B,H,T,dv]  dtype
 *   g, beta     [B,H,T]     fp32: raw decay logit, write strength
 *   a_min       decay floor, 0 < a_min <= 1
 *   init_state  [B,H,dk,dv] fp32, or NULL for a zero state
 *   out         [B,H,T,dv]  dtype
 *   final_state [B,H,dk,dv] fp32, or NULL to skip; may alias init_state
 *   chunk       tile length C of the chunked form
 * Work: the chunked form of the recurrence (per chunk: cumulative decay, the
 * intra-chunk WY/UT transform, the inter-chunk state step and the output),
 * which equals the token recurrence in exact arithmetic.
 * One launch, and the library allocates nothing: bf16 with dk = dv = 128 and
 * chunk = 64 runs a fused tensor-core kernel; fp32 and every other shape run
 * one CUDA-core kernel (one CTA per head and block of 32 value columns, walking
 * the chunks in order, every intermediate in shared memory).  With a
 * caller-owned workspace, gdr_chunk_fwd_ws runs faster multi-kernel paths.
 * T == 0 copies init_state (or zeros) to final_state.
 */
gdr_status_t gdr_chunk_fwd(const void *q, const void *k, const void *v,
                           const float *g, const float *beta, float a_min,
                           const float *init_state, void *out, float *final_state,
                           int B, int H, int T, int dk, int dv, int chunk,
                           gdr_dtype_t dtype, void *stream);

/*
 * One token per sequence: N sequences x H heads, state updated in place.
 * This is the inference step the fixed-size state exists for: the state does
 * not grow with the context, so a token costs one read and one write of it
 * however long the sequence already is ("Trillion-Parameter MoE Multimodal
 * LLMs: How to Evaluate the New Generation", section 2.1; the incremental
 * correct-on-write update of "How to Think About Trillion-Parameter Sparse
 * Multimodal LLMs", section 2.2).
 *   q, k [N,H,dk] dtype; v [N,H,dv] dtype; g, beta [N,H] fp32;
 *   state [N,H,dk,dv] fp32 (in/out, the M = S^T layout of the prefill's final
 *   state); out [N,H,dv] dtype.
 * Work: p = S k and r = S q in one pass over the state, u = v - alpha p,
 * o = alpha r + beta (q.k) u, S <- alpha S + beta u k^T (the same recurrence
 * with T = 1).  state must not alias q, k, v or out.  One launch; allocates
 * nothing.  Errors: N or H negative, a_min outside (0, 1] or a null pointer
 * (N H > 0): GDR_ERR_INVALID_ARG; dk or dv outside {16, 32, 64, 128}:
 * GDR_ERR_UNSUPPORTED.
 */
gdr_status_t gdr_decode_step(const void *q, const void *k, const void *v,
                             const float *g, const float *beta, float a_min,
                             float *state, void *out, int N, int H, int dk, int dv,
                             gdr_dtype_t dtype, void *stream);

/* ---- the staged steps of the chunked form (what gdr_chunk_fwd_ws runs, on
 *      its workspace, for fp32 and for shapes the tensor-core kernels do not
 *      cover), exposed so each step can be checked on its own.  BH = B * H;
 *      NC = ceil(T / chunk). ---- */

/*
 * Step 1, cumulative decay inside each chunk (the Gamma = exp(cumsum(log
 * decay)) of "Architecture Evolution and Training Engineering for
 * Trillion-Scale Sparse Multimodal Models", section 3.2):
 *   gamma[bh][t] = prod_{s = chunk start .. t} alpha_s,   fp32 [BH,T].
 * a_min^(r) <= gamma <= 1 for the r-th row of a chunk, so 1/gamma is finite.
 */
gdr_status_t gdr_chunk_decay(const float *g, float a_min, float *gamma,
                             int BH, int T, int chunk, void *stream);

/*
 * Step 2, intra-chunk WY/UT transform, per chunk (rows r, s of the chunk):
 *   A  = strict_lower(diag(beta*gamma) K (diag(1/gamma) K)^T),  T = (I + A)^-1
 *   U  = T diag(beta) V           -> U  fp32 [BH,T,dv]
 *   Wk = T diag(beta*gamma) K     -> Wk fp32 [BH,T,dk]
 * k [BH,T,dk], v [BH,T,dv] in dtype; beta, gamma fp32 [BH,T].
 */
gdr_status_t gdr_chunk_wy(const void *k, const void *v, const float *beta,
                          const float *gamma, float *U, float *Wk,
                          int BH, int T, int dk, int dv, int chunk,
                          gdr_dtype_t dtype, void *stream);

/*
 * Step 3, inter-chunk state pass, sequential over chunks n:
 *   W_n = U_n - Wk_n M_n;   M_{n+1} = gamma_C M_n + (diag(gamma_C/gamma) K_n)^T W_n
 * Writes W fp32 [BH,T,dv], the state at every chunk start Mn fp32
 * [BH,NC,dk,dv] (may be NULL) and final_state (may be NULL).
 * init_state may be NULL (zeros).
 */
gdr_status_t gdr_chunk_state(const void *k, const float *gamma, const float *U,
                             const float *Wk, const float *init_state, float *W,
                             float *Mn, float *final_state,
                             int BH, int T, int dk, int dv, int chunk,
                             gdr_dtype_t dtype, void *stream);

/*
 * Step 4, output of every chunk (intra-chunk causal tile plus state term):
 *   O_n = diag(gamma) Q M_n + lower_incl(diag(gamma) Q (diag(1/gamma) K)^T) W_n
 * q, k in dtype; gamma fp32 [BH,T]; Mn fp32 [BH,NC,dk,dv]; W fp32 [BH,T,dv];
 * out [BH,T,dv] in dtype.
 */
gdr_status_t gdr_chunk_output(const void *q, const void *k, const float *gamma,
                              const float *Mn, const float *W, void *out,
                              int BH, int T, int dk, int dv, int chunk,
                              gdr_dtype_t dtype, void *stream);

/*
 * Chunked prefill that allocates no device memory.  The pages have no
 * counterpart to this entry point; it exists for callers that must not
 * allocate while they run -- for example a plugin inside a framework that owns
 * all device memory through its own pool, or a deployment that forbids
 * allocation after start-up because it can stall or fail mid-stream.
 *
 * Same arguments, layouts and results as gdr_chunk_fwd, computed by the
 * staged kernels (steps 1-4 below) for every dtype and shape.  Their
 * intermediates live in a fixed 32 MiB device array inside the library,
 * which every GPU that loads the library holds until the process exits.
 *   - Size limit: 4 * (B*H*T*(1 + dk + 2*dv) + B*H*ceil(T/chunk)*dk*dv) bytes
 *     must not exceed 32 MiB (33554432); larger work returns
 *     GDR_ERR_UNSUPPORTED before anything is enqueued.
 *   - The array's device address depends on the CUDA context the library is
 *     loaded in (another context on the device, or the primary context made
 *     again after cudaDeviceReset, may place it elsewhere).  The first call in
 *     each context, on a thread where that context is current, looks the
 *     address up (cudaGetSymbolAddress) and caches it under the context's
 *     unique ID; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents
 *     (every value is rewritten before it is read, so nothing needs
 *     clearing).  Calls whose work overlaps on the GPU -- on different
 *     streams, or from different threads -- race on it: order them.
 */
gdr_status_t gdr_chunk_fwd_static(const void *q, const void *k, const void *v,
                                  const float *g, const float *beta, float a_min,
                                  const float *init_state, void *out, float *final_state,
                                  int B, int H, int T, int dk, int dv, int chunk,
                                  gdr_dtype_t dtype, void *stream);

/*
 * Chunked prefill over packed variable-length sequences (the serving shape:
 * the prompts of several requests in one launch, no padding).  Same method,
 * per sequence and head, as gdr_chunk_fwd.
 *
 * q, k, v  dtype [total_T][H][dk | dv], row-major, token-major: the tokens of
 *          sequence s are cu_seqlens[s] .. cu_seqlens[s+1] - 1.
 * g, beta  fp32 [total_T][H].
 * out      dtype [total_T][H][dv].
 * init_state, final_state  fp32 [S][H][dk][dv] (init may be NULL = zeros,
 *          final may be NULL; they may alias).  The final states are directly
 *          the decode states of gdr_decode_step with N = S.
 * cu_seqlens  DEVICE int32 [S + 1], nondecreasing, cu_seqlens[0] = 0,
 *          cu_seqlens[S] = total_T.  Read by the kernel; not checked on the host
 *          (that would need a copy).  Offsets outside [0, total_T] are clamped, so
 *          a malformed array gives wrong results but no out-of-bounds access.
 *          An empty sequence gets final = init.
 * Every shape and dtype of gdr_chunk_fwd: bf16 with dk = dv = 128 and chunk =
 * 64 on the fused tensor-core kernels (and on the two-kernel path of
 * gdr_chunk_fwd_varlen_ws), fp32 and the other shapes on the one-pass CUDA-core
 * kernel (one CTA per sequence, head and 32 value columns).  One launch, no
 * allocation.  Errors as gdr_chunk_fwd.
 */
gdr_status_t gdr_chunk_fwd_varlen(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, float a_min, const float *init_state,
                                  void *out, float *final_state, const int *cu_seqlens, int S,
                                  int H, int total_T, int dk, int dv, int chunk,
                                  gdr_dtype_t dtype, void *stream);

/*
 * Number of kernel launches one gdr_chunk_fwd call with these arguments
 * enqueues (1 on the fused path, 4 on the staged path, 0 for empty work), or
 * -1 if the call would be rejected.  Host-only; touches no device.
 */
int gdr_chunk_fwd_kernels(int B, int H, int T, int dk, int dv, int chunk, float a_min,
                          gdr_dtype_t dtype);

/*
 * Which code path one gdr_chunk_fwd call with these arguments takes on the
 * calling thread's current device: 0 no kernel (empty work), 2 the fused kernel
 * with one CTA per head, 3 the fused kernel with a cluster of two CTAs per head
 * (value columns split, chunk preparation alternated between the two), 6 the
 * one-pass CUDA-core kernel (fp32 and the other shapes), or -1 if the call
 * would be rejected.  The choice between 2 and 3 depends on how many two-CTA
 * clusters the device holds at once (queried once per process) and on the
 * GDR_OPT_FUSED_VARIANT option.  Launches nothing.
 */
int gdr_chunk_fwd_path(int B, int H, int T, int dk, int dv, int chunk, float a_min,
                       gdr_dtype_t dtype);

/*
 * The two-kernel prefill: a caller-owned workspace lets the preparation of
 * every chunk -- [K;Q]K^T, A, the triangular solve T = (I + A)^-1, Lb =
 * strict_lower(T) diag(beta) and P = lower_incl(D o Q K^T) with D[r][s] =
 * gamma_r / gamma_s ("What a Trillion-Parameter MoE Model Reveals About the
 * Next Stage of LLM Scaling", sections 3.1-3.3) -- run as one fully parallel
 * kernel that writes a 16 KB bf16 tile per chunk, so that the second kernel,
 * the sequential state chain with the outputs, does nothing else.  Same
 * method and results as gdr_chunk_fwd, within the bf16 tolerance.  The
 * preparation applies D as the diagonal scalings of the pages' 16-token tiles
 * (reference points every 16 rows) and the chain uses only factors at most 1,
 * so this path's range rule is 16 * (-ln a_min) <= 80 (a_min >= e^-5) or
 * 16 * (-g_min) <= 80 (g_min >= -5): the decay over a 64-token chunk may fall
 * far below fp32's range.
 *
 * gdr_chunk_fwd_workspace_size: bytes of workspace gdr_chunk_fwd_ws uses for
 *   these arguments, or 0 for empty work or unsupported arguments.  Host-only.
 *   bf16 with dk = dv = 128 and chunk = 64: the two-kernel path (B * H *
 *   ceil(T / 64) tiles of 16 KB; with S > 1 sequence segments also
 *   B * H * (3 S - 2) fp32 128 x 128 maps: each segment's offset and
 *   transition, and its first state).  fp32 and the other shapes: the four staged
 *   kernels (gdr_chunk_decay .. gdr_chunk_output) with their intermediates in
 *   the workspace, 4 * (B*H*T*(1 + dk + 2*dv) + B*H*ceil(T/chunk)*dk*dv) bytes;
 *   their WY/UT and output steps run every chunk in parallel, so they beat the
 *   one-pass kernel of gdr_chunk_fwd on long sequences.
 * gdr_chunk_fwd_ws: gdr_chunk_fwd with a workspace.  `workspace` is device
 *   memory owned by the caller, 16-byte aligned, at least the size above, not
 *   shared with a call still running on another stream; its contents on entry
 *   and exit are scratch.  With a null workspace, one that is too small, or
 *   arguments the two-kernel path does not take, the call is exactly
 *   gdr_chunk_fwd (the single-launch fused or staged path, with its chunk
 *   range rule).  Two launches (four with sequence segments), asynchronous on
 *   `stream`; errors as gdr_chunk_fwd.
 * gdr_chunk_fwd_varlen_workspace_size / gdr_chunk_fwd_varlen_ws: the same for
 *   packed sequences; the workspace holds H * (total_T / 64 + S + 1) tiles
 *   (sequence s starts at tile total offset cu_seqlens[s] / 64 + s of its head);
 *   the size is 0 (no workspace needed) for fp32 and the other shapes, which
 *   gdr_chunk_fwd_varlen runs on the one-pass kernel.
 * gdr_chunk_fwd_ws_path: the path gdr_chunk_fwd_ws takes given a large enough
 *   workspace: 1 the staged kernels, 4 two kernels with two CTAs per head in
 *   the chain kernel (value columns split), 5 two kernels with one CTA per
 *   head, 7 the two kernels over sequence segments (few heads, long
 *   sequences: every segment's state map and offset in parallel, a scan over
 *   the segments, then the chain over every (head, segment) at once; exact,
 *   the maps compose), else the value of gdr_chunk_fwd_path.  The split is
 *   two CTAs per head while every CTA has an SM of its own; the
 *   GDR_OPT_CHAIN_SPLIT option forces one.  Launches nothing.
 */
size_t gdr_chunk_fwd_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                    gdr_dtype_t dtype);
gdr_status_t gdr_chunk_fwd_ws(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, float a_min, const float *init_state, void *out,
                              float *final_state, int B, int H, int T, int dk, int dv, int chunk,
                              gdr_dtype_t dtype, void *workspace, size_t workspace_bytes,
                              void *stream);
size_t gdr_chunk_fwd_varlen_workspace_size(int S, int H, int total_T, int dk, int dv, int chunk,
                                           gdr_dtype_t dtype);
gdr_status_t gdr_chunk_fwd_varlen_ws(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, float a_min, const float *init_state,
                                     void *out, float *final_state, const int *cu_seqlens, int S,
                                     int H, int total_T, int dk, int dv, int chunk,
                                     gdr_dtype_t dtype, void *workspace, size_t workspace_bytes,
                                     void *stream);
int gdr_chunk_fwd_ws_path(int B, int H, int T, int dk, int dv, int chunk, float a_min,
                          gdr_dtype_t dtype);

/*
 * The prefill from host memory to host memory: the call a host-side caller makes
 * when its q, k, v, g, beta (and initial state) are in host memory and it wants the
 * output (and final state) back there.  On `stream`, in order: the host-to-device
 * copies of the inputs into `device_buffer`, the prefill of gdr_chunk_fwd_ws (the
 * two-kernel path when it applies, the buffer holding its workspace), and the
 * device-to-host copies of out and final_state.  Asynchronous: the host inputs must
 * stay unchanged and the host outputs untouched until `stream` reaches the end of
 * the call.  Page-locked host memory lets the copies overlap other streams' work
 * (two calls on two streams with two device buffers overlap one's copies with the
 * other's kernels); pageable memory works but the copies are staged by the driver.
 *
 * Pointers: q, k, v, g, beta, init_state (may be NULL), out, final_state (may be
 * NULL) are HOST pointers with the layouts of gdr_chunk_fwd.  device_buffer: device
 * memory owned by the caller, 256-byte aligned, at least
 * gdr_chunk_fwd_host_buffer_size bytes, not shared with a call still running on
 * another stream.  Errors as gdr_chunk_fwd (a_min in (0, 1]; the range rule of the
 * path taken: over a 16-token tile on the two-kernel path, over the chunk
 * elsewhere); a missing or small buffer is GDR_ERR_INVALID_ARG.
 */
size_t gdr_chunk_fwd_host_buffer_size(int B, int H, int T, int dk, int dv, int chunk,
                                      gdr_dtype_t dtype);
gdr_status_t gdr_chunk_fwd_host(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float a_min, const float *init_state,
                                void *out, float *final_state, int B, int H, int T, int dk, int dv,
                                int chunk, gdr_dtype_t dtype, void *device_buffer,
                                size_t device_bytes, void *stream);

/*
 * The two lower-bounded decays ("Trillion-Parameter MoE Multimodal LLMs: How to
 * Evaluate the New Generation", section 3.1; "What a Trillion-Parameter MoE Model
 * Reveals About the Next Stage of LLM Scaling", section 3.2):
 *   GDR_DECAY_AFFINE: alpha = a_min + (1 - a_min) sigmoid(g), bound = a_min in (0, 1]
 *                     (the decay of every other entry point);
 *   GDR_DECAY_LOG:    log alpha = g_min sigmoid(g), bound = g_min <= 0 (the pages'
 *                     own form; g_min = -5 with 16-token chunks is their setting).
 * The range rule applies to both: chunk * (-ln a_min) or chunk * (-g_min) must not
 * exceed 80 (GDR_ERR_RANGE otherwise), over a 16-token tile on the two-kernel
 * workspace path.  So the pages' setting g_min = -5 runs on the two-kernel path
 * (bf16, d = 128, chunk 64, with a workspace) or with chunk 16 on the staged
 * kernels; the single-launch fused kernels take g_min >= -1.25.
 *
 * gdr_chunk_fwd_ex: gdr_chunk_fwd_ws with the decay chosen by (decay, bound);
 *   workspace may be NULL (the single-launch or staged path).
 * gdr_decode_step_ex: gdr_decode_step with the decay chosen by (decay, bound).
 * An unknown mode or a bound outside its range returns GDR_ERR_INVALID_ARG.
 */
typedef enum { GDR_DECAY_AFFINE = 0, GDR_DECAY_LOG = 1 } gdr_decay_t;
gdr_status_t gdr_chunk_fwd_ex(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, gdr_decay_t decay, float bound,
                              const float *init_state, void *out, float *final_state, int B,
                              int H, int T, int dk, int dv, int chunk, gdr_dtype_t dtype,
                              void *workspace, size_t workspace_bytes, void *stream);
gdr_status_t gdr_decode_step_ex(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, gdr_decay_t decay, float bound, float *state,
                                void *out, int N, int H, int dk, int dv, gdr_dtype_t dtype,
                                void *stream);

/*
 * Backward of the chunked prefill: the gradients of a loss L with respect to
 * every input of gdr_chunk_fwd, given dL/dout and dL/dfinal_state (the chain
 * rule through the same chunk algebra, "What a Trillion-Parameter MoE Model
 * Reveals About the Next Stage of LLM Scaling", sections 3.1-3.3, taken in
 * reverse).  The forward's intermediates (the decay, the W tiles and the state
 * at every chunk start) are recomputed from the inputs, then one sequential
 * reverse pass over the chunks carries dL/dM, and one fully parallel pass
 * forms every chunk's gradients.  fp32 arithmetic throughout, except for bf16
 * with dk = dv = 128, chunk 64 and 16-byte aligned d_q, d_k, d_v: there the
 * products run on tensor cores with bf16 operands and fp32 accumulation, and
 * the intermediates come from gdr_chunk_fwd_train's kernels run into the
 * workspace, followed by gdr_chunk_bwd_saved's (four launches; six with the
 * sequence segments of few heads); the gradients measure ~3e-3 relative L2
 * against an fp64 reference.  GDR_OPT_BWD_VARIANT 1 or 2 recompute them with
 * the backward's own tiles kernel and forward-state pass instead (near-fp32
 * states through split-bf16 operands, d_init ~2e-3; five launches).  Other
 * shapes and fp32 stay on the fp32 kernels (~3e-7).
 *
 * q, k, v, g, beta, (decay, bound), init_state: as gdr_chunk_fwd_ex (the
 *          forward whose gradients are taken; init_state may be NULL = zeros).
 * d_out    [B,H,T,dv] in dtype: dL/dout (required when T > 0).
 * d_final  fp32 [B,H,dk,dv] (M layout) or NULL (zero): dL/dfinal_state.
 * d_q, d_k [B,H,T,dk] and d_v [B,H,T,dv] in dtype; d_g, d_beta fp32 [B,H,T];
 * d_init   fp32 [B,H,dk,dv] or NULL (not wanted): the gradients.  Every output
 *          is overwritten (no accumulation into existing values).
 * workspace  device memory of at least gdr_chunk_bwd_workspace_size bytes,
 *          16-byte aligned, owned by the caller; scratch on entry and exit.
 * q, k, v and d_out must be 16-byte aligned (GDR_ERR_INVALID_ARG otherwise).
 * Supported: dk in {32, 64, 128}, dv in {16, 32, 64, 128}, chunk in {16, 32,
 * 64}, fp32 or bf16 (GDR_ERR_UNSUPPORTED otherwise); the range rule over the
 * chunk (GDR_ERR_RANGE).  Four or five launches, asynchronous on `stream`.
 * gdr_chunk_bwd_workspace_size returns 0 for unsupported arguments or empty
 * work (T = 0 needs no workspace: d_init = d_final, or zeros).
 */
size_t gdr_chunk_bwd_workspace_size(int B, int H, int T, int dk, int dv, int chunk,
                                    gdr_dtype_t dtype);
gdr_status_t gdr_chunk_bwd(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, gdr_decay_t decay, float bound,
                           const float *init_state, const void *d_out, const float *d_final,
                           void *d_q, void *d_k, void *d_v, float *d_g, float *d_beta,
                           float *d_init, int B, int H, int T, int dk, int dv, int chunk,
                           gdr_dtype_t dtype, void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * Training: a forward that keeps what its backward needs.  The chain of the
 * two-kernel path already forms, chunk by chunk, the state M_n at every chunk
 * start and the tile W_n = T diag(beta) E of the chunk ("What a Trillion-Parameter
 * MoE Model Reveals About the Next Stage of LLM Scaling", sections 3.2-3.3), and
 * its per-chunk kernel the triangular inverse T = (I + A)^-1, the masked decayed
 * scores P and the cumulative decay; the backward of gdr_chunk_bwd recomputes all
 * of them from the inputs.  gdr_chunk_fwd_train writes them out as it goes, and
 * gdr_chunk_bwd_saved reads them instead of recomputing: no forward-state pass,
 * no decay or per-chunk tile kernel in the backward.
 *
 * Shape: bf16, dk = dv = 128, chunk 64 (GDR_ERR_UNSUPPORTED otherwise), dense
 * [B,H,T,d] tensors.
 *
 * gdr_chunk_saved_size: bytes of the saved buffer, B * H * ceil(T / 64) * 66560,
 *   four regions each over (b, h, chunk n) in that order: the states M_n
 *   transposed (bf16 [128 value rows][128 key columns]); the tiles W_n
 *   transposed (bf16 [128 value rows][64 chunk positions], zero past T); T_n and
 *   P_n (bf16 [64][64] each, T first; past T the rows of T are the identity's and
 *   those of P zero; their 128-byte rows hold the 16-byte chunks swizzled, chunk c
 *   of row r at byte 128 r + 16 (c XOR (r mod 8))); the row scalars (fp32 [4][64]: gamma_r, 1 / gamma_r, beta_r,
 *   d log(alpha_r) / d g_r; 1, 1, 0, 0 past T).  0 for unsupported arguments or
 *   empty work.  Host-only.
 * gdr_chunk_fwd_train: gdr_chunk_fwd_ex on the two-kernel path (sequence
 *   segments included) that also fills `saved`.  The workspace is required (at
 *   least gdr_chunk_fwd_workspace_size bytes) and so is `saved` (device memory
 *   owned by the caller, 16-byte aligned, at least gdr_chunk_saved_size bytes):
 *   GDR_ERR_INVALID_ARG when either is missing, small or misaligned.  The range
 *   rule is over the 16-token tile as on the two-kernel path.  Two to four
 *   launches, asynchronous on `stream`; out and final_state as gdr_chunk_fwd.
 * gdr_chunk_bwd_saved: gdr_chunk_bwd given the saved buffer of the forward with
 *   the same q, k, v, g, beta, decay, bound, init_state and sizes (not checked:
 *   another forward's buffer gives wrong gradients, not an error).  `saved` is
 *   read only and may be released once `stream` has passed the call.  d_q, d_k,
 *   d_v must be 16-byte aligned as well (GDR_ERR_INVALID_ARG otherwise); the
 *   workspace is gdr_chunk_bwd_workspace_size bytes; the range rule over the
 *   chunk as gdr_chunk_bwd.  Two launches.  The states are the forward's bf16
 *   operands, so the gradients differ from gdr_chunk_bwd's by about the bf16
 *   rounding of the states (both ~3e-3 relative L2 against an fp64 reference).
 *   B * H = 0 or T = 0 is gdr_chunk_bwd.
 */
size_t gdr_chunk_saved_size(int B, int H, int T, int dk, int dv, int chunk, gdr_dtype_t dtype);
gdr_status_t gdr_chunk_fwd_train(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, gdr_decay_t decay, float bound,
                                 const float *init_state, void *out, float *final_state, int B,
                                 int H, int T, int dk, int dv, int chunk, gdr_dtype_t dtype,
                                 void *workspace, size_t workspace_bytes, void *saved,
                                 size_t saved_bytes, void *stream);
gdr_status_t gdr_chunk_bwd_saved(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, gdr_decay_t decay, float bound,
                                 const float *init_state, const void *d_out, const float *d_final,
                                 void *d_q, void *d_k, void *d_v, float *d_g, float *d_beta,
                                 float *d_init, int B, int H, int T, int dk, int dv, int chunk,
                                 gdr_dtype_t dtype, const void *saved, size_t saved_bytes,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * One decode step of gated multi-head latent attention, the exact-attention
 * layer the pages interleave with the linear attention: the key/value
 * projections are compressed into a latent space so the cache holds one latent
 * vector per token, exact softmax attention keeps precise retrieval, and a gate
 * is added ("Trillion-Parameter MoE Multimodal LLMs: How to Evaluate the New
 * Generation", section 2.1; "How to Think About Trillion-Parameter Sparse
 * Multimodal LLMs", section 2.3).  With the key up-projection absorbed into the
 * query (q_abs = W_uk,h^T q_h), per sequence n and head h:
 *   s_t = scale * q_abs[n,h] . ckv[n,t]            for t < seqlens[n]
 *   o   = w_uv[h] * sum_t softmax(s)_t ckv[n,t]     (dh values)
 *   out[n,h] = sigmoid(gate[n,h]) * o              (elementwise)
 * A sequence of length 0 gives a zero output.
 *
 *   q_abs   bf16 [N,H,dc]      the absorbed queries
 *   ckv     bf16 [N,Lmax,dc]   the latent cache (rows at and past seqlens[n] are
 *                              never used, whatever they hold)
 *   seqlens DEVICE int32 [N]   cache rows in use, clamped into [0, Lmax]
 *   w_uv    bf16 [H,dh,dc]     the value up-projection
 *   gate    fp32 [N,H,dh]      the gate's pre-activation
 *   scale   score scale, > 0 (typically 1/sqrt(dh))
 *   out     bf16 [N,H,dh]
 *   workspace  device memory owned by the caller, 16-byte aligned, of at least
 *           gdr_mla_decode_workspace_size bytes (each split of a sequence's cache
 *           leaves its unnormalised partial result there); scratch on entry and exit.
 * Supported: dc = 512, H a multiple of 64, dh a multiple of 4 up to 1024
 * (GDR_ERR_UNSUPPORTED otherwise).  q_abs, ckv and w_uv must be 16-byte aligned
 * (GDR_ERR_INVALID_ARG).  Two launches: the split attention on tensor cores,
 * then the merge of the splits with the up-projection and the gate.
 * gdr_mla_decode_workspace_size returns 0 for unsupported arguments.
 */
size_t gdr_mla_decode_workspace_size(int N, int H, int Lmax, int dc, int dh);
gdr_status_t gdr_mla_decode(const void *q_abs, const void *ckv, const int *seqlens,
                            const void *w_uv, const float *gate, float scale, void *out, int N,
                            int H, int Lmax, int dc, int dh, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * Process-wide options, for tests and tuning.  Each takes effect for calls made
 * after it is set, on every thread; the defaults suit production use.
 *   GDR_OPT_WAIT_LIMIT_NS  bound of every device-side wait, in ns (default
 *                          2e9).  0 makes every wait give up at once: the
 *                          kernels unwind and gdr_last_device_error reports
 *                          GDR_ERR_TIMEOUT, which drives the error path without
 *                          a GPU fault.
 *   GDR_OPT_FUSED_VARIANT  the single-launch bf16 kernel: 0 chosen by head count
 *                          (default), 1 one CTA per head, 2 cluster pair.
 *   GDR_OPT_CHAIN_SPLIT    CTAs per head in the chain kernel of the two-kernel
 *                          path: 0 chosen by head count (default), 1 or 2.
 *   GDR_OPT_SEGMENTS       sequence segments of the two-kernel path: 0 chosen by
 *                          a cost model of the heads, the sequence length and the
 *                          SM count (default), else that many (at most 4096).
 *   GDR_OPT_BWD_VARIANT    the bf16 d = 128 chunk-64 backward: 0 default (the
 *                          training forward's kernels recompute the intermediates,
 *                          per-chunk gradients on tensor cores), 1 the backward's own
 *                          recomputation with the warp-level-MMA per-chunk kernel,
 *                          2 the same with the tensor-core per-chunk kernel.
 * gdr_set_option returns GDR_ERR_INVALID_ARG for an unknown option or a value
 * out of its range; gdr_get_option returns the current value (-1 if unknown).
 * The library reads no environment variable.
 */
typedef enum {
    GDR_OPT_WAIT_LIMIT_NS = 0,
    GDR_OPT_FUSED_VARIANT = 1,
    GDR_OPT_CHAIN_SPLIT = 2,
    GDR_OPT_SEGMENTS = 3,
    GDR_OPT_BWD_VARIANT = 4
} gdr_option_t;
gdr_status_t gdr_set_option(gdr_option_t option, int64_t value);
int64_t gdr_get_option(gdr_option_t option);

/*
 * Synchronises `stream`, then returns and clears the device error word:
 * GDR_ERR_TIMEOUT if a kernel's bounded wait gave up since the last call,
 * GDR_ERR_CUDA if the stream reports an error, else GDR_OK.
 */
gdr_status_t gdr_last_device_error(void *stream);

/* Static, NUL-terminated description of a status code. */
const char *gdr_status_string(gdr_status_t status);

/* Library version string, e.g. "gdr 0.1.0 sm_103a". */
const char *gdr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H */
