// gdr_internal.h -- launchers shared between the C-ABI layer and the kernel
// translation units of libgdr.so.  Not installed; the public surface is
// include/gdr.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace gdr {

// Element type of q, k, v and out.
enum class Elem { F32 = 0, BF16 = 1 };

// ---- staged chunked form (gdr_staged.cu) ----
cudaError_t launch_decay(const float *g, float a_min, float *gamma, int BH, int T, int C,
                         cudaStream_t s);
cudaError_t launch_wy(const void *k, const void *v, const float *beta, const float *gamma,
                      float *U, float *Wk, int BH, int T, int dk, int dv, int C, Elem e,
                      cudaStream_t s);
cudaError_t launch_state(const void *k, const float *gamma, const float *U, const float *Wk,
                         const float *init, float *W, float *Mn, float *final_state, int BH,
                         int T, int dk, int dv, int C, Elem e, cudaStream_t s);
cudaError_t launch_output(const void *q, const void *k, const float *gamma, const float *Mn,
                          const float *W, void *out, int BH, int T, int dk, int dv, int C,
                          Elem e, cudaStream_t s);
// final_state <- init (or zeros) for T == 0.
cudaError_t launch_copy_state(const float *init, float *final_state, int64_t n, cudaStream_t s);
// Bytes of fp32 intermediates the four staged steps need for one prefill:
// gamma, U, Wk, W per token-head and the state at every chunk start.
size_t staged_scratch_bytes(int64_t BH, int T, int dk, int dv, int C);
// The whole prefill as the four staged steps on caller-provided scratch of at
// least staged_scratch_bytes (16-byte aligned); every value in it is written
// before it is read.
cudaError_t launch_staged(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float d, const float *init, void *out,
                          float *final_state, void *scratch, int BH, int T, int dk, int dv,
                          int C, Elem e, cudaStream_t s);

// ---- the prefill in one CUDA-core launch with no scratch (gdr_onepass.cu):
// fp32, and every shape the tensor-core kernels do not take ----
// cu_seqlens != nullptr: packed sequences (BH = S H states, tokens [total_T][H], as
// gdr_chunk_fwd_varlen; T unused).
cudaError_t launch_onepass(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float d, const float *init, void *out,
                           float *final_state, int BH, int T, int dk, int dv, int C, Elem e,
                           cudaStream_t s, const int *cu_seqlens = nullptr, int H = 0,
                           int total_T = 0);

// ---- process-wide options (gdr_set_option in gdr_api.cu) ----
// Bound of every device-side wait in ns (0: every wait gives up at once, the
// fault-injection setting of the tests).
uint64_t opt_wait_limit_ns();
// Single-launch fused kernel: 0 by head count, 1 one CTA per head, 2 cluster pair.
int opt_fused_variant();
// CTAs per head of the chain kernel: 0 by head count, else 1 or 2.
int opt_chain_split();
// Sequence segments of the two-kernel path: 0 by head count, else that many (at
// most the sequence's chunk count).
int opt_segments();
int opt_bwd_variant();

// ---- backward of the chunked form (gdr_bwd.cu) ----
bool bwd_supported(int dk, int dv, int C);
size_t bwd_workspace_bytes(int BH, int T, int dk, int dv, int C);
// The part of that workspace the saved-state backward (launch_bwd with `saved`) leaves
// untouched: [offset, offset + bytes), 16-byte aligned.
void bwd_free_region(int BH, int T, int dk, int dv, int C, size_t *offset, size_t *bytes);
// saved != nullptr: the states and W^T saved by the forward (launch_chain's saved
// buffer); the forward-state recomputation is skipped.  Only the bf16 d = 128 chunk-64
// shape with 16-byte aligned d_q, d_k, d_v (bwd_saved_shape).
cudaError_t launch_bwd(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, float d, const float *init, const void *dout,
                       const float *dfinal, void *dq, void *dk_out, void *dv_out, float *dg,
                       float *dbeta, float *dinit, int BH, int T, int dk, int dv, int C,
                       void *ws, Elem e, cudaStream_t s, const void *saved = nullptr);
bool bwd_saved_shape(int dk, int dv, int C, Elem e, const void *dq, const void *dk_out,
                     const void *dv_out);

// ---- single-token decode (gdr_decode.cu) ----
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float a_min, float *state, void *out, int N,
                          int H, int dk, int dv, Elem e, cudaStream_t s);

// ---- fused tensor-core prefill (gdr_fused.cu) ----
bool fused_supported(int dk, int dv, int C, Elem e);
cudaError_t launch_fused(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, float a_min, const float *init, void *out,
                         float *final_state, int B, int H, int T, int dk, int dv, int C,
                         cudaStream_t s);
// Packed variable-length sequences on the fused path (bf16, dk = dv = 128, C = 64).
cudaError_t launch_fused_varlen(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float a_min, const float *init, void *out,
                                float *final_state, const int *cu_seqlens, int S, int H,
                                int total_T, cudaStream_t s);

// ---- fused tensor-core prefill on a cluster of two CTAs per head (value columns
// split, preparation alternated; gdr_fused_pair.cu); chosen by launch_fused when
// every head's cluster is resident at once ----
// cu_seqlens == nullptr: dense [BH][T] layout.  Otherwise packed sequences
// (BH = S H states, tokens [total_T][H]), see gdr_chunk_fwd_varlen.
cudaError_t launch_fused_pair(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, float a_min, const float *init, void *out,
                              float *final_state, int BH, int T, const int *cu_seqlens, int H,
                              int total_T, cudaStream_t s);
// Clusters of the pair kernel resident at once on the current device (0 if unknown).
int fused_pair_max_clusters();
// Whether launch_fused runs the cluster-pair kernel for BH heads on the current device.
bool fused_uses_pair(int BH);
// Reads and clears the device error word of the pair kernel (synchronous).
cudaError_t take_pair_error_word(unsigned *value);

// ---- two-kernel prefill (bf16, dk = dv = 128, C = 64): the preparation of every
// chunk in parallel (gdr_prep.cu) into a caller-owned workspace of [Lb | P] tiles,
// then the state chain and outputs (gdr_chain.cu).  Same dense / packed layouts as
// launch_fused_pair.
size_t prep_workspace_bytes(int BH, int T, const int *cu_seqlens, int H, int total_T);
// tpb, tsc (training, dense only): also every chunk's T and P as bf16 [64][64] tiles
// ([BH][NC][2][64][64]; T plain, P with the 128-byte swizzle of the prep tile) and its row scalars ([BH][NC][4][64] fp32: gamma, 1/gamma, beta,
// d log(alpha)/dg), the inputs the backward's tiles and decay kernels would recompute.
cudaError_t launch_prep(const void *q, const void *k, const float *g, const float *beta, float a_min,
                        void *ws, int BH, int T, const int *cu_seqlens, int H, int total_T,
                        cudaStream_t s, void *tpb = nullptr, float *tsc = nullptr);
// nseg > 1 (dense only): the chain of every segment of every head at once, each
// from its state in seg_init ([BH][nseg][dk][dv], from launch_segment_states).
// saved != nullptr (dense only): every chunk's state M_n^T ([BH][NC][128 j][128 i]) and
// W_n^T ([BH][NC][128 j][64 s]) as value-major bf16 tiles, for gdr_chunk_bwd_saved;
// states_only (with saved): those only, without the output products (out is not written).
cudaError_t launch_chain(const void *q, const void *k, const void *v, const float *g, const float *beta,
                         float a_min, const float *init, void *out, float *final_state, const void *ws,
                         int BH, int T, const int *cu_seqlens, int H, int total_T, cudaStream_t s,
                         int nseg = 1, const float *seg_init = nullptr, void *saved = nullptr,
                         bool states_only = false);
// The saved buffer, per (head, chunk) tile x of X = BH ceil(T / 64), in four parts: the
// states M_x^T (bf16 [128][128]), then W_x^T (bf16 [128][64]), then T_x and P_x (bf16
// [2][64][64]), then the row scalars (fp32 [4][64]).  Offsets of the parts and the size.
inline size_t saved_tiles(int64_t BH, int T) { return (size_t)BH * ((T + 63) / 64); }
inline size_t saved_state_bytes(int64_t BH, int T) { return saved_tiles(BH, T) * 128 * 128 * 2; }
inline size_t saved_tp_offset(int64_t BH, int T) { return saved_tiles(BH, T) * 128 * (128 + 64) * 2; }
inline size_t saved_sc_offset(int64_t BH, int T) {
    return saved_tp_offset(BH, T) + saved_tiles(BH, T) * 2 * 64 * 64 * 2;
}
inline size_t saved_bytes(int64_t BH, int T) { return saved_sc_offset(BH, T) + saved_tiles(BH, T) * 4 * 64 * 4; }
// CTAs per view of the chain kernel for BH views on the current device (2 or 1).
int chain_split(int BH);

// ---- sequence segments of the two-kernel path (gdr_segment.cu) ----
// Segments per head for BH heads of T tokens on the current device (1 = none).
int segment_count(int BH, int T);
// Chunks per segment (the last segment may have fewer).
int segment_chunks(int T, int S);
// Workspace bytes of the segment maps and states (0 for S <= 1).
size_t segment_workspace_bytes(int BH, int S);
// Pass 1 (each segment's offset map Delta and transition Phi, every segment at once)
// and the scan over segments, writing every segment's initial state into the last
// part of seg_ws ([BH][S][dk][dv]); ws_tiles holds the preparation's tiles.
cudaError_t launch_segment_states(const void *k, const void *v, const float *g, const float *beta,
                                  float a_min, const float *init, const void *ws_tiles,
                                  float *seg_ws, int BH, int T, int S, cudaStream_t s);
// The segment states of seg_ws (its last BH S dk dv floats).
inline float *segment_states(float *seg_ws, int BH, int S) {
    return seg_ws + (size_t)2 * BH * (S - 1) * 128 * 128;
}
cudaError_t take_segment_error_word(unsigned *value);
// Read and clear the device error words of the two kernels (synchronous).
cudaError_t take_prep_error_word(unsigned *value);
cudaError_t take_bwd_error_word(unsigned *value);
// TMA map of a bf16 [BH][T][128] tensor: 64 x 64 boxes, 128-byte swizzle, zero fill past T
bool make_rows_map(CUtensorMap *m, const void *ptr, int BH, int T);
// Store maps of the backward's reverse chain: dR fp32 [BH][T][128] (16 x 64 boxes) and the
// per-chunk dM' tiles bf16 [X][128][128] (64 x 16 boxes, 128-byte swizzle)
bool make_dr_store_map(CUtensorMap *m, void *ptr, int BH, int T);
bool make_ds_store_map(CUtensorMap *m, void *ptr, int64_t X);
cudaError_t take_chain_error_word(unsigned *value);

// ---- one decode step of gated multi-head latent attention (gdr_mla.cu) ----
bool mla_supported(int H, int dc, int dh);
// Splits of each sequence's cache (CTAs per (sequence, group of 64 heads)).
int mla_splits(int N, int H, int Lmax);
size_t mla_workspace_bytes(int N, int H, int Lmax);
cudaError_t launch_mla_decode(const void *q_abs, const void *ckv, const int *seqlens, const void *w_uv,
                              const float *gate, float scale, void *out, int N, int H, int Lmax, int dh,
                              void *ws, cudaStream_t s);
cudaError_t take_mla_error_word(unsigned *value);

// ---- the per-chunk gradients of the bf16 d = 128 chunk-64 backward on tcgen05
// (gdr_bwd_tc.cu): Wt, Sb, dSb are the value-major bf16 tiles [BH][NC][128][64 / 128]
// (W^T, the states, the state gradients), dR the fp32 [BH][T][128] rows of the reverse
// chain, tsc the fp32 row scalars [BH][NC][4][64] of every chunk (gamma, 1 / gamma, beta,
// d log(alpha) / dg; rows past the end 1, 1, 0, 0); writes dq, dk, dv, dg, dbeta.
cudaError_t launch_bwd_chunk_tc(const void *q, const void *k, const void *v, const float *tsc,
                                const void *Wt, const void *Sb, const void *dout, const float *dR,
                                const void *dSb, void *dq, void *dk, void *dv, float *dg,
                                float *dbeta, int BH, int T, cudaStream_t s);
cudaError_t take_bwd_tc_error_word(unsigned *value);

// Device error word shared by every kernel with a bounded wait.
// Returns the word's value and clears it (synchronous on `s`).
cudaError_t read_and_clear_device_error(cudaStream_t s, unsigned *value);

// Codes stored in the device error word.
constexpr unsigned kDevErrTimeout = 1u;

}  // namespace gdr
