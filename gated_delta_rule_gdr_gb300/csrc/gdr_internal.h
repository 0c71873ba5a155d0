// gdr_internal.h -- launchers shared between the C-ABI layer and the kernel
// translation units of libgdr.so.  Not installed; the public surface is
// include/gdr.h.
#pragma once

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

// ---- backward of the chunked form (gdr_bwd.cu) ----
bool bwd_supported(int dk, int dv, int C);
size_t bwd_workspace_bytes(int BH, int T, int dk, int dv, int C);
cudaError_t launch_bwd(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, float d, const float *init, const void *dout,
                       const float *dfinal, void *dq, void *dk_out, void *dv_out, float *dg,
                       float *dbeta, float *dinit, int BH, int T, int dk, int dv, int C,
                       void *ws, Elem e, cudaStream_t s);

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
cudaError_t launch_prep(const void *q, const void *k, const float *g, const float *beta, float a_min,
                        void *ws, int BH, int T, const int *cu_seqlens, int H, int total_T,
                        cudaStream_t s);
cudaError_t launch_chain(const void *q, const void *k, const void *v, const float *g, const float *beta,
                         float a_min, const float *init, void *out, float *final_state, const void *ws,
                         int BH, int T, const int *cu_seqlens, int H, int total_T, cudaStream_t s);
// CTAs per head of the chain kernel for BH heads on the current device (2 or 1).
int chain_split(int BH);
// Read and clear the device error words of the two kernels (synchronous).
cudaError_t take_prep_error_word(unsigned *value);
cudaError_t take_chain_error_word(unsigned *value);

// Device error word shared by every kernel with a bounded wait.
// Returns the word's value and clears it (synchronous on `s`).
cudaError_t read_and_clear_device_error(cudaStream_t s, unsigned *value);

// Codes stored in the device error word.
constexpr unsigned kDevErrTimeout = 1u;

}  // namespace gdr
