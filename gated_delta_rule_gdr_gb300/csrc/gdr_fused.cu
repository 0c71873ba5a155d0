// gdr_fused.cu -- fused tensor-core chunked prefill (placeholder: the fused
// kernel is not wired in yet, so every shape takes the staged path) and the
// device error word shared by kernels with bounded waits.

#include "gdr_internal.h"

namespace gdr {

__device__ unsigned g_device_error_word = 0;

bool fused_supported(int, int, int, Elem) { return false; }

cudaError_t launch_fused(const void *, const void *, const void *, const float *,
                         const float *, float, const float *, void *, float *, int, int, int,
                         int, int, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t read_and_clear_device_error(cudaStream_t s, unsigned *value) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    unsigned word = 0;
    e = cudaMemcpyFromSymbol(&word, g_device_error_word, sizeof(word));
    if (e != cudaSuccess) return e;
    *value = word;
    if (word != 0) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero));
    }
    return e;
}

}  // namespace gdr
