// gdr_math.cuh -- scalar pieces of the lower-bounded decay shared by the
// kernels of libgdr.so.
#pragma once

namespace gdr {

// The decay parameter d of every kernel selects one of the two lower-bounded
// decays ("Trillion-Parameter MoE Multimodal LLMs: How to Evaluate the New
// Generation", section 3.1; "What a Trillion-Parameter MoE Model Reveals About
// the Next Stage of LLM Scaling", section 3.2):
//   d > 0:  alpha = d + (1 - d) sigmoid(g)      (linear domain, floor a_min = d)
//   d <= 0: log alpha = d sigmoid(g)             (log domain, floor g_min = d)
// log(alpha) of the linear form is written through 1 - alpha = (1 - d)/(1 + e^g)
// so that alpha close to 1 keeps its relative accuracy.
__device__ __forceinline__ float log_alpha(float g, float d) {
    return d > 0.0f ? log1pf(-(1.0f - d) / (1.0f + expf(g))) : d / (1.0f + expf(-g));
}
__device__ __forceinline__ float decay_alpha(float g, float d) {
    return d > 0.0f ? d + (1.0f - d) / (1.0f + expf(-g)) : expf(d / (1.0f + expf(-g)));
}
// d log(alpha) / d g of the two forms: (1 - d) s (1 - s) / alpha and d s (1 - s), s = sigmoid(g).
__device__ __forceinline__ float decay_dlog_dg(float g, float d) {
    const float s = 1.0f / (1.0f + expf(-g));
    return d > 0.0f ? (1.0f - d) * s * (1.0f - s) / decay_alpha(g, d) : d * s * (1.0f - s);
}

}  // namespace gdr
