// gdr_math.cuh -- scalar pieces of the lower-bounded decay shared by the
// kernels of libgdr.so.
#pragma once

namespace gdr {

// log(alpha) for alpha = a_min + (1 - a_min) sigmoid(g), the lower-bounded
// decay ("Trillion-Parameter MoE Multimodal LLMs: How to Evaluate the New
// Generation", section 3.1, read in the linear domain with floor a_min).
// Written through 1 - alpha = (1 - a_min) / (1 + e^g) so that alpha close to
// 1 keeps its relative accuracy.
__device__ __forceinline__ float log_alpha(float g, float a_min) {
    return log1pf(-(1.0f - a_min) / (1.0f + expf(g)));
}

}  // namespace gdr
