// kda_conv_math.cuh -- the arithmetic of the short convolutions, shared by the
// standalone kernels (kda_short_conv.cu) and the split prefill with the
// convolutions fused (kda_split_phases.cuh), so that both give the same bits.
#pragma once

#include <cuda_runtime.h>

namespace kda {

// y * sigmoid(y) = y / (1 + 2^(-y log2 e)), without a branch: below about
// y = -88 the power overflows to +inf and the approximate reciprocal returns
// +0, the function's limit (the exact value is below 1e-36 there).  The
// approximate ex2 and rcp keep the relative error near 1e-7, far below the
// bf16 rounding of the stored result.
__device__ __forceinline__ float silu_f(float y) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-1.4426950408889634f * y));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return y * r;
}

// One output of the causal depthwise convolution of width R + 1: the current
// input times the last tap, then the earlier inputs oldest first,
//     acc = w[R] x_t;  acc = fma(w[r], x_{t-R+r}, acc) for r = 0 .. R-1,
// then the SiLU if asked.  win[3 - R + r] holds x_{t-R+r}.
template <int R>
__device__ __forceinline__ float conv_step(const float (&w)[4], const float (&win)[3], float cur,
                                           bool silu) {
    float acc = w[R] * cur;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        acc = fmaf(w[r], win[3 - R + r], acc);
    }
    return silu ? silu_f(acc) : acc;
}

}  // namespace kda
