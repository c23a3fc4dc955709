// kda_state_io.cu -- movement of the persistent fp32 KDA states by slot.
//
// A state is H * d_k * d_v fp32 values (d_v contiguous), the fixed-size
// per-request memory that "Kimi K3 Open Weights: What Is Actually New In Its
// 2.8 Trillion Parameter Architecture" (section "Why 104B active still
// understates the systems problem") lists as the KDA half of the serving
// cache.  These kernels hand prefill's final states to the decode pool and
// back.  All of them are plain 128-bit streaming copies: one CTA per state,
// grid-stride over its float4s.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;

// mode 0: dst[slot(i)] = 0;  mode 1: dst[i] = src[slot(i)];  mode 2: dst[slot(i)] = src[i].
// A slot outside [0, pool_size) skips its state, except that a gather fills
// dst[i] with NaN so that a bad slot cannot pass a stale state on unnoticed
// (as decode writes NaN to the o row of such a slot).
__global__ void __launch_bounds__(kThreads)
state_slot_kernel(float* __restrict__ dst, const float* __restrict__ src,
                  const int32_t* __restrict__ slots, int32_t pool_size,
                  size_t state_vec4, int mode) {
    const int i = blockIdx.x;
    const int32_t s = slots ? slots[i] : i;
    if (s < 0 || s >= pool_size) {
        if (mode == 1) {
            const float qnan = __int_as_float(0x7fc00000);
            float4* d = reinterpret_cast<float4*>(dst) + (size_t)i * state_vec4;
            for (size_t e = threadIdx.x; e < state_vec4; e += kThreads) {
                __stcs(d + e, make_float4(qnan, qnan, qnan, qnan));
            }
        }
        return;
    }
    float4* d;
    const float4* sp = nullptr;
    if (mode == 0) {
        d = reinterpret_cast<float4*>(dst) + (size_t)s * state_vec4;
    } else if (mode == 1) {
        d = reinterpret_cast<float4*>(dst) + (size_t)i * state_vec4;
        sp = reinterpret_cast<const float4*>(src) + (size_t)s * state_vec4;
    } else {
        d = reinterpret_cast<float4*>(dst) + (size_t)s * state_vec4;
        sp = reinterpret_cast<const float4*>(src) + (size_t)i * state_vec4;
    }
    for (size_t e = threadIdx.x; e < state_vec4; e += kThreads) {
        const float4 x = sp ? __ldcs(sp + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        __stcs(d + e, x);
    }
}

cudaError_t launch_slot(float* dst, const float* src, const int32_t* slots, int32_t n,
                        int32_t pool_size, size_t state_floats, int mode,
                        cudaStream_t stream) {
    if (n <= 0) {
        return cudaSuccess;
    }
    state_slot_kernel<<<n, kThreads, 0, stream>>>(dst, src, slots, pool_size,
                                                  state_floats / 4, mode);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state_zero_slots(float* dst, const int32_t* slots, int32_t n,
                                    int32_t pool_size, size_t state_floats,
                                    cudaStream_t stream) {
    return launch_slot(dst, nullptr, slots, n, pool_size, state_floats, 0, stream);
}

cudaError_t launch_state_gather(float* dst, const float* src, const int32_t* slots,
                                int32_t n, int32_t pool_size, size_t state_floats,
                                cudaStream_t stream) {
    return launch_slot(dst, src, slots, n, pool_size, state_floats, 1, stream);
}

cudaError_t launch_state_scatter(float* dst, const float* src, const int32_t* slots,
                                 int32_t n, int32_t pool_size, size_t state_floats,
                                 cudaStream_t stream) {
    return launch_slot(dst, src, slots, n, pool_size, state_floats, 2, stream);
}

}  // namespace kda
