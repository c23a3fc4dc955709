// Warp-level sums for the token-serial kernels' state layout: a CTA's 32
// value columns spread as 8 lanes x float4 per state row, 4 row groups per
// warp (lane = 8 * row group + column group).
#pragma once

namespace kda {

// Sum of a float4 of column partials over the warp's 4 row groups (lane bits 3
// and 4), transposed: each exchange halves what a lane carries (3 shuffles
// instead of 8).  Returns component (lane >> 3) of the lane's column group,
// i.e. the sum for column 4 * (lane & 7) + (lane >> 3).
__device__ __forceinline__ float rowgroups_sum4(float4 v, int lane) {
    const bool b4 = lane & 16, b3 = lane & 8;
    float k0 = (b4 ? v.z : v.x) + __shfl_xor_sync(0xffffffffu, b4 ? v.x : v.z, 16);
    float k1 = (b4 ? v.w : v.y) + __shfl_xor_sync(0xffffffffu, b4 ? v.y : v.w, 16);
    return (b3 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, b3 ? k0 : k1, 8);
}

// Sum of a float4 of column partials over all 32 lanes of a warp (rows):
// transposed over lane bits 4 and 3 as above, then butterflies over bits 2,
// 1, 0 (6 shuffles).  Returns the sum of component (lane >> 3), on every lane.
__device__ __forceinline__ float warp_colsum4(float4 v, int lane) {
    float s = rowgroups_sum4(v, lane);
    s += __shfl_xor_sync(0xffffffffu, s, 4);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    return s;
}

// The float4 whose component c is on lanes 8c .. 8c+7 (the layout
// warp_colsum4 leaves), on every lane.
__device__ __forceinline__ float4 gather4(float x) {
    return make_float4(__shfl_sync(0xffffffffu, x, 0), __shfl_sync(0xffffffffu, x, 8),
                       __shfl_sync(0xffffffffu, x, 16), __shfl_sync(0xffffffffu, x, 24));
}

}  // namespace kda
