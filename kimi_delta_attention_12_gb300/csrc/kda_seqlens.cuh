// kda_seqlens.cuh -- sequence bounds read from a device cu_seqlens array,
// clamped so that a malformed array can never send a kernel outside the
// packed token range.
//
// The C ABI takes cu_seqlens as a device array and validates it only when the
// caller also passes a host mirror.  Every kernel therefore derives a
// sequence's tokens from it through these helpers: each entry is clamped to
// [0, total_T] and a sequence ends no earlier than it starts, so
//     0 <= bos <= eos <= total_T
// whatever the array holds.  For a valid array (starting at 0, non-decreasing,
// ending at total_T) the clamps change nothing.  A malformed array gives
// meaningless (possibly overlapping) sequences, but every read of q, k, v, z,
// beta and every write of o stays inside the caller's buffers.
#pragma once

#include <stdint.h>

namespace kda {

__device__ __forceinline__ int64_t clamp_token(int64_t t, int64_t total_T) {
    return t < 0 ? 0 : (t > total_T ? total_T : t);
}

// [bos, eos) of sequence n: cu_seqlens when given, else N equal sequences.
__device__ __forceinline__ void clamped_seq(const int32_t* cu_seqlens, int n, int N,
                                            int64_t total_T, int64_t& bos, int64_t& eos) {
    if (cu_seqlens) {
        bos = clamp_token(cu_seqlens[n], total_T);
        const int64_t e = clamp_token(cu_seqlens[n + 1], total_T);
        eos = e < bos ? bos : e;
    } else {
        const int64_t len = total_T / N;
        bos = (int64_t)n * len;
        eos = bos + len;
    }
}

// Length of sequence n, as clamped_seq defines it.
__device__ __forceinline__ int64_t clamped_len(const int32_t* cu_seqlens, int n, int N,
                                               int64_t total_T) {
    int64_t bos, eos;
    clamped_seq(cu_seqlens, n, N, total_T, bos, eos);
    return eos - bos;
}

}  // namespace kda
