// kda_short_conv.cu -- the short convolutions of q, k and v for prefill.
//
// "Kimi K3 Open Weights: What Is Actually New In Its 2.8 Trillion Parameter
// Architecture", section 1, lists short convolutions first among the KDA
// prefill steps and keeps a convolution state persistent through decode.
// The operation (the pages give no formula; this is the plain reading): a
// causal depthwise convolution along time of width W on every channel,
//     y_t[c] = sum_{j<W} w[c][j] * x_{t-W+1+j}[c],   optionally y * sigmoid(y),
// where inputs before a sequence's first token are the rows of its conv state
// (the W-1 inputs that preceded it, oldest first) and the final conv state is
// the last W-1 inputs of the sequence.
//
// Memory-bound: every input element is read once from HBM (plus W-1 halo rows
// per block of tokens, from L2) and every output written once.  A thread owns
// one 8-byte vector of channels of one tensor (4 bf16 or 2 fp32 channels) for
// a block of TB consecutive tokens and slides a window of the last W-1 rows
// through registers.  Consecutive threads own consecutive vectors of the same
// token row, so a warp reads and writes 256 contiguous bytes per token.
// Loads are issued eight rows ahead of their use; at 64 registers four CTAs
// of 256 threads share an SM, which keeps enough loads in flight.
//
// Grid: x = token blocks, then one block per sequence that writes that
// sequence's final conv state; y = groups of 256 channel vectors.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_conv_math.cuh"
#include "kda_internal.h"
#include "kda_seqlens.cuh"

namespace kda {
namespace {

constexpr int kConvThreads = 256;
constexpr int kConvTB = 32;     // tokens per block
constexpr int kConvAhead = 8;   // rows per copy group
constexpr int kConvStages = 3;  // copy groups in the per-thread ring (two ahead)

// 8-byte asynchronous copy global -> shared (the thread's own ring slot).
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// An 8-byte vector of channels: 4 bf16 or 2 fp32.
template <typename T>
struct VecTraits;
template <>
struct VecTraits<float> {
    static constexpr int kN = 2;
    __device__ static void unpack(const uint2& r, float* f) {
        f[0] = __uint_as_float(r.x);
        f[1] = __uint_as_float(r.y);
    }
    __device__ static uint2 pack(const float* f) {
        return make_uint2(__float_as_uint(f[0]), __float_as_uint(f[1]));
    }
};
template <>
struct VecTraits<__nv_bfloat16> {
    static constexpr int kN = 4;
    __device__ static void unpack(const uint2& r, float* f) {
        f[0] = __uint_as_float(r.x << 16);
        f[1] = __uint_as_float(r.x & 0xffff0000u);
        f[2] = __uint_as_float(r.y << 16);
        f[3] = __uint_as_float(r.y & 0xffff0000u);
    }
    __device__ static uint2 pack(const float* f) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(f[0], f[1]);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(f[2], f[3]);
        return make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                          *reinterpret_cast<const uint32_t*>(&hi));
    }
};


__device__ __forceinline__ uint2 ld8(const void* base, size_t elem_off, int eb) {
    return __ldg(reinterpret_cast<const uint2*>(static_cast<const char*>(base) +
                                                elem_off * eb));
}

// Which tensor, head and channel a channel vector is.
struct ChanVec {
    int tensor;      // 0 q, 1 k, 2 v
    int h;
    int c0;          // first channel within the tensor's head
    int d;           // head dim of the tensor
    int off;         // first channel within the head's packed q | k | v channels
};

template <int VEC>
__device__ __forceinline__ bool chan_vec(int H, int d_k, int d_v, int gv, ChanVec* cv) {
    const int vq = H * d_k / VEC;
    const int vv = H * d_v / VEC;
    int lin = gv;
    if (lin < vq) {
        cv->tensor = 0; cv->d = d_k;
    } else if (lin < 2 * vq) {
        lin -= vq; cv->tensor = 1; cv->d = d_k;
    } else if (lin < 2 * vq + vv) {
        lin -= 2 * vq; cv->tensor = 2; cv->d = d_v;
    } else {
        return false;
    }
    const int per_head = cv->d / VEC;
    cv->h = lin / per_head;
    cv->c0 = (lin % per_head) * VEC;
    cv->off = (cv->tensor == 0 ? 0 : cv->tensor == 1 ? d_k : 2 * d_k) + cv->c0;
    return true;
}

// The taps of VEC consecutive channels, w[h][off + i][j] (VEC * W contiguous
// floats, 16-byte aligned when W = 4), as wt[j][i].
template <int VEC, int W>
__device__ __forceinline__ void load_taps(const float* wbase, float (&wt)[W][VEC]) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        if constexpr (W == 4) {
            const float4 t = __ldg(reinterpret_cast<const float4*>(wbase) + i);
            wt[0][i] = t.x; wt[1][i] = t.y; wt[2][i] = t.z; wt[3][i] = t.w;
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) {
                wt[j][i] = __ldg(wbase + i * W + j);
            }
        }
    }
}

__device__ __forceinline__ void seq_bounds(const ShortConvParams& p, int n, int64_t* bos,
                                           int64_t* eos) {
    clamped_seq(p.cu_seqlens, n, p.N, p.total_T, *bos, *eos);
}

// The sequence that holds token t (t < total_T): the last n with start <= t.
__device__ __forceinline__ int seq_of(const ShortConvParams& p, int64_t t) {
    if (!p.cu_seqlens) {
        return (int)(t / (p.total_T / p.N));
    }
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.cu_seqlens[mid] <= t) {
            lo = mid;
        } else {
            hi = mid - 1;
        }
    }
    return lo;
}

// One token of one channel vector: y = sum_j wt[j] x_{t-R+j} (x_t the raw row
// rw, the earlier inputs in the window), then the SiLU if asked, stored at yp;
// the window of the last R = W - 1 inputs then slides by one.
template <typename T, int W, bool kSilu>
__device__ __forceinline__ void conv_token(const float (&wt)[W][VecTraits<T>::kN],
                                           float (&win)[W > 1 ? W - 1 : 1][VecTraits<T>::kN],
                                           const uint2& rw, char* yp) {
    using VT = VecTraits<T>;
    constexpr int VEC = VT::kN;
    constexpr int R = W - 1;
    float cur[VEC], out[VEC];
    VT::unpack(rw, cur);
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
        float acc = wt[R][c] * cur[c];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            acc = fmaf(wt[r][c], win[r][c], acc);
        }
        out[c] = kSilu ? silu_f(acc) : acc;
    }
    *reinterpret_cast<uint2*>(yp) = VT::pack(out);
#pragma unroll
    for (int r = 0; r + 1 < R; ++r) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            win[r][c] = win[r + 1][c];
        }
    }
    if (R > 0) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            win[R > 0 ? R - 1 : 0][c] = cur[c];
        }
    }
}

template <typename T, int W, bool kSilu>
__global__ void __launch_bounds__(kConvThreads, 4)
short_conv_kernel(const ShortConvParams p, int n_token_blocks) {
    using VT = VecTraits<T>;
    constexpr int VEC = VT::kN;
    constexpr int R = W - 1;
    constexpr int EB = sizeof(T);

    ChanVec cv;
    if (!chan_vec<VEC>(p.H, p.d_k, p.d_v, blockIdx.y * kConvThreads + threadIdx.x, &cv)) {
        return;
    }
    const int Cc = 2 * p.d_k + p.d_v;
    // (selected, not indexed: a dynamic index into the parameter block would
    // copy it to local memory)
    const void* x = cv.tensor == 0 ? p.x[0] : cv.tensor == 1 ? p.x[1] : p.x[2];
    const int H = p.H;
    // element offset of (token t, this vector) in x / y
    auto xoff = [=](int64_t t) { return ((size_t)t * H + cv.h) * cv.d + cv.c0; };
    // element offset of (sequence n, row r, this vector) in a conv state
    auto soff = [=](int n, int r) { return (((size_t)n * H + cv.h) * R + r) * Cc + cv.off; };

    if ((int)blockIdx.x >= n_token_blocks) {
        // final conv state of sequence n: its last W-1 inputs, oldest first
        const int n = blockIdx.x - n_token_blocks;
        if (R == 0 || !p.state_out) {
            return;
        }
        int64_t bos, eos;
        seq_bounds(p, n, &bos, &eos);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t tau = eos - R + r;
            uint2 val = make_uint2(0u, 0u);
            if (tau >= bos) {
                val = ld8(x, xoff(tau), EB);
            } else if (p.state_in) {
                val = ld8(p.state_in, soff(n, (int)(tau - bos + R)), EB);
            }
            *reinterpret_cast<uint2*>(static_cast<char*>(p.state_out) + soff(n, r) * EB) = val;
        }
        return;
    }

    const int64_t t0 = (int64_t)blockIdx.x * kConvTB;
    const int64_t t1 = min((int64_t)p.total_T, t0 + kConvTB);

    float wt[W][VEC];
    load_taps<VEC, W>(p.w + ((size_t)cv.h * Cc + cv.off) * W, wt);

    int n = seq_of(p, t0);
    int64_t bos, eos;
    seq_bounds(p, n, &bos, &eos);
    float win[R > 0 ? R : 1][VEC];   // inputs t-R .. t-1
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t tau = t0 - R + r;
        uint2 raw = make_uint2(0u, 0u);
        if (tau >= bos) {
            raw = ld8(x, xoff(tau), EB);
        } else if (p.state_in && tau >= bos - R) {   // (false only for a malformed cu_seqlens)
            raw = ld8(p.state_in, soff(n, (int)(tau - bos + R)), EB);
        }
        VT::unpack(raw, win[r]);
    }

    void* y = cv.tensor == 0 ? p.y[0] : cv.tensor == 1 ? p.y[1] : p.y[2];
    // row pointers of this vector, advanced one token (H * d elements) at a time
    const size_t row_bytes = (size_t)H * cv.d * EB;
    const char* xi = static_cast<const char*>(x) + xoff(t0) * EB;   // next row to copy
    char* yr = static_cast<char*>(y) + xoff(t0) * EB;
    // The block's rows reach each thread through its own ring of copy groups in
    // shared memory (cp.async, kConvStages - 1 groups ahead of the one being
    // worked on): more bytes in flight than registers could hold.  A thread
    // reads only the slots it copied itself, so no barrier is needed.
    __shared__ __align__(16) uint2 ring[kConvStages][kConvAhead][kConvThreads];
    int64_t ti = t0;   // first token of the next group to copy
    auto copy_group = [&](int slot) {
#pragma unroll
        for (int i = 0; i < kConvAhead; ++i) {
            if (ti + i < t1) {
                cp_async8(&ring[slot][i][threadIdx.x], xi + i * row_bytes);
            }
        }
        cp_async_commit();
        ti += kConvAhead;
        xi += kConvAhead * row_bytes;
    };
#pragma unroll
    for (int g = 0; g + 1 < kConvStages; ++g) {
        copy_group(g);
    }
    int slot = 0;
    for (int64_t tb = t0; tb < t1; tb += kConvAhead) {
        // the group kConvStages - 1 ahead, into the slot worked on last time
        copy_group(slot == 0 ? kConvStages - 1 : slot - 1);
        cp_async_wait<kConvStages - 1>();   // this group's rows have landed
        const uint2 (&raw)[kConvAhead][kConvThreads] = ring[slot];
        slot = slot + 1 == kConvStages ? 0 : slot + 1;
        if (tb + kConvAhead <= t1 && tb + kConvAhead <= eos) {
            // the whole group lies in the block and in the current sequence
#pragma unroll
            for (int i = 0; i < kConvAhead; ++i) {
                conv_token<T, W, kSilu>(wt, win, raw[i][threadIdx.x], yr + i * row_bytes);
            }
        } else {
#pragma unroll
            for (int i = 0; i < kConvAhead; ++i) {
                const int64_t t = tb + i;
                if (t >= t1) {
                    continue;
                }
                if (t >= eos) {
                    // first token of a later sequence (skipping empty ones):
                    // the window restarts from that sequence's conv state
                    while (t >= eos && n + 1 < p.N) {
                        ++n;
                        seq_bounds(p, n, &bos, &eos);
                    }
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        uint2 s = make_uint2(0u, 0u);
                        if (p.state_in) {
                            s = ld8(p.state_in, soff(n, r), EB);
                        }
                        VT::unpack(s, win[r]);
                    }
                }
                conv_token<T, W, kSilu>(wt, win, raw[i][threadIdx.x], yr + i * row_bytes);
            }
        }
        yr += kConvAhead * row_bytes;
    }
    cp_async_wait<0>();   // (copies past the block's end were never issued)
}

template <typename T, bool kSilu>
void launch_width(const ShortConvParams& p, dim3 grid, int ntb, cudaStream_t stream) {
    switch (p.W) {
        case 1: short_conv_kernel<T, 1, kSilu><<<grid, kConvThreads, 0, stream>>>(p, ntb); break;
        case 2: short_conv_kernel<T, 2, kSilu><<<grid, kConvThreads, 0, stream>>>(p, ntb); break;
        case 3: short_conv_kernel<T, 3, kSilu><<<grid, kConvThreads, 0, stream>>>(p, ntb); break;
        default: short_conv_kernel<T, 4, kSilu><<<grid, kConvThreads, 0, stream>>>(p, ntb); break;
    }
}

template <typename T>
cudaError_t launch_typed(const ShortConvParams& p, cudaStream_t stream) {
    constexpr int VEC = VecTraits<T>::kN;
    const int64_t vecs = (int64_t)p.H * (2 * p.d_k + p.d_v) / VEC;
    const int64_t ntb = ((int64_t)p.total_T + kConvTB - 1) / kConvTB;
    const int64_t gx = ntb + (p.state_out ? p.N : 0);
    if (gx == 0 || vecs == 0) {
        return cudaSuccess;
    }
    if (gx > 0x7fffffffLL || p.W < 1 || p.W > 4) {
        return cudaErrorInvalidValue;
    }
    const dim3 grid((unsigned)gx, (unsigned)((vecs + kConvThreads - 1) / kConvThreads));
    if (p.silu) {
        launch_width<T, true>(p, grid, (int)ntb, stream);
    } else {
        launch_width<T, false>(p, grid, (int)ntb, stream);
    }
    return cudaGetLastError();
}

// One decode token per batch row: thread = one 8-byte channel vector of one
// tensor of row b (grid y = b).  It reads the vector's W-1 conv-state rows
// and the token, writes the convolved vector to y and the shifted rows back
// in place; no other thread touches those channels of that row.
template <typename T, int W, bool kSilu>
__global__ void __launch_bounds__(kConvThreads)
short_conv_decode_kernel(const ShortConvDecodeParams p) {
    using VT = VecTraits<T>;
    constexpr int VEC = VT::kN;
    constexpr int R = W - 1;
    constexpr int EB = sizeof(T);
    ChanVec cv;
    if (!chan_vec<VEC>(p.H, p.d_k, p.d_v, blockIdx.x * kConvThreads + threadIdx.x, &cv)) {
        return;
    }
    const int b = blockIdx.y;
    const int slot = p.slots ? p.slots[b] : b;
    if (slot < 0 || slot >= p.pool_size) {
        return;
    }
    const int Cc = 2 * p.d_k + p.d_v;
    const void* x = cv.tensor == 0 ? p.x[0] : cv.tensor == 1 ? p.x[1] : p.x[2];
    void* y = cv.tensor == 0 ? p.y[0] : cv.tensor == 1 ? p.y[1] : p.y[2];
    const size_t xo = ((size_t)b * p.H + cv.h) * cv.d + cv.c0;
    char* rows = R > 0 ? static_cast<char*>(p.state) +
                             ((((size_t)slot * p.H + cv.h) * R) * Cc + cv.off) * EB
                       : nullptr;
    const size_t row_bytes = (size_t)Cc * EB;

    uint2 raw[R > 0 ? R : 1];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        raw[r] = *reinterpret_cast<const uint2*>(rows + r * row_bytes);
    }
    const uint2 xr = ld8(x, xo, EB);
    float wt[W][VEC];
    load_taps<VEC, W>(p.w + ((size_t)cv.h * Cc + cv.off) * W, wt);

    float cur[VEC], out[VEC];
    VT::unpack(xr, cur);
#pragma unroll
    for (int c = 0; c < VEC; ++c) {
        out[c] = wt[R][c] * cur[c];
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float prev[VEC];
        VT::unpack(raw[r], prev);
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            out[c] = fmaf(wt[r][c], prev[c], out[c]);
        }
    }
    if constexpr (kSilu) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            out[c] = silu_f(out[c]);
        }
    }
    *reinterpret_cast<uint2*>(static_cast<char*>(y) + xo * EB) = VT::pack(out);
    // shift: row r takes row r + 1, the last row takes the token
#pragma unroll
    for (int r = 0; r < R; ++r) {
        *reinterpret_cast<uint2*>(rows + r * row_bytes) = r + 1 < R ? raw[r + 1 < R ? r + 1 : 0] : xr;
    }
}

template <typename T, bool kSilu>
void launch_decode_width(const ShortConvDecodeParams& p, dim3 grid, cudaStream_t stream) {
    switch (p.W) {
        case 1: short_conv_decode_kernel<T, 1, kSilu><<<grid, kConvThreads, 0, stream>>>(p); break;
        case 2: short_conv_decode_kernel<T, 2, kSilu><<<grid, kConvThreads, 0, stream>>>(p); break;
        case 3: short_conv_decode_kernel<T, 3, kSilu><<<grid, kConvThreads, 0, stream>>>(p); break;
        default: short_conv_decode_kernel<T, 4, kSilu><<<grid, kConvThreads, 0, stream>>>(p); break;
    }
}

template <typename T>
cudaError_t launch_decode_typed(const ShortConvDecodeParams& p, cudaStream_t stream) {
    constexpr int VEC = VecTraits<T>::kN;
    const int64_t vecs = (int64_t)p.H * (2 * p.d_k + p.d_v) / VEC;
    if (p.B == 0 || vecs == 0) {
        return cudaSuccess;
    }
    if (p.B > 65535 || p.W < 1 || p.W > 4) {
        return cudaErrorInvalidValue;
    }
    const dim3 grid((unsigned)((vecs + kConvThreads - 1) / kConvThreads), (unsigned)p.B);
    if (p.silu) {
        launch_decode_width<T, true>(p, grid, stream);
    } else {
        launch_decode_width<T, false>(p, grid, stream);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_short_conv_decode(const ShortConvDecodeParams& p, int dtype,
                                     cudaStream_t stream) {
    return dtype == 0 ? launch_decode_typed<float>(p, stream)
                      : launch_decode_typed<__nv_bfloat16>(p, stream);
}

cudaError_t launch_short_conv(const ShortConvParams& p, int dtype, cudaStream_t stream) {
    return dtype == 0 ? launch_typed<float>(p, stream) : launch_typed<__nv_bfloat16>(p, stream);
}

}  // namespace kda
