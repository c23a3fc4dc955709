// kda_internal.h -- declarations shared by the C-ABI layer (kda_api.cpp) and
// the CUDA translation units.  Not part of the public interface.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

// Parameters of the fused recurrent kernel (one CTA per (row, head)).
// Prefill: row = sequence n, tokens cu_seqlens[n] .. cu_seqlens[n+1]-1,
//          state_in = initial_state (may be null), state_out = final_state
//          (may be null), slots = null.
// Decode:  row = batch entry b, one token (index b), state_in = state_out =
//          the pool, state index = slots ? slots[b] : b.
struct RecurrentParams {
    const void* q;
    const void* k;
    const void* v;
    const void* z;
    const void* beta;
    const float* A;
    const float* state_in;
    float* state_out;
    const int32_t* slots;
    const int32_t* cu_seqlens;
    void* o;
    int32_t rows;       // N (prefill) or B (decode)
    int32_t total_T;
    int32_t H;
    int32_t pool_size;  // decode only
    float scale;
    int32_t l2norm;
    int32_t decode;
    int32_t softplus_gate;  // Kimi Linear's gate -softplus(e^A z) instead of -5 sigmoid(e^A z)
    // prefill only: state checkpoints every ckpt_interval tokens (0 = none)
    int32_t ckpt_interval;
    float* ckpt_pool;
    const int32_t* ckpt_slots;
    int32_t ckpt_pool_size;
    int64_t ckpt_count;     // checkpoints with index >= this are skipped (ckpt_slots bound)
};

// Short convolutions of q, k and v (kda_short_conv.cu).  Conv weights and
// states use the per-head packed channel order q | k | v (Cc = 2 d_k + d_v):
// w [H, Cc, W] fp32, states [N, H, W-1, Cc] in the input dtype.
struct ShortConvParams {
    const void* x[3];            // q, k [total_T, H, d_k]; v [total_T, H, d_v]
    void* y[3];                  // convolved q, k, v, same layouts
    const float* w;
    const void* state_in;        // or null (zeros)
    void* state_out;             // or null
    const int32_t* cu_seqlens;   // device [N + 1], or null for equal lengths
    int32_t N;
    int32_t total_T;
    int32_t H;
    int32_t d_k;
    int32_t d_v;
    int32_t W;                   // 1 .. 4
    int32_t silu;
};
cudaError_t launch_short_conv(const ShortConvParams& p, int dtype, cudaStream_t stream);

// One decode token of short convolutions per batch row: y = the convolved q,
// k, v (layouts [B, H, d]); the row's conv state (pool row slots[b], or b) is
// shifted by the token in place.  Rows with a slot outside [0, pool_size)
// are skipped (their y is left unwritten).
struct ShortConvDecodeParams {
    const void* x[3];            // q, k [B, H, d_k]; v [B, H, d_v]
    void* y[3];
    const float* w;              // [H, 2 d_k + d_v, W] fp32
    void* state;                 // [pool_size, H, W-1, 2 d_k + d_v]
    const int32_t* slots;        // or null (identity)
    int32_t B;
    int32_t pool_size;
    int32_t H;
    int32_t d_k;
    int32_t d_v;
    int32_t W;                   // 1 .. 4
    int32_t silu;
};
cudaError_t launch_short_conv_decode(const ShortConvDecodeParams& p, int dtype,
                                     cudaStream_t stream);

// Training backward of the recurrence (kda_backward.cu): d_v / 32 CTAs per
// (sequence, head); the states every kBwChunk tokens in `pool` (the layout of
// the checkpointed prefill: checkpoint m >= 1 of sequence n at row
// (checkpoints of sequences before n) + m - 1), per-pair scratch of kBwChunk
// states, per-CTA column partials [d_v / 32][total_T][H][3 d_k + 1] of dqh,
// dkh, da, db, per-token dA shares.
constexpr int kBwChunk = 64;
struct BackwardParams {
    const void* q;
    const void* k;
    const void* v;
    const void* z;
    const void* beta;
    const float* A;
    const float* initial_state;  // or null
    const int32_t* cu_seqlens;   // or null (equal lengths)
    const void* dO;              // [total_T, H, d_v]
    const float* dS_final;       // [N, H, d_k, d_v] or null
    float* dq;                   // [total_T, H, d_k] fp32
    float* dk;
    float* dv;                   // [total_T, H, d_v]
    float* dz;
    float* dbeta;                // [total_T, H]
    float* dA;                   // [H]
    float* dS0;                  // [N, H, d_k, d_v]
    const float* pool;           // workspace: the chunk-start states
    int64_t pool_rows;           // states in the pool (reads beyond it are skipped)
    float* scratch;
    float* part;
    float* dA_tok;               // [total_T, H]
    int32_t N;
    int32_t total_T;
    int32_t H;
    float scale;
    int32_t l2norm;
    int32_t softplus_gate;
};
cudaError_t launch_backward(const BackwardParams& p, int d_k, int d_v, int dtype,
                            cudaStream_t stream);
// dA[h] = the sum over tokens of dA_tok[t][h] (fixed order).
cudaError_t launch_backward_dA(const float* dA_tok, float* dA, int64_t total_T, int H,
                               cudaStream_t stream);

// Launches the recurrent kernel for (d_k, d_v) in {32, 64, 128}^2 and
// dtype (0 = fp32, 1 = bf16).  Returns a cudaError_t.
cudaError_t launch_recurrent(const RecurrentParams& p, int d_k, int d_v, int dtype,
                             cudaStream_t stream);

// State movement kernels (kda_state_io.cu).
cudaError_t launch_state_zero_slots(float* dst, const int32_t* slots, int32_t n,
                                    int32_t pool_size, size_t state_floats,
                                    cudaStream_t stream);
cudaError_t launch_state_gather(float* dst, const float* src, const int32_t* slots,
                                int32_t n, int32_t pool_size, size_t state_floats,
                                cudaStream_t stream);
cudaError_t launch_state_scatter(float* dst, const float* src, const int32_t* slots,
                                 int32_t n, int32_t pool_size, size_t state_floats,
                                 cudaStream_t stream);

}  // namespace kda

#include "kda_chunked.h"
