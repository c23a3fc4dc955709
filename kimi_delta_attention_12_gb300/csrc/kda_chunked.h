// kda_chunked.h -- declarations of the chunked tensor-core prefill
// (kda_prefill_sm103.cu, kda_chunk_phases.cuh) shared with the C-ABI layer.
// Kept apart from kda_internal.h so that the chunked kernels are compiled
// from this header, the two sources and the PTX wrappers alone.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

// Chunked tensor-core prefill (kda_prefill_sm103.cu): bf16, d_k = d_v = 128.
struct ChunkedParams {
    const void* q;
    const void* k;
    const void* v;
    const void* z;
    const void* beta;
    const float* A;
    const float* initial_state;
    float* final_state;
    const int32_t* cu_seqlens;   // device, [N+1]; null -> equal split
    void* o;                     // (split mode: null skips the output stores)
    int32_t* status;             // device status word (workspace)
    int32_t* work_counter;       // device work counter (workspace)
    const int32_t* schedule;     // optional device list of unit ids (workspace), or null
    // split mode (see SplitPlan): ring slots of published chunks
    int32_t* flags;              // [consumers][ring]: stream index + 1 of the chunk in the slot
    int32_t* cons_done;          // [consumers]: chunks each consumer has copied out
    uint8_t* handoff;            // [consumers][ring] slots of published chunk tiles
    int32_t n_cons;              // consumer CTAs (units per batch)
    int32_t n_batches;           // batches of units, walked one after another
    int32_t ring;                // slots per consumer
    int32_t N;
    int32_t total_T;
    int32_t H;
    float scale;
    int32_t l2norm;
    // state checkpoints every ckpt_interval tokens (a multiple of the chunk; 0 = none)
    int32_t ckpt_interval;
    float* ckpt_pool;
    const int32_t* ckpt_slots;
    int32_t ckpt_pool_size;
    int64_t ckpt_count;          // checkpoints with index >= this are skipped (ckpt_slots bound)
    // polls of a wait on another CTA (split mode) before it gives up
    uint32_t peer_wait_polls;
    // split mode only: when set, producers write every chunk into its own
    // chunk record (REC_BYTES each, record (chunk base of its sequence +
    // chunk) * H + head, the chunk base being the sum of ceil(length / 64)
    // over earlier sequences) instead of a ring slot, with the extra tiles
    // of the record; the ring flags still hand it to the consumer, which
    // copies it from there
    uint8_t* records;
    int64_t rec_chunks;          // records per head the buffer holds (a bound on the chunk count)
    // split mode only: the short convolutions of q, k, v fused in (conv_w
    // non-null), as kda_short_conv computes them: taps [H][2*128+128][W] fp32,
    // conv states [N][H][W-1][384] bf16 in (or null: zeros) and out (or null);
    // the slots then carry the convolved v tile (HO_BYTES_CONV each)
    const float* conv_w;
    const void* conv_state_in;
    void* conv_state_out;
    int32_t conv_W;
    int32_t conv_silu;
};
constexpr uint32_t kChunkRecordBytes = 132096;  // one chunk record (REC_BYTES)

// Split mode: the N*H (sequence, head) units are cut into `batches` batches of
// at most `consumers` units; consumer CTA i carries the state of unit
// b * consumers + i of every batch b in turn, and producer CTAs (the other
// SMs) compute the chunks' state-independent operands, passing them through a
// ring of `ring` workspace slots per consumer.
struct SplitPlan {
    int32_t consumers;
    int32_t batches;
    int32_t ring;
};
constexpr int kSplitMaxSeqs = 1024;
constexpr int kSplitMaxHeads = 256;
constexpr int kSplitMaxBatches = 256;

// Chunked training backward (kda_bwd_chunked.cu): bf16 inputs, d_k = d_v =
// 128, the bounded gate.  Runs after the split prefill has written the chunk
// records (each with its chunk's start state).
struct BwdChunkedParams {
    const void* q;               // [total_T][H][128] bf16, as the forward
    const void* k;
    const void* v;
    const void* z;
    const void* beta;            // [total_T][H] bf16
    const float* A;              // [H]
    const void* dO;              // [total_T][H][128] bf16
    const float* dS_final;       // [N][H][128][128] or null (zero)
    const int32_t* cu_seqlens;   // device [N+1]; null -> equal split
    const uint8_t* records;      // chunk records of the split prefill (with the start states)
    uint8_t* dsl;                // [chunks][H] dL/dS at each chunk's end (bf16 operand tiles)
    int32_t* chunk_map;          // [max_chunks][4]: sequence (-1: unused), chunk
    int32_t max_chunks;          // total_T / 64 + N, a bound on the chunk count
    float* dq;                   // gradients, fp32, layouts of their inputs
    float* dk;
    float* dv;
    float* dz;
    float* dbeta;
    float* dA_tok;               // [total_T][H] per-token shares of dL/dA
    float* dS0;                  // [N][H][128][128]
    int32_t* status;             // device status word
    int32_t N;
    int32_t total_T;
    int32_t H;
    float scale;
    int32_t l2norm;
};
constexpr uint32_t kBwdDslBytes = 32768;   // one chunk's dL/dS tile: 2 x [128 c][64 v] bf16

// The reverse state chain (one CTA per (sequence, head)) and the chunk-parallel
// gradient assembly; the caller sets chunk_map to -1 first and sums dA_tok.
cudaError_t launch_bwd_chunked(const BwdChunkedParams& p, cudaStream_t stream);

// True once the chunked kernel is compiled into the library.
constexpr bool kChunkedPrefillBuilt = true;

// Workspace layout for the chunked prefill.  Single pass: a 256-byte header
// (status word, work counter) and one int per unit.  Split mode: the header,
// the ring flags and consumer counters (zeroed on every call), then the ring
// slots.
size_t chunked_workspace_bytes(int32_t N, int32_t H);
// Smallest workspace kda_prefill accepts (it then runs the single-pass kernel).
size_t min_prefill_workspace_bytes(int32_t N, int32_t H);
// The split plan for these sizes on a GPU with num_sms SMs; false if they do
// not run in split mode.
bool split_plan(int32_t N, int32_t H, int num_sms, SplitPlan* plan);
size_t split_zeroed_bytes(const SplitPlan& plan);
// (conv: slots with the convolved v tile, for the fused short convolutions)
size_t split_workspace_bytes(const SplitPlan& plan, bool conv = false);
// Points p's split-mode fields into a workspace laid out for plan.
void split_bind(const SplitPlan& plan, void* workspace, ChunkedParams* p);
// TMA map of a packed [total_T][H][128] bf16 tensor with a box of 64 tokens
// by 128 channels (no swizzle: one 16 KB row-major tile) or, swizzled, 64
// channels (128-byte swizzle: one 8 KB operand half per load).
bool make_token_map(CUtensorMap* map, const void* base, int total_T, int H, bool swizzled);
cudaError_t launch_chunked_prefill(const ChunkedParams& p, cudaStream_t stream);
cudaError_t launch_split_prefill(const ChunkedParams& p, int num_sms, cudaStream_t stream);

}  // namespace kda
