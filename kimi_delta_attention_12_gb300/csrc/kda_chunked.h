// kda_chunked.h -- declarations of the chunked tensor-core prefill
// (kda_prefill_sm103.cu, kda_chunk_phases.cuh) shared with the C-ABI layer.
// Kept apart from kda_internal.h so that the chunked kernels are compiled
// from this header, the two sources and the PTX wrappers alone.
#pragma once

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
    void* o;
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
};

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
size_t split_workspace_bytes(const SplitPlan& plan);
// Points p's split-mode fields into a workspace laid out for plan.
void split_bind(const SplitPlan& plan, void* workspace, ChunkedParams* p);
cudaError_t launch_chunked_prefill(const ChunkedParams& p, cudaStream_t stream);
cudaError_t launch_split_prefill(const ChunkedParams& p, int num_sms, cudaStream_t stream);

}  // namespace kda
