// Host-side declarations shared by the library's translation units:
// kernel argument blocks, launchers, workspace layouts.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kv_common.cuh"

namespace kvb {

// Batches up to this many sequences keep the builder's arrays in shared memory.
constexpr int kSmemSeqs = 2048;

struct WorkqueueArgs {
  const int32_t* seq_lens;
  int B, Hkv, page_size, max_pages;
  long long chunk_req;   // > 0: fixed chunk; 0: automatic
  long long n_workers;   // decode workers the automatic chunk spreads over
  int min_chunk;
  int32_t* tasks;        // [max_tasks][8]
  long long max_tasks;
  int32_t* chunk_begin;  // [max_chunks]
  long long max_chunks;
  int32_t* seq_group_begin;  // [B]
  int32_t* seq_nsplit;       // [B]
  long long* seq_page_off;   // [B] scratch (used when B > kSmemSeqs)
  int32_t* scratch_np;       // [B] scratch (used when B > kSmemSeqs)
  int32_t* meta;             // [5]
  int* status;
  // decode call only (NULL otherwise)
  int32_t* row_done;  // [B * Hkv] split-merge completion counters, zeroed here
  float* out;         // [B][Hq][d]: rows of empty sequences set to 0
  float* lse;         // [B][Hq]:    rows of empty sequences set to -inf
  int Hq, d;
};

size_t workqueue_smem_bytes(int B);
cudaError_t launch_build_workqueue(const WorkqueueArgs& a, cudaStream_t stream);

// Smallest automatic split (pages): keeps merge traffic small on tiny batches.
constexpr int kMinChunk = 8;

// Decode workspace layout (offsets from the start of the workspace).
struct DecodeLayout {
  size_t tasks, chunk_begin, seq_group_begin, seq_nsplit, seq_page_off, scratch_np, row_done,
      meta, part_o, part_lse, total;
  long long max_tasks, max_chunks;
};
DecodeLayout decode_layout(int B, int Hq, int Hkv, int d, int max_pages, int page_size,
                           int pages_per_split, long long n_workers);

// Decode entry used by both the device-pointer and the host-IO calls.
int decode_launch(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                  const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                  int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                  int pages_per_split, float* out, float* lse, void* ws, size_t ws_bytes,
                  cudaStream_t stream);
int decode_num_workers(int Hq, int Hkv, int d, int page_size, int dtype);

// One-shot profiling events for the next decode on this host thread.
void set_profile_events(cudaEvent_t before, cudaEvent_t after);
void take_profile_events(cudaEvent_t* before, cudaEvent_t* after);

}  // namespace kvb
