// Host-side declarations shared by the library's translation units:
// kernel argument blocks, launchers, workspace layouts.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kv_common.cuh"

namespace kvb {

// Record a failed CUDA runtime call for kv_last_error (per host thread) and
// return KV_ECUDA.
int cuda_failed(cudaError_t err, const char* what);

#define KV_CUDA_CHECK(expr)                                              \
  do {                                                                   \
    const cudaError_t kv_err_ = (expr);                                  \
    if (kv_err_ != cudaSuccess) return ::kvb::cuda_failed(kv_err_, #expr); \
  } while (0)

// Launch through cudaLaunchKernelEx so the returned code is this launch's
// own (a bare <<<>>> launch is checked with cudaGetLastError, which also
// reports errors left behind by unrelated calls).  `pdl` allows programmatic
// dependent launch: the kernel may start while its predecessor on the
// stream finishes, and must call griddepcontrol.wait before touching that
// predecessor's outputs.
template <class... KArgs, class... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

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
};

size_t workqueue_smem_bytes(int B);
cudaError_t launch_build_workqueue(const WorkqueueArgs& a, cudaStream_t stream);

// Decode batches up to this many sequences compute their page offsets inside
// every decode CTA; larger ones take them from page_offsets_kernel.
constexpr int kFusedMaxB = 1024;

struct OffsetsArgs {
  const int32_t* seq_lens;
  int B, page_size, max_pages;
  int len_shift;      // lengths are taken as max(0, L - len_shift) (0: as given)
  int32_t* page_off;  // [B + 1]
  int* status;
};
cudaError_t launch_page_offsets(const OffsetsArgs& a, cudaStream_t stream);

// Smallest automatic split (pages): keeps merge traffic small on tiny batches.
constexpr int kMinChunk = 8;

// Decode workspace layout (offsets from the start of the workspace).
struct DecodeLayout {
  size_t row_done, group_done, page_off, part_o, part_lse, total;
  long long max_chunks, max_slots;
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

// Tensor-core attention of T * G <= 64 query rows per KV head (d = 128,
// page_size 16): one TMA-fed CTA per chunk of the batch's pages and a merge
// kernel.  Its scratch starts `region` bytes into the workspace (the status
// word stays at the workspace's start), so it can share a workspace with
// the decode kernel's merge tickets.
// Query tokens per pass of the tensor-core kernel (T * G <= 64 rows per KV
// head); 0 where the kernel does not apply.
int mma_attend_max_tokens(int Hq, int Hkv, int d);
bool mma_attend_supported(int Hq, int Hkv, int d, int Tq);
size_t mma_attend_workspace_size(int B, int Hkv, int rows, int d, int max_pages,
                                 int pages_per_split, size_t region);
// q, out and lse hold Tstride query tokens per sequence; this call serves Tq
// of them (from row 0 of the pointers passed), which see max(0, L - len_shift)
// cached tokens causally (decode: Tq = Tstride = 1, len_shift = 0).
int mma_attend_launch(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                      int Tq, int Tstride, int len_shift, int Hq, int Hkv, int d, int dtype,
                      float scale, int pages_per_split, float* out, float* lse, void* ws,
                      size_t ws_bytes, size_t region, cudaStream_t stream);

// One-shot profiling events for the next decode on this host thread.
void set_profile_events(cudaEvent_t before, cudaEvent_t after);
void take_profile_events(cudaEvent_t* before, cudaEvent_t* after);

// Failure-path test mode of the decode kernels (0 = off): every consumer
// warp first waits this many nanoseconds on a barrier nothing completes.
unsigned long long test_consumer_wait_ns();
void set_test_consumer_wait_ns(unsigned long long ns);

}  // namespace kvb
