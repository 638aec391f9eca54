// C ABI entry points: status handling, decode (device and host buffers), and
// the stand-alone workqueue builder.  Argument checks happen here, on the
// host, before anything is enqueued.
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "kv_internal.h"

namespace kvb {
namespace {

// Up to three byte ranges copied by one kernel (each a multiple of 4 bytes,
// 4-byte aligned; 16-byte words where both ends allow).  Used to move the
// host-buffer call's inputs and outputs through mapped host memory: one
// launch instead of one DMA operation per buffer.
struct CopySegs {
  const void* src[3];
  void* dst[3];
  size_t bytes[3];
  int n;
};

__global__ void __launch_bounds__(256) segs_copy_kernel(const CopySegs c) {
  pdl_wait();  // the sources may come from the previous kernel on the stream
  pdl_launch_dependents();
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t nth = (size_t)gridDim.x * blockDim.x;
  for (int k = 0; k < c.n; ++k) {
    const uintptr_t s = reinterpret_cast<uintptr_t>(c.src[k]), d = reinterpret_cast<uintptr_t>(c.dst[k]);
    if (((s | d | c.bytes[k]) & 15) == 0) {
      const uint4* src = reinterpret_cast<const uint4*>(s);
      uint4* dst = reinterpret_cast<uint4*>(d);
      for (size_t i = tid; i < c.bytes[k] / 16; i += nth) dst[i] = src[i];
    } else {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(s);
      uint32_t* dst = reinterpret_cast<uint32_t*>(d);
      for (size_t i = tid; i < c.bytes[k] / 4; i += nth) dst[i] = src[i];
    }
  }
}

cudaError_t launch_segs_copy(const CopySegs& c, cudaStream_t s) {
  size_t total = 0;
  for (int k = 0; k < c.n; ++k) total += c.bytes[k];
  const size_t words = (total + 15) / 16;
  const unsigned blocks = (unsigned)std::min<size_t>(148 * 4, std::max<size_t>(1, (words + 255) / 256));
  return launch(segs_copy_kernel, dim3(blocks), dim3(256), 0, s, true, c);
}

// Reads n16 16-byte words through L2 (used by the calibration's L2 flush, on
// the half of the flush buffer that the preceding memset already pushed out
// of L2): the lines it brings in are clean, so the dirty lines the memset
// left behind are written back here rather than inside the next timed call.
// A store to *sink depends on the xor of what was read, so the loads cannot
// be dropped.
__global__ void __launch_bounds__(256) l2_clean_kernel(const uint4* src, size_t n16, uint4* sink) {
  uint4 x = make_uint4(0u, 0u, 0u, 0u);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint4 v = __ldcg(src + i);
    x.x ^= v.x;
    x.y ^= v.y;
    x.z ^= v.z;
    x.w ^= v.w;
  }
  if ((x.x | x.y | x.z | x.w) == 0x9e3779b9u) *sink = x;  // practically never; keeps the loads
}

}  // namespace
}  // namespace kvb

using namespace kvb;

namespace kvb {
namespace {
thread_local char t_last_error[256] = "";
}
int cuda_failed(cudaError_t err, const char* what) {
  snprintf(t_last_error, sizeof t_last_error, "%s: %s (%s, %d)", what, cudaGetErrorString(err),
           cudaGetErrorName(err), (int)err);
  // A failed call leaves its (non-sticky) error pending in the runtime; it is
  // reported here, so clear it rather than let the caller's next CUDA call
  // pick it up.
  (void)cudaGetLastError();
  return KV_ECUDA;
}
}  // namespace kvb

extern "C" {

const char* kv_last_error(void) { return t_last_error; }

const char* kv_status_string(int code) {
  switch (code) {
    case KV_OK: return "ok";
    case KV_EINVAL: return "invalid argument";
    case KV_EBADPAGE: return "page id outside the pool";
    case KV_ENOSPACE: return "free list exhausted";
    case KV_EWORKSPACE: return "workspace too small";
    case KV_ECUDA: return "CUDA runtime error";
    case KV_EFULL: return "block-table row full";
    case KV_ETIMEOUT: return "kernel wait timed out";
    default: return "unknown status";
  }
}

size_t kv_status_workspace_size(void) { return kHeaderBytes; }

int kv_workspace_reset(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < kHeaderBytes) return KV_EINVAL;
  KV_CUDA_CHECK(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
  return KV_OK;
}

int kv_get_status(void* ws, void* stream) {
  if (!ws) return KV_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  KV_CUDA_CHECK(cudaMemcpyAsync(&host, ws, sizeof(int), cudaMemcpyDeviceToHost, s));
  KV_CUDA_CHECK(cudaStreamSynchronize(s));
  if (host != 0) {
    KV_CUDA_CHECK(cudaMemsetAsync(ws, 0, sizeof(int), s));
    KV_CUDA_CHECK(cudaStreamSynchronize(s));
  }
  return host;
}

int kv_decode_num_workers(int Hq, int Hkv, int d, int page_size, int dtype) {
  return decode_num_workers(Hq, Hkv, d, page_size, dtype);
}

namespace {

int decode_workers_both(int Hq, int Hkv, int d, int page_size) {
  // the worker count can differ between the fp16 and bf16 kernels: size for both
  return std::max(decode_num_workers(Hq, Hkv, d, page_size, KV_F16),
                  decode_num_workers(Hq, Hkv, d, page_size, KV_BF16));
}

bool tensor_core_ok(int page_size, int Hq, int Hkv, int d) {
  return page_size == 16 && mma_attend_supported(Hq, Hkv, d, 1);
}

// Where the tensor-core engine's scratch starts inside a decode workspace:
// past the decode kernel's merge tickets for every split size (the finest
// split, one page, has the most) and past its whole automatic-split layout,
// so the two engines can take turns on one workspace (as kv_decode_tune
// does) without touching each other's state.  Shapes the fused kernel does
// not support need no room for it.
size_t tensor_core_region(int B, int Hq, int Hkv, int d, int max_pages, int page_size) {
  const int nw = decode_workers_both(Hq, Hkv, d, page_size);
  if (nw <= 0) return kHeaderBytes;
  const DecodeLayout a = decode_layout(B, Hq, Hkv, d, max_pages, page_size, 0, nw);
  const DecodeLayout f = decode_layout(B, Hq, Hkv, d, max_pages, page_size, 1, nw);
  return align_up(std::max(a.total, f.page_off), 256);
}

// One decode step with the engine `pages_per_split` names: >= 0 the fused
// decode kernel with that split size, KV_DECODE_TENSOR_CORE the tensor-core
// engine (automatic split).
int engine_launch(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                  const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                  int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                  int pages_per_split, float* out, float* lse, void* ws, size_t ws_bytes,
                  cudaStream_t s) {
  if (pages_per_split != KV_DECODE_TENSOR_CORE)
    return decode_launch(q, k_pool, v_pool, num_pages, block_table, max_pages, seq_lens, B,
                         page_size, Hq, Hkv, d, dtype, scale, pages_per_split, out, lse, ws,
                         ws_bytes, s);
  if (B < 0 || max_pages < 0 || Hq <= 0 || Hkv <= 0) return KV_EINVAL;
  if (!tensor_core_ok(page_size, Hq, Hkv, d)) return KV_EINVAL;
  if (B == 0) return KV_OK;
  const size_t region = tensor_core_region(B, Hq, Hkv, d, max_pages, page_size);
  if (!region) return KV_EINVAL;
  return mma_attend_launch(q, k_pool, v_pool, num_pages, block_table, max_pages, seq_lens, B, 1,
                           1, 0, Hq, Hkv, d, dtype, scale, 0, out, lse, ws, ws_bytes, region, s);
}

}  // namespace

size_t kv_decode_workspace_size(int B, int Hq, int Hkv, int d, int max_pages, int page_size,
                                int pages_per_split) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || max_pages < 0) return 0;
  if (pages_per_split == KV_DECODE_TENSOR_CORE) {
    if (!tensor_core_ok(page_size, Hq, Hkv, d)) return 0;
    const size_t region = tensor_core_region(B, Hq, Hkv, d, max_pages, page_size);
    return region ? mma_attend_workspace_size(B, Hkv, Hq / Hkv, d, max_pages, 0, region) : 0;
  }
  if (pages_per_split < 0) return 0;
  const int nw = decode_workers_both(Hq, Hkv, d, page_size);
  if (nw <= 0) return 0;
  return decode_layout(B, Hq, Hkv, d, max_pages, page_size, pages_per_split, nw).total;
}

int kv_decode(const void* q, const void* k_pool, const void* v_pool, int num_pages,
              const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
              int page_size, int Hq, int Hkv, int d, int dtype, float scale, int pages_per_split,
              float* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
  return engine_launch(q, k_pool, v_pool, num_pages, block_table, max_pages, seq_lens, B,
                       page_size, Hq, Hkv, d, dtype, scale, pages_per_split, out, lse, ws, ws_bytes,
                       static_cast<cudaStream_t>(stream));
}

namespace {

// Device address of a host buffer the GPU can reach directly (page-locked
// and mapped, as every pinned allocation is under unified addressing), or
// null for pageable memory.
void* mapped_host(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // pageable memory on older runtimes reports an error
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

struct HostIoLayout {
  size_t q, table, seq_lens, out, lse, total;
};
HostIoLayout hostio_layout(size_t base, int B, int Hq, int d, int max_pages) {
  HostIoLayout L{};
  size_t off = align_up(base, 256);
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.q = take((size_t)B * Hq * d * 2);
  L.table = take((size_t)B * max_pages * 4);
  L.seq_lens = take((size_t)B * 4);
  L.out = take((size_t)B * Hq * d * 4);
  L.lse = take((size_t)B * Hq * 4);
  L.total = off;
  return L;
}
}  // namespace

size_t kv_decode_hostio_workspace_size(int B, int Hq, int Hkv, int d, int max_pages, int page_size,
                                       int pages_per_split) {
  const size_t base = kv_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size, pages_per_split);
  if (!base) return 0;
  return hostio_layout(base, B, Hq, d, max_pages).total;
}

int kv_decode_hostio(const void* h_q, const void* k_pool, const void* v_pool, int num_pages,
                     const int32_t* h_block_table, int max_pages, const int32_t* h_seq_lens, int B,
                     int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                     int pages_per_split, float* h_out, float* h_lse, void* ws, size_t ws_bytes,
                     void* stream) {
  if (B < 0 || max_pages < 0) return KV_EINVAL;
  if (B == 0) return KV_OK;
  if (!h_q || !h_block_table || !h_seq_lens || !h_out || !h_lse || !ws) return KV_EINVAL;
  const size_t base = kv_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size, pages_per_split);
  if (!base) return KV_EINVAL;
  const HostIoLayout L = hostio_layout(base, B, Hq, d, max_pages);
  if (ws_bytes < L.total) return KV_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t qb = (size_t)B * Hq * d * 2, tb = (size_t)B * max_pages * 4, sb = (size_t)B * 4;
  const size_t ob = (size_t)B * Hq * d * 4, lb = (size_t)B * Hq * 4;
  // pinned host buffers are read and written in place by copy kernels;
  // pageable ones take one cudaMemcpyAsync each
  void* m_q = mapped_host(h_q);
  void* m_t = mapped_host(h_block_table);
  void* m_l = mapped_host(h_seq_lens);
  void* m_o = mapped_host(h_out);
  void* m_s = mapped_host(h_lse);
  const bool in_mapped = m_q && m_t && m_l && !((uintptr_t)m_q & 3) && !((uintptr_t)m_t & 3) &&
                         !((uintptr_t)m_l & 3);
  // the kernels store out with 16-byte writes
  const bool out_direct = m_o && m_s && !((uintptr_t)m_o & 15) && !((uintptr_t)m_s & 3);
  if (in_mapped) {
    CopySegs c{};
    c.src[0] = m_q; c.dst[0] = w + L.q; c.bytes[0] = qb;
    c.src[1] = m_t; c.dst[1] = w + L.table; c.bytes[1] = tb;
    c.src[2] = m_l; c.dst[2] = w + L.seq_lens; c.bytes[2] = sb;
    c.n = 3;
    KV_CUDA_CHECK(launch_segs_copy(c, s));
  } else {
    KV_CUDA_CHECK(cudaMemcpyAsync(w + L.q, h_q, qb, cudaMemcpyHostToDevice, s));
    KV_CUDA_CHECK(cudaMemcpyAsync(w + L.table, h_block_table, tb, cudaMemcpyHostToDevice, s));
    KV_CUDA_CHECK(cudaMemcpyAsync(w + L.seq_lens, h_seq_lens, sb, cudaMemcpyHostToDevice, s));
  }
  // Page-locked outputs are written in place by the decode kernels (the
  // device addresses host memory directly; the writes are visible to the
  // host once the stream has reached them); others are staged.
  float* dev_out = out_direct ? static_cast<float*>(m_o) : reinterpret_cast<float*>(w + L.out);
  float* dev_lse = out_direct ? static_cast<float*>(m_s) : reinterpret_cast<float*>(w + L.lse);
  int rc = engine_launch(w + L.q, k_pool, v_pool, num_pages,
                         reinterpret_cast<const int32_t*>(w + L.table), max_pages,
                         reinterpret_cast<const int32_t*>(w + L.seq_lens), B, page_size, Hq, Hkv, d,
                         dtype, scale, pages_per_split, dev_out, dev_lse, ws, base, s);
  if (rc) return rc;
  if (!out_direct) {
    KV_CUDA_CHECK(cudaMemcpyAsync(h_out, w + L.out, ob, cudaMemcpyDeviceToHost, s));
    KV_CUDA_CHECK(cudaMemcpyAsync(h_lse, w + L.lse, lb, cudaMemcpyDeviceToHost, s));
  }
  return KV_OK;
}

int kv_build_workqueue(const int32_t* seq_lens, int B, int Hkv, int page_size, int max_pages,
                       int pages_per_split, int n_workers, int32_t* tasks, int max_tasks,
                       int32_t* chunk_begin, int max_chunks, int32_t* seq_group_begin,
                       int32_t* seq_nsplit, int32_t* meta, void* ws, void* stream) {
  if (B < 0 || Hkv <= 0 || page_size <= 0 || max_pages < 0 || pages_per_split < 0 ||
      max_tasks < 0 || max_chunks < 1)
    return KV_EINVAL;
  if (pages_per_split == 0 && n_workers <= 0) return KV_EINVAL;
  if (!tasks || !chunk_begin || !meta || !ws || (B > 0 && (!seq_lens || !seq_group_begin || !seq_nsplit)))
    return KV_EINVAL;
  if (((uintptr_t)tasks & 15) || ((uintptr_t)ws & 255)) return KV_EINVAL;
  // scratch for per-sequence page offsets lives after the workspace header
  WorkqueueArgs a{};
  a.seq_lens = seq_lens;
  a.B = B;
  a.Hkv = Hkv;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.chunk_req = pages_per_split;
  a.n_workers = n_workers;
  a.min_chunk = kMinChunk;
  a.tasks = tasks;
  a.max_tasks = max_tasks;
  a.chunk_begin = chunk_begin;
  a.max_chunks = max_chunks;
  a.seq_group_begin = seq_group_begin;
  a.seq_nsplit = seq_nsplit;
  a.seq_page_off = reinterpret_cast<long long*>(static_cast<uint8_t*>(ws) + kHeaderBytes);
  a.scratch_np = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + kHeaderBytes +
                                            align_up((size_t)(B > 0 ? B : 1) * 8, 256));
  a.meta = meta;
  a.status = static_cast<int*>(ws);
  KV_CUDA_CHECK(launch_build_workqueue(a, static_cast<cudaStream_t>(stream)));
  return KV_OK;
}

int kv_decode_tune(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                   const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                   int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                   const int32_t* candidates, int n_candidates, int reps, float* out, float* lse,
                   float* us, int32_t* best, void* ws, size_t ws_bytes, void* flush,
                   size_t flush_bytes, void* stream) {
  if (!candidates || n_candidates < 1 || reps < 1 || !us || !best) return KV_EINVAL;
  if (!flush) flush_bytes = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // read-back part of the flush: the first half of the buffer, 16-byte words
  const uintptr_t flush_base = align_up(reinterpret_cast<uintptr_t>(flush), 16);
  const uintptr_t flush_end = reinterpret_cast<uintptr_t>(flush) + flush_bytes;
  const size_t clean_n16 =
      flush_bytes && flush_end >= flush_base + 64 ? (flush_end - flush_base) / 32 : 0;
  int clean_blocks = 0;
  if (clean_n16) {
    int dev = 0, sms = 0;
    KV_CUDA_CHECK(cudaGetDevice(&dev));
    KV_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    clean_blocks = sms * 8;
  }
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  KV_CUDA_CHECK(cudaEventCreate(&e0));
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return cuda_failed(cudaErrorUnknown, "cudaEventCreate");
  }
  int rc = KV_OK;
  int best_i = 0;
  for (int c = 0; c < n_candidates && rc == KV_OK; ++c) {
    float times[64];
    const int n = reps < 64 ? reps : 64;
    // one untimed call first (launch shape set-up, caches)
    rc = engine_launch(q, k_pool, v_pool, num_pages, block_table, max_pages, seq_lens, B,
                       page_size, Hq, Hkv, d, dtype, scale, candidates[c], out, lse, ws, ws_bytes,
                       s);
    for (int r = 0; r < n && rc == KV_OK; ++r) {
      // the L2 flush (when asked for) stays outside the timed events: the
      // whole buffer overwritten, then its first half read back so that the
      // lines left in L2 are clean ones
      if (flush_bytes && cudaMemsetAsync(flush, r & 0xff, flush_bytes, s) != cudaSuccess) {
        rc = cuda_failed(cudaErrorUnknown, "cudaMemsetAsync (L2 flush)");
        break;
      }
      if (clean_n16 &&
          launch(l2_clean_kernel, dim3(clean_blocks), dim3(256), 0, s, false,
                 reinterpret_cast<const uint4*>(flush_base), clean_n16,
                 reinterpret_cast<uint4*>(flush_base) + (flush_end - flush_base) / 16 - 1) !=
              cudaSuccess) {
        rc = cuda_failed(cudaErrorUnknown, "L2 flush read-back");
        break;
      }
      if (cudaEventRecord(e0, s) != cudaSuccess) { rc = cuda_failed(cudaErrorUnknown, "cudaEventRecord"); break; }
      rc = engine_launch(q, k_pool, v_pool, num_pages, block_table, max_pages, seq_lens, B,
                         page_size, Hq, Hkv, d, dtype, scale, candidates[c], out, lse, ws,
                         ws_bytes, s);
      if (rc) break;
      if (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
          cudaEventElapsedTime(&times[r], e0, e1) != cudaSuccess) {
        rc = cuda_failed(cudaErrorUnknown, "timing events");
        break;
      }
    }
    if (rc) break;
    // mean of the middle half of the sorted times: as robust as the median
    // to a stray slow call, and finer than one event reading (elapsed times
    // come in steps of about 2 us here, which made close candidates tie)
    std::sort(times, times + n);
    const int lo = n / 4, hi = n - n / 4;
    float sum = 0.f;
    for (int i = lo; i < hi; ++i) sum += times[i];
    us[c] = sum / (float)(hi - lo) * 1e3f;
    if (us[c] < us[best_i]) best_i = c;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (rc == KV_OK) *best = candidates[best_i];
  return rc;
}

int kv_test_consumer_timeout(unsigned long long ns) {
  set_test_consumer_wait_ns(ns);
  return KV_OK;
}

int kv_profile_next_decode(void* event_before, void* event_after) {
  set_profile_events(static_cast<cudaEvent_t>(event_before), static_cast<cudaEvent_t>(event_after));
  return KV_OK;
}

size_t kv_workqueue_workspace_size(int B) {
  const size_t nb = (size_t)(B > 0 ? B : 1);
  return kHeaderBytes + align_up(nb * 8, 256) + align_up(nb * 4, 256);
}

}  // extern "C"
