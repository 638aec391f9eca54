// Device-side builder of the decode workqueue: the non-empty
// (sequence, KV-head, split) tasks of one decode step (PersistentKV,
// aissential.tech -- Summary and Method: a compact workqueue that executes
// only non-empty tasks).
//
// Split rule (this library's): the batch's non-empty pages are laid end to
// end (sequence offsets O_b), the range is cut into chunks of `chunk` pages
// and every (sequence, chunk) overlap is one split.  With the automatic chunk
// (ceil(W / workers), at least min_chunk) every decode worker streams the same
// number of pages whatever the length mix, and a sequence is split only where
// a worker boundary falls inside it.
//
// One CTA builds the whole queue.  Per-sequence arrays live in shared memory
// for batches up to kSmemSeqs sequences (global scratch beyond), so the build
// costs one read of seq_lens plus a few block-wide scans.  The decode kernel
// does not read this materialised queue: each decode CTA derives the tasks
// of its own chunks from the same page offsets and the same split helpers
// (kv_common.cuh), so the builder is the inspectable form of that queue.
// This file also holds the page-offset kernel large decode batches use.
#include "kv_internal.h"

namespace kvb {

namespace {

constexpr int kWqThreads = 1024;

// Largest b with gbeg[b] <= gi: the sequence that owns group gi (sequences
// without splits share their successor's begin and are skipped over).
__device__ int owner_of_group(const int32_t* gbeg, int B, long long gi) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (gbeg[mid] <= gi) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kWqThreads, 1) build_workqueue_kernel(WorkqueueArgs a) {
  // The decode kernel that follows may start its prologue now; it waits for
  // this grid to finish before reading the queue.
  pdl_launch_dependents();
  extern __shared__ long long wq_dyn[];
  __shared__ long long sm[32];
  const int tid = threadIdx.x, nth = blockDim.x;
  const bool in_smem = a.B <= kSmemSeqs;
  int32_t* np_arr = in_smem ? reinterpret_cast<int32_t*>(wq_dyn) : a.scratch_np;
  int32_t* gbeg = in_smem ? np_arr + a.B : a.seq_group_begin;
  int32_t* nspl = in_smem ? gbeg + a.B : a.seq_nsplit;
  long long* poff = in_smem ? reinterpret_cast<long long*>(wq_dyn) + ceil_div(3 * a.B, 2) + 1
                            : a.seq_page_off;
  const int per = ceil_div(a.B, nth);
  const int b0 = min(a.B, tid * per), b1 = min(a.B, b0 + per);

  // pass 1: pages per sequence (0 for an invalid length), page offsets
  long long my_pages = 0;
  bool bad = false;
  for (int b = b0; b < b1; ++b) {
    const int L = a.seq_lens[b];
    long long np = L > 0 ? ceil_div_ll(L, a.page_size) : 0;
    if (L < 0 || np > a.max_pages) {
      bad = true;
      np = 0;
    }
    np_arr[b] = (int32_t)np;
    my_pages += np;
  }
  if (bad) set_status(a.status, KV_EINVAL);
  long long page_off;
  const long long W = block_exclusive_scan(my_pages, &page_off, sm);
  const long long chunk = a.chunk_req > 0 ? a.chunk_req : auto_chunk(W, a.n_workers, a.min_chunk);
  const long long nchunks = W > 0 ? ceil_div_ll(W, chunk) : 0;

  // pass 2: splits per sequence
  long long my_groups = 0;
  {
    long long O = page_off;
    for (int b = b0; b < b1; ++b) {
      const long long np = np_arr[b];
      const long long ns = split_count(O, np, chunk);
      poff[b] = O;
      nspl[b] = (int32_t)ns;
      my_groups += ns;
      O += np;
    }
  }
  long long group_off;
  const long long G_total = block_exclusive_scan(my_groups, &group_off, sm);
  const long long T = G_total * a.Hkv;
  // On overflow nothing is emitted and every sequence reports zero splits, so
  // no consumer of the queue reads past the buffers.
  const bool overflow = T > a.max_tasks || nchunks + 1 > a.max_chunks ||
                        W > 0x7fffffffll || G_total > 0x7fffffffll;
  {
    long long g = group_off;
    for (int b = b0; b < b1; ++b) {
      const int ns = nspl[b];
      gbeg[b] = (int32_t)g;
      if (in_smem) {
        a.seq_group_begin[b] = overflow ? 0 : (int32_t)g;
        a.seq_nsplit[b] = overflow ? 0 : ns;
      } else if (overflow) {
        gbeg[b] = 0;
        nspl[b] = 0;
      }
      g += ns;
    }
  }
  __syncthreads();  // sequence arrays visible to the whole block
  if (overflow) {
    if (tid == 0) {
      set_status(a.status, KV_EWORKSPACE);
      a.meta[0] = 0; a.meta[1] = 0; a.meta[2] = (int32_t)chunk; a.meta[3] = 0; a.meta[4] = 0;
      if (a.max_chunks > 0) a.chunk_begin[0] = 0;
    }
    return;
  }

  // emission: one thread per task
  for (long long ti = tid; ti < T; ti += nth) {
    const long long gi = ti / a.Hkv;
    const int h = (int)(ti - gi * a.Hkv);
    const int b = owner_of_group(gbeg, a.B, gi);
    const int s = (int)(gi - gbeg[b]);
    const long long np = np_arr[b];
    const long long O = poff[b];
    const long long c = O / chunk + s;
    long long lo, hi;
    split_range(O, np, chunk, c, &lo, &hi);
    int4* rec = reinterpret_cast<int4*>(a.tasks + ti * 8);
    rec[0] = make_int4(b, h, s, nspl[b]);
    rec[1] = make_int4((int)lo, (int)hi, (int)c, a.seq_lens[b]);
    if (h == 0) {
      // chunk c' starts at this group for every c' in (cidx(gi-1), c]
      long long prev;
      if (gi == 0) {
        prev = -1;
      } else if (s > 0) {
        prev = c - 1;
      } else {
        const int pb = owner_of_group(gbeg, a.B, gi - 1);
        prev = (poff[pb] + np_arr[pb] - 1) / chunk;
      }
      for (long long cc = prev + 1; cc <= c; ++cc) a.chunk_begin[cc] = (int32_t)gi;
    }
  }
  if (tid == 0) {
    a.chunk_begin[nchunks] = (int32_t)G_total;
    a.meta[0] = (int32_t)T;
    a.meta[1] = (int32_t)G_total;
    a.meta[2] = (int32_t)chunk;
    a.meta[3] = (int32_t)nchunks;
    a.meta[4] = (int32_t)W;
  }
}

// Page offsets of the batch for decode calls too large to compute them in
// every decode CTA: page_off[b] = sum of ceil(L_b' / page_size) over b' < b,
// page_off[B] = total, with L = max(0, seq_lens[b] - len_shift).  Invalid
// lengths count as 0 pages and set KV_EINVAL; a total beyond int32 sets
// KV_EINVAL and yields an empty batch.
__global__ void __launch_bounds__(kWqThreads, 1) page_offsets_kernel(const OffsetsArgs a) {
  __shared__ long long sm[32];
  pdl_wait();  // seq_lens may come from the previous kernel on the stream
  pdl_launch_dependents();
  const int tid = threadIdx.x, nth = blockDim.x;
  const int per = ceil_div(a.B, nth);
  const int b0 = min(a.B, tid * per), b1 = min(a.B, b0 + per);
  long long mine = 0;
  bool bad = false;
  auto len = [&](int b) {
    const int L = a.seq_lens[b];
    return L < 0 ? L : max(0, L - a.len_shift);  // a negative length stays negative
  };
  for (int b = b0; b < b1; ++b) {
    const int L = len(b);
    long long np = L > 0 ? ceil_div_ll(L, a.page_size) : 0;
    if (L < 0 || np > a.max_pages) {
      bad = true;
      np = 0;
    }
    mine += np;
  }
  if (bad) set_status(a.status, KV_EINVAL);
  long long off;
  const long long W = block_exclusive_scan(mine, &off, sm);
  const bool overflow = W > 0x7fffffffll;
  if (overflow && tid == 0) set_status(a.status, KV_EINVAL);
  for (int b = b0; b < b1; ++b) {
    a.page_off[b] = overflow ? 0 : (int32_t)off;
    const int L = len(b);
    const long long np = L > 0 ? ceil_div_ll(L, a.page_size) : 0;
    if (L >= 0 && np <= a.max_pages) off += np;
  }
  if (tid == 0) a.page_off[a.B] = overflow ? 0 : (int32_t)W;
}

}  // namespace

cudaError_t launch_page_offsets(const OffsetsArgs& a, cudaStream_t stream) {
  return launch(page_offsets_kernel, dim3(1), dim3(kWqThreads), 0, stream, true, a);
}

size_t workqueue_smem_bytes(int B) {
  return B <= kSmemSeqs ? ((size_t)ceil_div(3 * B, 2) + 1 + B) * 8 : 0;
}

cudaError_t launch_build_workqueue(const WorkqueueArgs& a, cudaStream_t stream) {
  return launch(build_workqueue_kernel, dim3(1), dim3(kWqThreads), workqueue_smem_bytes(a.B), stream,
                false, a);
}

}  // namespace kvb
