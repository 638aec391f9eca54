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
// costs one read of seq_lens plus a few block-wide scans.  For a decode call it
// also zeroes the per-(sequence, KV head) completion counters the decode
// kernel's split merge uses, and writes out = 0 / lse = -inf for sequences
// with no tokens (the decode kernel never visits them).
#include "kv_internal.h"

namespace kvb {

namespace {

constexpr int kWqThreads = 1024;

// Exclusive block-wide scan of one value per thread; returns the total.
__device__ long long block_exclusive_scan(long long v, long long* out_excl, long long* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nwarps ? sm[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nwarps) sm[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  long long base = warp > 0 ? sm[warp - 1] : 0;
  *out_excl = base + x - v;
  long long total = sm[nwarps - 1];
  __syncthreads();
  return total;
}

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
  long long chunk = a.chunk_req > 0 ? a.chunk_req
                                    : max((long long)a.min_chunk, ceil_div_ll(W, a.n_workers));
  if (chunk < 1) chunk = 1;
  const long long nchunks = W > 0 ? ceil_div_ll(W, chunk) : 0;

  // pass 2: splits per sequence
  long long my_groups = 0;
  {
    long long O = page_off;
    for (int b = b0; b < b1; ++b) {
      const long long np = np_arr[b];
      const long long ns = np > 0 ? (O + np - 1) / chunk - O / chunk + 1 : 0;
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
  // decode only: completion counters of the split merge, empty-sequence outputs
  if (a.row_done)
    for (long long i = tid; i < (long long)a.B * a.Hkv; i += nth) a.row_done[i] = 0;
  if (a.out) {
    const int per_seq = a.Hq * a.d;
    for (int b = 0; b < a.B; ++b) {
      if (np_arr[b] != 0 && !overflow) continue;
      for (int i = tid; i < per_seq; i += nth) a.out[(size_t)b * per_seq + i] = 0.f;
      for (int i = tid; i < a.Hq; i += nth) a.lse[(size_t)b * a.Hq + i] = -INFINITY;
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
    const long long lo = max(O, c * chunk) - O;
    const long long hi = min(O + np, (c + 1) * chunk) - O;
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

}  // namespace

size_t workqueue_smem_bytes(int B) {
  return B <= kSmemSeqs ? ((size_t)ceil_div(3 * B, 2) + 1 + B) * 8 : 0;
}

cudaError_t launch_build_workqueue(const WorkqueueArgs& a, cudaStream_t stream) {
  build_workqueue_kernel<<<1, kWqThreads, workqueue_smem_bytes(a.B), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvb
