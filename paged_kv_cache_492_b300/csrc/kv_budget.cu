// Page budgeting (GrowPage, mlsanity.com -- Abstract; aitrending.vip summary
// -- Technical Details): query summaries at two time scales, page key summaries,
// page scores, top-k retention with compress-or-grow at capacity boundaries,
// compaction of the block table (and K/V for token-granular masks), and the
// per-token append that draws pages from the integer free list (Elastic KV
// Cache, paperlayer.ai -- section 2).
//
// Every floating-point value that decides an integer (EMAs, summaries,
// scores, the drift threshold) is computed in fp32 with explicitly rounded
// operations (__fadd_rn / __fmul_rn / __fdiv_rn, no contraction) in the order
// stated in include/kv.h, so selections are reproducible bit for bit.
#include <math.h>

#include <algorithm>

#include "kv_internal.h"

namespace kvb {
namespace {

constexpr unsigned FULL = 0xffffffffu;

template <class T>
__device__ __forceinline__ float ld16(const uint16_t* p, size_t i) {
  return T::to_f(p[i]);
}

// ------------------------------------------------------------------ EMA
template <class T>
__global__ void ema_kernel(const uint16_t* __restrict__ q, int Hq, int Hkv, int d, float a_fast,
                           float a_slow, int first, float* __restrict__ ema) {
  const int b = blockIdx.x / Hkv, h = blockIdx.x - b * Hkv;
  const int G = Hq / Hkv;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float acc = 0.0f;
    for (int g = 0; g < G; ++g)
      acc = __fadd_rn(acc, ld16<T>(q, ((size_t)b * Hq + (size_t)h * G + g) * d + c));
    const float gm = __fdiv_rn(acc, (float)G);
    for (int u = 0; u < 2; ++u) {
      float* e = ema + (((size_t)b * 2 + u) * Hkv + h) * d + c;
      const float a = u == 0 ? a_fast : a_slow;
      *e = first ? gm : __fadd_rn(__fmul_rn(a, *e), __fmul_rn(__fsub_rn(1.0f, a), gm));
    }
  }
}

// ------------------------------------------------------------------ boundary marks
__global__ void mark_kernel(const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ budget,
                            int B, int ps, int mode, uint8_t* __restrict__ active) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const long long L = seq_lens[b];
  if (mode == 0)
    active[b] = ceil_div_ll(L, ps) > budget[b];
  else
    active[b] = L > 0 && L % ps == 0 && L / ps >= budget[b];
}

// ------------------------------------------------------------------ page summaries
// One block per (listed page, KV head); thread c: mean/min/max over the page's slots.
template <class T>
__global__ void summary_kernel(const uint16_t* __restrict__ k_pool, int num_pages,
                               const int32_t* __restrict__ page_ids, int n,
                               const int32_t* __restrict__ table, int max_pages,
                               const int32_t* __restrict__ seq_lens,
                               const uint8_t* __restrict__ active, int Hkv, int ps, int d,
                               float* __restrict__ summ, int* status) {
  const int i = blockIdx.x / Hkv, h = blockIdx.x - i * Hkv;
  int page;
  if (page_ids) {
    page = page_ids[i];
  } else {
    // last full page of an active sequence
    if (active && !active[i]) return;
    const int L = seq_lens[i];
    if (L < ps) return;
    page = table[(size_t)i * max_pages + (L / ps - 1)];
  }
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0) set_status(status, KV_EBADPAGE);
    return;
  }
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float acc = 0.0f, mn = INFINITY, mx = -INFINITY;
    for (int t = 0; t < ps; ++t) {
      const float x = ld16<T>(k_pool, (((size_t)page * Hkv + h) * ps + t) * d + c);
      acc = __fadd_rn(acc, x);
      mn = x < mn ? x : mn;
      mx = x > mx ? x : mx;
    }
    float* s = summ + ((size_t)page * Hkv + h) * 3 * d;
    s[c] = __fdiv_rn(acc, (float)ps);
    s[d + c] = mn;
    s[2 * d + c] = mx;
  }
}

// ------------------------------------------------------------------ scores
// One warp per (sequence, logical page); lane l owns channels l*CPL.. of every head.
template <int CPL>
__global__ void score_kernel(const float* __restrict__ ema, const float* __restrict__ summ,
                             int num_pages, const int32_t* __restrict__ table, int max_pages,
                             const int32_t* __restrict__ seq_lens, const uint8_t* __restrict__ active,
                             int B, int Hkv, int ps, float* __restrict__ scores, int* status) {
  constexpr int d = 32 * CPL;
  const int lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= (long long)B * max_pages) return;
  const int b = (int)(wid / max_pages), j = (int)(wid - (long long)b * max_pages);
  if (active && !active[b]) return;
  float2* out = reinterpret_cast<float2*>(scores + ((size_t)b * max_pages + j) * 2);
  const long long np = ceil_div_ll(seq_lens[b], ps);
  if (j >= np) {
    if (lane == 0) *out = make_float2(-INFINITY, -INFINITY);
    return;
  }
  const int page = table[(size_t)b * max_pages + j];
  if (page < 0 || page >= num_pages) {
    if (lane == 0) set_status(status, KV_EBADPAGE);
    return;
  }
  float af = 0.0f, as = 0.0f;
  for (int h = 0; h < Hkv; ++h) {
    const float* uf = ema + (((size_t)b * 2 + 0) * Hkv + h) * d + lane * CPL;
    const float* us = ema + (((size_t)b * 2 + 1) * Hkv + h) * d + lane * CPL;
    const float* sm = summ + ((size_t)page * Hkv + h) * 3 * d + lane * CPL;
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const float mu = sm[i], mn = sm[d + i], mx = sm[2 * d + i];
      {
        const float u = uf[i];
        const float ta = __fmul_rn(u, mn), tb = __fmul_rn(u, mx);
        af = __fadd_rn(af, __fadd_rn(__fmul_rn(u, mu), ta > tb ? ta : tb));
      }
      {
        const float u = us[i];
        const float ta = __fmul_rn(u, mn), tb = __fmul_rn(u, mx);
        as = __fadd_rn(as, __fadd_rn(__fmul_rn(u, mu), ta > tb ? ta : tb));
      }
    }
  }
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    af = __fadd_rn(af, __shfl_xor_sync(FULL, af, s));
    as = __fadd_rn(as, __shfl_xor_sync(FULL, as, s));
  }
  if (lane == 0) *out = make_float2(af, as);
}

// ------------------------------------------------------------------ selection
constexpr int kSelThreads = 1024;
constexpr int kMaxSelectPages = 8192;

__device__ __forceinline__ int block_sum_int(int v, int* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  __syncthreads();
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  int t = 0;
  for (int w = 0; w < nw; ++w) t += sm[w];
  __syncthreads();
  return t;
}

// rank of candidate j among candidates by key (larger first, ties: lower index)
__device__ __forceinline__ int rank_of(const float* key, const uint8_t* is_cand, int n, int j) {
  const float kj = key[j];
  int r = 0;
  for (int i = 0; i < n; ++i) r += is_cand[i] && (key[i] > kj || (key[i] == kj && i < j));
  return r;
}

// The order rank_of counts in: candidates first, then the larger key, then
// the lower index (equal keys, -0 and +0 included, tie on the index);
// non-candidates and padding after, by index.  A strict total order when no
// candidate key is NaN.
__device__ __forceinline__ bool rank_before(const float* key, const uint8_t* is_cand, int n, int x,
                                            int y) {
  const bool cx = x < n && is_cand[x], cy = y < n && is_cand[y];
  if (cx != cy) return cx;
  if (cx) {
    const float kx = key[x], ky = key[y];
    if (kx > ky) return true;
    if (kx < ky) return false;
  }
  return x < y;
}

// rank[j] = rank_of(key, is_cand, n, j) for every candidate j.  Up to 1024
// pages: the counting definition itself, spread over the block -- a group
// of up to 32 lanes per candidate counts a strided share of the keys and
// the group sums by shuffles (the same indicator sum, so the same result,
// NaN keys included).  Longer rows: a block-wide bitonic sort of the indices
// (idx holds next_pow2(n) entries) in rank_before's order; with a NaN key
// among the candidates that order is not total and the counting definition
// is applied directly instead.
__device__ void rank_candidates(const float* key, const uint8_t* is_cand, int n, uint16_t* idx,
                                uint16_t* rank) {
  if (n <= 1024) {
    int tpc = 1;  // lanes per candidate
    while (tpc < 32 && tpc * 2 * n <= (int)blockDim.x) tpc <<= 1;
    const int per_pass = blockDim.x / tpc, sub = threadIdx.x & (tpc - 1);
    for (int j0 = 0; j0 < n; j0 += per_pass) {
      const int j = j0 + threadIdx.x / tpc;
      const bool mine = j < n && is_cand[j];
      int r = 0;
      if (mine) {
        const float kj = key[j];
        for (int i = sub; i < n; i += tpc) r += is_cand[i] && (key[i] > kj || (key[i] == kj && i < j));
      }
      for (int o = tpc >> 1; o; o >>= 1) r += __shfl_xor_sync(FULL, r, o);
      if (mine && sub == 0) rank[j] = (uint16_t)r;
    }
    __syncthreads();
    return;
  }
  int bad = 0;
  for (int j = threadIdx.x; j < n; j += blockDim.x) bad |= is_cand[j] && isnan(key[j]);
  if (__syncthreads_or(bad)) {
    for (int j = threadIdx.x; j < n; j += blockDim.x)
      if (is_cand[j]) rank[j] = (uint16_t)rank_of(key, is_cand, n, j);
    __syncthreads();
    return;
  }
  int P2 = 1;
  while (P2 < n) P2 <<= 1;
  for (int i = threadIdx.x; i < P2; i += blockDim.x) idx[i] = (uint16_t)i;
  __syncthreads();
  for (int k = 2; k <= P2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P2; i += blockDim.x) {
        const int l = i ^ j;
        if (l > i) {
          const int x = idx[i], y = idx[l];
          const bool asc = (i & k) == 0;
          if (asc ? rank_before(key, is_cand, n, y, x) : rank_before(key, is_cand, n, x, y)) {
            idx[i] = (uint16_t)y;
            idx[l] = (uint16_t)x;
          }
        }
      }
      __syncthreads();
    }
  }
  // candidates come first, in rank order
  for (int p = threadIdx.x; p < P2; p += blockDim.x) {
    const int j = idx[p];
    if (j < n && is_cand[j]) rank[j] = (uint16_t)p;
  }
  __syncthreads();
}

struct SelectArgs {
  const float* scores;
  const int32_t* seq_lens;
  const uint8_t* active;
  int32_t* budget;
  int B, max_pages, ps, n_first, n_last, mode;
  float delta, ws_frac;
  uint8_t* keep;
  uint8_t* grow;
  int32_t* drift;
  int32_t* wants;  // [B] workspace
  int* status;
};

// One row (one block): ranks, drift and the compaction keep set of sequence
// b; writes keep[b], drift[b], grow[b] = 0, and returns (on every thread)
// whether the row wants to grow.  Inactive rows keep every page.
__device__ int select_row(const SelectArgs& a, int b, float* sel_sm, int* red) {
  const int n = (int)ceil_div_ll(a.seq_lens[b], a.ps);
  uint8_t* keep = a.keep + (size_t)b * a.max_pages;
  const bool act = a.active ? a.active[b] != 0 : true;
  if (threadIdx.x == 0) {
    a.grow[b] = 0;
    if (a.drift) a.drift[b] = 0;
  }
  if (!act || n > a.max_pages) {
    if (n > a.max_pages && threadIdx.x == 0) set_status(a.status, KV_EINVAL);
    for (int j = threadIdx.x; j < a.max_pages; j += blockDim.x) keep[j] = j < n;
    return 0;
  }
  float* sf = sel_sm;
  float* ss = sf + n;
  float* rr = ss + n;
  uint16_t* idx = reinterpret_cast<uint16_t*>(rr + n);  // [next_pow2(n)]
  int P2 = 1;
  while (P2 < n) P2 <<= 1;
  uint16_t* rank = idx + P2;                               // [n]
  uint8_t* in_f = reinterpret_cast<uint8_t*>(rank + n);    // [n]
  uint8_t* cand = in_f + n;                                // [n]
  int my_forced = 0;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const float2 s = reinterpret_cast<const float2*>(a.scores + (size_t)b * a.max_pages * 2)[j];
    sf[j] = s.x;
    ss[j] = s.y;
    rr[j] = __fadd_rn(s.x, s.y);
    const bool forced = j < a.n_first || j >= n - a.n_last;
    cand[j] = !forced;
    my_forced += forced;
  }
  __syncthreads();
  const int nf = block_sum_int(my_forced, red);
  const int nc = n - nf;
  int k;
  int wants = 0;
  if (a.mode == KV_SELECT_TOPK) {
    k = a.budget[b] - nf;
  } else {
    k = n - 1 - nf;
    if (nc == 0) {
      wants = 1;
    } else {
      int w = (int)ceilf(__fmul_rn(a.ws_frac, (float)nc));
      w = max(1, min(w, nc));
      rank_candidates(sf, cand, n, idx, rank);
      for (int j = threadIdx.x; j < n; j += blockDim.x) in_f[j] = cand[j] && rank[j] < w;
      __syncthreads();
      rank_candidates(ss, cand, n, idx, rank);
      int my_d = 0;
      for (int j = threadIdx.x; j < n; j += blockDim.x) {
        if (!cand[j]) continue;
        const bool in_s = rank[j] < w;
        my_d += in_f[j] && !in_s;
      }
      const int D = block_sum_int(my_d, red);
      wants = (float)D > __fmul_rn(a.delta, (float)w);
      if (threadIdx.x == 0 && a.drift) a.drift[b] = D;
    }
  }
  if (k < 0) k = 0;
  rank_candidates(rr, cand, n, idx, rank);
  for (int j = threadIdx.x; j < a.max_pages; j += blockDim.x) {
    uint8_t kp = 0;
    if (j < n) kp = cand[j] ? (rank[j] < k) : 1;
    keep[j] = kp;
  }
  return wants;
}

// Phase 1: one block per sequence: ranks, drift, the compaction keep set.
__global__ void __launch_bounds__(kSelThreads) select_rank_kernel(const SelectArgs a) {
  extern __shared__ float sel_sm[];
  __shared__ int red[32];
  const int b = blockIdx.x;
  const int wants = select_row(a, b, sel_sm, red);
  if (threadIdx.x == 0) a.wants[b] = wants;
}

// Phase 2 (boundary mode): grant grows in ascending b while free pages last.
__global__ void __launch_bounds__(1024) select_grant_kernel(const SelectArgs a,
                                                            const int32_t* __restrict__ free_top) {
  __shared__ int sm[32];
  __shared__ int s_carry;
  const int free_count = *free_top;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    const int w = b < a.B ? a.wants[b] : 0;
    // inclusive scan of w across the block
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = w;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sm[warp] = x;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += sm[i];
    const int carry = s_carry;
    const int excl = carry + before + x - w;
    if (b < a.B && w && excl < free_count) {
      a.grow[b] = 1;
      a.budget[b] += 1;
      const int n = (int)ceil_div_ll(a.seq_lens[b], a.ps);
      uint8_t* keep = a.keep + (size_t)b * a.max_pages;
      for (int j = 0; j < n && j < a.max_pages; ++j) keep[j] = 1;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_carry = carry + before + x;
    __syncthreads();
  }
}

// ------------------------------------------------------------------ compaction
struct CompactArgs {
  int32_t* table;
  int max_pages;
  int32_t* seq_lens;
  const uint8_t* keep;
  int token_granular;
  uint8_t* k_pool;
  uint8_t* v_pool;
  int num_pages;
  int32_t* free_list;
  int32_t* free_top;
  int B, Hkv, d, ps;
  // workspace
  int32_t* new_len;    // [B]
  int32_t* pop_base;   // [B]
  int32_t* push_base;  // [B]
  int32_t* fresh_ids;  // [max_fresh]
  long long max_fresh;
  int32_t* ctl;        // [0] abort flag, [1] top after pops
  int* status;
  // shared pages (refcnt != NULL)
  int32_t* refcnt;     // [num_pages] block-table references per pool page
  uint8_t* freed_flag; // [B][max_pages] 1: old page j of b not reused; 2: and pushed
  int32_t* page_cnt;   // [num_pages] references freed in this call
  int32_t* page_key;   // [num_pages] largest (b * max_pages + j) freeing the page
};

// keep bit of token t (valid token of b)
__device__ __forceinline__ bool kept_token(const CompactArgs& a, int b, long long t) {
  if (a.token_granular) return a.keep[(size_t)b * a.max_pages * a.ps + t] != 0;
  return a.keep[(size_t)b * a.max_pages + t / a.ps] != 0;
}

// Per source page j of b: kept count c, whether the kept slots are a prefix.
__device__ __forceinline__ void page_keep_info(const CompactArgs& a, int b, int j, int L, int* c,
                                               bool* prefix) {
  const int lo = j * a.ps, hi = min(L, lo + a.ps);
  if (!a.token_granular) {  // one keep bit for the whole page: all or none, a prefix either way
    *c = a.keep[(size_t)b * a.max_pages + j] != 0 ? hi - lo : 0;
    *prefix = true;
    return;
  }
  int cnt = 0;
  bool pre = true, gap = false;
  for (int t = lo; t < hi; ++t) {
    const bool k = kept_token(a, b, t);
    if (k) {
      if (gap) pre = false;
      ++cnt;
    } else {
      gap = true;
    }
  }
  *c = cnt;
  *prefix = pre;
}

// Plan, in three steps (four with shared pages):
//  count  -- one block per sequence: kept tokens K, pages reused in place,
//            fresh and freed page counts (block-wide scan over its pages);
//  free   -- shared pages only: which freed reference returns each page to
//            the free list (the last one in (b, j) order, when the call frees
//            every reference), and the reference counts after the call;
//  scan   -- one block: exclusive scans of the counts over b, the free-list
//            check, the popped page ids.
constexpr int kCountThreads = 256;

__global__ void __launch_bounds__(kCountThreads) compact_count_kernel(const CompactArgs a) {
  __shared__ int sm[kCountThreads / 32];
  __shared__ int s_carry;
  const int b = blockIdx.x;
  const int L = a.seq_lens[b];
  const int np = (int)ceil_div_ll(L, a.ps);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int mine = 0;
  for (int j = threadIdx.x; j < np; j += blockDim.x) {
    int c = 0;
    bool pre = true;
    page_keep_info(a, b, j, L, &c, &pre);
    mine += c;
  }
  const int K = block_sum_int(mine, sm);
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  int reused_mine = 0;
  for (int base = 0; base < np; base += blockDim.x) {
    const int j = base + threadIdx.x;
    int c = 0;
    bool pre = true;
    if (j < np) page_keep_info(a, b, j, L, &c, &pre);
    int x = c;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sm[warp] = x;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += sm[i];
    const int carry = s_carry;
    const int kb = carry + before + x - c;  // kept tokens before page j
    const bool reuse = j < np && c > 0 && pre && (kb % a.ps == 0) && (c == a.ps || kb + c == K);
    reused_mine += reuse ? 1 : 0;
    if (a.refcnt && j < np) {
      a.freed_flag[(size_t)b * a.max_pages + j] = reuse ? 0 : 1;
      if (!reuse) {
        const int pg = a.table[(size_t)b * a.max_pages + j];
        if (pg >= 0 && pg < a.num_pages) {
          atomicAdd(&a.page_cnt[pg], 1);
          atomicMax(&a.page_key[pg], b * a.max_pages + j);
        } else {
          set_status(a.status, KV_EBADPAGE);
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_carry = carry + before + x;
    __syncthreads();
  }
  const int reused = block_sum_int(reused_mine, sm);
  if (threadIdx.x == 0) {
    const int n_new = (int)ceil_div_ll(K, a.ps);
    a.new_len[b] = K;
    a.pop_base[b] = n_new - reused;  // fresh pages (scanned below)
    a.push_base[b] = np - reused;    // freed pages (scanned below)
  }
}

// Shared pages: per-call reference tallies start empty.
__global__ void compact_clear_kernel(const CompactArgs a) {
  for (long long pg = (long long)blockIdx.x * blockDim.x + threadIdx.x; pg < a.num_pages;
       pg += (long long)gridDim.x * blockDim.x) {
    a.page_cnt[pg] = 0;
    a.page_key[pg] = -1;
  }
}

// Shared pages: a freed page goes back on the free list with the reference
// that takes its count to zero -- the last one in (b, j) order, if the call
// frees all of them.  That reference also lowers the count by the call's
// total.  One block per sequence.
__global__ void __launch_bounds__(kCountThreads) compact_free_kernel(const CompactArgs a) {
  __shared__ int sm[kCountThreads / 32];
  const int b = blockIdx.x;
  const int np = (int)ceil_div_ll(a.seq_lens[b], a.ps);
  int pushed = 0;
  for (int j = threadIdx.x; j < np; j += blockDim.x) {
    if (!a.freed_flag[(size_t)b * a.max_pages + j]) continue;
    const int pg = a.table[(size_t)b * a.max_pages + j];
    if (pg >= 0 && pg < a.num_pages && a.page_key[pg] == b * a.max_pages + j) {
      const bool push = a.page_cnt[pg] == a.refcnt[pg];
      a.refcnt[pg] -= a.page_cnt[pg];
      if (push) {
        a.freed_flag[(size_t)b * a.max_pages + j] = 2;
        ++pushed;
      }
    }
  }
  const int total = block_sum_int(pushed, sm);
  if (threadIdx.x == 0) a.push_base[b] = total;
}

__global__ void __launch_bounds__(1024) compact_scan_kernel(const CompactArgs a) {
  __shared__ long long sm[32];
  __shared__ int s_info[4];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // exclusive scans over b (single block, sequential chunks)
  if (threadIdx.x == 0) {
    s_info[0] = 0;
    s_info[1] = 0;
  }
  __syncthreads();
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    const int f = b < a.B ? a.pop_base[b] : 0;
    const int r = b < a.B ? a.push_base[b] : 0;
    long long xf = f, xr = r;
    for (int o = 1; o < 32; o <<= 1) {
      const long long yf = __shfl_up_sync(FULL, xf, o), yr = __shfl_up_sync(FULL, xr, o);
      if (lane >= o) { xf += yf; xr += yr; }
    }
    if (lane == 31) sm[warp] = (xf << 32) | xr;
    __syncthreads();
    long long bf = 0, br = 0;
    for (int i = 0; i < warp; ++i) { bf += sm[i] >> 32; br += sm[i] & 0xffffffffll; }
    const int cf = s_info[0], cr = s_info[1];
    if (b < a.B) {
      a.pop_base[b] = (int)(cf + bf + xf - f);
      a.push_base[b] = (int)(cr + br + xr - r);
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) {
      s_info[0] = (int)(cf + bf + xf);
      s_info[1] = (int)(cr + br + xr);
    }
    __syncthreads();
  }
  const int pops = s_info[0], pushes = s_info[1];
  const int top = *a.free_top;
  const bool fail = pops > top || pops > a.max_fresh;
  if (fail) {
    if (threadIdx.x == 0) {
      a.ctl[0] = 1;
      set_status(a.status, pops > top ? KV_ENOSPACE : KV_EWORKSPACE);
    }
    return;
  }
  for (int i = threadIdx.x; i < pops; i += blockDim.x) {
    const int pg = a.free_list[top - 1 - i];
    a.fresh_ids[i] = pg;
    if (a.refcnt && pg >= 0 && pg < a.num_pages) a.refcnt[pg] = 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a.ctl[0] = 0;
    a.ctl[1] = top - pops;
    *a.free_top = top - pops + pushes;
  }
}

// Apply: one block per sequence rewrites its row, gathers tokens into fresh
// pages, pushes its freed pages.
constexpr int kApplyThreads = 256;

__global__ void __launch_bounds__(kApplyThreads) compact_apply_kernel(const CompactArgs a) {
  extern __shared__ int32_t cs[];
  __shared__ int sm[kApplyThreads / 32];
  __shared__ int s_carry[3];
  if (a.ctl[0]) return;
  const int b = blockIdx.x;
  const int L = a.seq_lens[b];
  const int np = (int)ceil_div_ll(L, a.ps);
  const int K = a.new_len[b];
  const int n_new = (int)ceil_div_ll(K, a.ps);
  int32_t* old_row = cs;                // [max_pages]
  int32_t* dest_src = cs + a.max_pages; // [max_pages] old page j reused by dest m, or -1
  int32_t* kb_arr = dest_src + a.max_pages;  // [max_pages] kept tokens before page j
  const int32_t* row = a.table + (size_t)b * a.max_pages;
  for (int j = threadIdx.x; j < a.max_pages; j += blockDim.x) {
    old_row[j] = j < np ? row[j] : -1;
    dest_src[j] = -1;
  }
  if (threadIdx.x == 0) { s_carry[0] = 0; s_carry[1] = 0; s_carry[2] = 0; }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // pass over source pages: kept-before, reuse, freed ranks
  for (int base = 0; base < np; base += blockDim.x) {
    const int j = base + threadIdx.x;
    int c = 0;
    bool pre = true;
    if (j < np) page_keep_info(a, b, j, L, &c, &pre);
    int x = c;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sm[warp] = x;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += sm[i];
    const int carry = s_carry[0];
    const int kb = carry + before + x - c;
    const bool reuse = j < np && c > 0 && pre && (kb % a.ps == 0) && (c == a.ps || kb + c == K);
    if (j < np) {
      kb_arr[j] = kb;
      if (reuse) dest_src[kb / a.ps] = j;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_carry[0] = carry + before + x;
    __syncthreads();
  }
  // freed pages (old pages not reused), pushed in j order
  const int top_after_pops = a.ctl[1];
  for (int base = 0; base < np; base += blockDim.x) {
    const int j = base + threadIdx.x;
    // page j is reused iff dest_src[kb_arr[j] / ps] == j
    bool freed = false;
    if (j < np) {
      const int m = kb_arr[j] / a.ps;
      freed = !(m < a.max_pages && dest_src[m] == j && (kb_arr[j] % a.ps) == 0);
      // with shared pages only the reference that frees the page pushes it
      if (a.refcnt) freed = a.freed_flag[(size_t)b * a.max_pages + j] == 2;
    }
    const unsigned bal = __ballot_sync(FULL, freed);
    const int x = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) sm[warp] = __popc(bal);
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += sm[i];
    const int carry = s_carry[1];
    if (freed) {
      const int page = old_row[j];
      a.free_list[top_after_pops + a.push_base[b] + carry + before + x] = page;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += sm[i];
      s_carry[1] = carry + tot;
    }
    __syncthreads();
  }
  // new row: reused pages in place, fresh pages in order of m
  int32_t* out_row = a.table + (size_t)b * a.max_pages;
  int32_t* new_row = kb_arr;  // reuse: kb_arr no longer needed after the pass above
  __syncthreads();
  for (int base = 0; base < a.max_pages; base += blockDim.x) {
    const int m = base + threadIdx.x;
    const bool fresh = m < n_new && dest_src[m] < 0;
    const unsigned bal = __ballot_sync(FULL, fresh);
    const int x = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) sm[warp] = __popc(bal);
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += sm[i];
    const int carry = s_carry[2];
    if (m < a.max_pages) {
      int page = -1;
      if (m < n_new) page = fresh ? a.fresh_ids[a.pop_base[b] + carry + before + x] : old_row[dest_src[m]];
      new_row[m] = page;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += sm[i];
      s_carry[2] = carry + tot;
    }
    __syncthreads();
  }
  // gather tokens that land in fresh pages (token-granular masks only)
  if (a.token_granular) {
    const size_t row_bytes = (size_t)a.d * 2;            // one (token, head) row
    const size_t head_stride = (size_t)a.ps * row_bytes;  // one (page, head) tile
    const size_t page_stride = head_stride * a.Hkv;
    const int vec_per_row = (int)(row_bytes / 16);
    // walk kept tokens in order with a running rank
    if (threadIdx.x == 0) s_carry[0] = 0;
    __syncthreads();
    for (int base = 0; base < L; base += blockDim.x) {
      const int t = base + threadIdx.x;
      const bool k = t < L && kept_token(a, b, t);
      const unsigned bal = __ballot_sync(FULL, k);
      const int x = __popc(bal & ((1u << lane) - 1u));
      if (lane == 0) sm[warp] = __popc(bal);
      __syncthreads();
      int before = 0;
      for (int i = 0; i < warp; ++i) before += sm[i];
      const int carry = s_carry[0];
      if (k) {
        const int r = carry + before + x;
        const int m = r / a.ps, slot = r % a.ps;
        if (dest_src[m] < 0) {
          const int src_page = old_row[t / a.ps];
          const int dst_page = new_row[m];
          if (src_page >= 0 && src_page < a.num_pages && dst_page >= 0 && dst_page < a.num_pages) {
            for (int h = 0; h < a.Hkv; ++h) {
              const size_t so = (size_t)src_page * page_stride + h * head_stride + (size_t)(t % a.ps) * row_bytes;
              const size_t dof = (size_t)dst_page * page_stride + h * head_stride + (size_t)slot * row_bytes;
              const uint4* ks = reinterpret_cast<const uint4*>(a.k_pool + so);
              const uint4* vs = reinterpret_cast<const uint4*>(a.v_pool + so);
              uint4* kd = reinterpret_cast<uint4*>(a.k_pool + dof);
              uint4* vd = reinterpret_cast<uint4*>(a.v_pool + dof);
              for (int v = 0; v < vec_per_row; ++v) {
                kd[v] = ks[v];
                vd[v] = vs[v];
              }
            }
          } else {
            set_status(a.status, KV_EBADPAGE);
          }
        }
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int tot = 0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += sm[i];
        s_carry[0] = carry + tot;
      }
      __syncthreads();
    }
  }
  __syncthreads();
  for (int m = threadIdx.x; m < a.max_pages; m += blockDim.x) out_row[m] = new_row[m];
  if (threadIdx.x == 0) a.seq_lens[b] = K;
}

// ------------------------------------------------------------------ append
struct AppendArgs {
  const uint8_t* k_new;
  const uint8_t* v_new;
  uint8_t* k_pool;
  uint8_t* v_pool;
  int num_pages;
  int32_t* table;
  int max_pages;
  int32_t* seq_lens;
  int32_t* free_list;
  int32_t* free_top;
  int B, Hkv, d, ps;
  int2* dest;    // [B] (page, slot) workspace
  int32_t* ctl;  // [0] abort
  int* status;
  // shared pages (refcnt != NULL)
  int32_t* refcnt;   // [num_pages] block-table references per pool page
  int32_t* cand;     // [B] shared, partly filled last page of b, or -1
  int32_t* cow_src;  // [B] page b copies before writing (copy-on-write), or -1
};

__global__ void __launch_bounds__(1024) append_plan_kernel(const AppendArgs a) {
  __shared__ int sm[32];
  __shared__ int s_err[3];
  __shared__ int s_carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) { s_err[0] = s_err[1] = 0; s_carry = 0; }
  __syncthreads();
  // pass A: rows full, bad page ids already in use, number of pops
  int my_need = 0;
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    const int L = a.seq_lens[b];
    int cand = -1;
    if (L < 0) {
      s_err[1] = 1;
    } else if (L % a.ps == 0) {
      if (L / a.ps >= a.max_pages) s_err[0] = 1;
      ++my_need;
    } else {
      const int p = a.table[(size_t)b * a.max_pages + L / a.ps];
      if (p < 0 || p >= a.num_pages) s_err[1] = 1;
      else if (a.refcnt && a.refcnt[p] > 1) cand = p;
    }
    if (a.refcnt) a.cand[b] = cand;
  }
  if (a.refcnt) {
    // Copy-on-write in ascending b: sequence b copies its shared last page p
    // unless the sharers before it have already copied so that it is the
    // only reference left (then it writes in place).
    __syncthreads();
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
      const int p = a.cand[b];
      int cow = -1;
      if (p >= 0) {
        int rank = 0;
        for (int b2 = 0; b2 < b; ++b2) rank += a.cand[b2] == p;
        if (a.refcnt[p] - rank > 1) cow = p;
      }
      a.cow_src[b] = cow;
      my_need += cow >= 0;
    }
  }
  int need = my_need;
  for (int o = 16; o; o >>= 1) need += __shfl_xor_sync(FULL, need, o);
  if (lane == 0) sm[warp] = need;
  __syncthreads();
  int total = 0;
  for (int i = 0; i < nw; ++i) total += sm[i];
  const int top = *a.free_top;
  // pass B: ids that would be popped must be pool pages
  if (total <= top)
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
      const int p = a.free_list[top - 1 - i];
      if (p < 0 || p >= a.num_pages) s_err[1] = 1;
    }
  __syncthreads();
  const int err = s_err[0] ? KV_EFULL : (s_err[1] ? KV_EBADPAGE : (total > top ? KV_ENOSPACE : 0));
  if (err) {
    if (threadIdx.x == 0) {
      a.ctl[0] = 1;
      set_status(a.status, err);
    }
    return;
  }
  // pass C: pops in ascending b, table and length updates
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    const int L = b < a.B ? a.seq_lens[b] : 1;
    const bool cow = a.refcnt && b < a.B && a.cow_src[b] >= 0;
    const bool nd = b < a.B && (L % a.ps == 0 || cow);
    const unsigned bal = __ballot_sync(FULL, nd);
    const int x = __popc(bal & ((1u << lane) - 1u));
    __syncthreads();
    if (lane == 0) sm[warp] = __popc(bal);
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += sm[i];
    const int carry = s_carry;
    if (b < a.B) {
      int32_t* slot = &a.table[(size_t)b * a.max_pages + L / a.ps];
      if (nd) {
        const int fresh = a.free_list[top - 1 - (carry + before + x)];
        if (a.refcnt) {
          a.refcnt[fresh] = 1;
          if (cow) atomicSub(&a.refcnt[*slot], 1);
        }
        *slot = fresh;
      }
      a.dest[b] = make_int2(*slot, L % a.ps);
      a.seq_lens[b] = L + 1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int i = 0; i < nw; ++i) tot += sm[i];
      s_carry = carry + tot;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    a.ctl[0] = 0;
    *a.free_top = top - total;
  }
}

// Copy-on-write: the filled slots of the shared page b leaves, into its
// fresh page (all heads, K and V).  Runs before any token is written, so a
// sharer that writes into the old page in place cannot race with the copy.
__global__ void append_cow_kernel(const AppendArgs a) {
  if (a.ctl[0]) return;
  const int b = blockIdx.x;
  const int src = a.cow_src[b];
  if (src < 0) return;
  const int2 dst = a.dest[b];
  const size_t row_bytes = (size_t)a.d * 2;
  const int vec = (int)(row_bytes / 16);
  const int n = dst.y * vec;  // filled slots x 16-byte pieces per row
  for (int i = threadIdx.x; i < a.Hkv * n; i += blockDim.x) {
    const int h = i / n, r = i - h * n;
    const size_t so = ((size_t)src * a.Hkv + h) * a.ps * row_bytes + (size_t)r * 16;
    const size_t dof = ((size_t)dst.x * a.Hkv + h) * a.ps * row_bytes + (size_t)r * 16;
    *reinterpret_cast<uint4*>(a.k_pool + dof) = *reinterpret_cast<const uint4*>(a.k_pool + so);
    *reinterpret_cast<uint4*>(a.v_pool + dof) = *reinterpret_cast<const uint4*>(a.v_pool + so);
  }
}

// Copy the new token's K and V rows (all heads) into place; 16 bytes per thread.
__global__ void append_copy_kernel(const AppendArgs a) {
  if (a.ctl[0]) return;
  const int b = blockIdx.x;
  const int2 dst = a.dest[b];
  const size_t row_bytes = (size_t)a.d * 2;
  const int vec = (int)(row_bytes / 16);
  for (int i = threadIdx.x; i < a.Hkv * vec; i += blockDim.x) {
    const int h = i / vec, v = i - h * vec;
    const size_t so = ((size_t)b * a.Hkv + h) * row_bytes + (size_t)v * 16;
    const size_t dof = (((size_t)dst.x * a.Hkv + h) * a.ps + dst.y) * row_bytes + (size_t)v * 16;
    *reinterpret_cast<uint4*>(a.k_pool + dof) = *reinterpret_cast<const uint4*>(a.k_new + so);
    *reinterpret_cast<uint4*>(a.v_pool + dof) = *reinterpret_cast<const uint4*>(a.v_new + so);
  }
}

// ------------------------------------------------------------------ fused steady-state step
// The budgeting part of one steady-state step in one launch, equal bit for
// bit to kv_update_query_summaries (first = 0), kv_mark_active (mode 1),
// kv_summarize_last_pages, kv_score_pages, kv_select_pages (boundary),
// kv_compact (page masks) and kv_append issued in that order, for a valid
// batch (finite scores) without shared pages.  Every value is computed by
// the same rounded operations in the same order as in those kernels.
//  * S blocks per sequence (one for a sequence not at a capacity boundary)
//    each form the sequence's updated EMAs in shared memory and score a
//    stride-S share of its pages, one warp per page; the block that owns the
//    last page first summarises it (the page that just filled).
//  * The last of those blocks to finish (a ticket; nobody waits) writes the
//    EMAs, ranks the candidates under both summaries in one pass (working
//    sets and drift), and -- unless the sequence wants to grow -- compacts
//    it: a boundary compaction keeps all candidates but the last in
//    retention order, the one with the smallest S_fast + S_slow (the higher
//    logical index among equal keys).
//  * The last sequence to finish (a second ticket) grants the grows in
//    ascending b, compacts the sequences that wanted a page and got none,
//    pushes the freed pages in (b, j) order and appends the step's token.
struct StepArgs {
  const uint16_t* q;
  const uint8_t* k_new;
  const uint8_t* v_new;
  uint8_t* k_pool;
  uint8_t* v_pool;
  int num_pages;
  int32_t* table;
  int max_pages;
  int32_t* seq_lens;
  int32_t* budget;
  int B, Hq, Hkv, d, ps, S;
  float a_fast, a_slow;
  int n_first, n_last;
  float delta, ws_frac;
  int update_ema;     // 0: the EMAs are used as they are (the first step after the fit)
  float* ema;
  float* summ;
  float* scores;
  uint8_t* active;
  uint8_t* keep;
  uint8_t* grow;
  int32_t* drift;
  int32_t* free_list;
  int32_t* free_top;
  // workspace
  int32_t* wants;     // [B]
  int32_t* new_len;   // [B] length after compaction, then the final length (step_copy_kernel
                      // stores it in seq_lens, which stays as the step found it until then)
  int32_t* drop_cnt;  // [B] pages freed by the compaction
  int32_t* drop_ids;  // [B][max_pages] their ids, in j order
  int32_t* row_tk;    // [B] per-sequence tickets; zero between calls
  int2* dest;         // [B] (page, slot) of each sequence's token, for step_copy_kernel
  unsigned* ticket;   // in the status header: sequences finished; zero between calls
  unsigned* grab;     // in the status header: items handed out; zero between calls
  unsigned* exits;    // in the status header: blocks done taking items; zero between calls
  int* ctl;           // in the status header: 1 when the append failed (nothing to copy)
  int* status;
};

constexpr int kStepThreads = 512;
constexpr int kStepSplit = 16;             // blocks per sequence at a boundary
constexpr int kStepListMax = 2048;         // sequences the step lists in shared memory
constexpr size_t kStepTicketOffset = 64;  // bytes into the status header: ticket,
constexpr size_t kStepGrabOffset = 68;    // item counter,
constexpr size_t kStepExitOffset = 72;    // exit counter,
constexpr size_t kStepCtlOffset = 76;     // append-failed flag

// Page-granular compaction of one row (whole block): the kept pages move to
// the front in order (each reused where it is; no K/V moves), the row is -1
// padded, the dropped page ids are listed in j order.  Returns the kept
// token count K and sets *n_drops (both on every thread).  The row and its
// keep mask are read through L2 (another block may have written them).
__device__ int compact_row_pages(int32_t* row, const uint8_t* keep_row, int n, int L, int ps,
                                 int max_pages, int32_t* drops, int* n_drops, int* sm, int* carry) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) carry[0] = carry[1] = 0;
  __syncthreads();
  int K_mine = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int j = base + threadIdx.x;
    const bool in = j < n;
    const bool kept = in && __ldcg(keep_row + j) != 0;
    const int old = in ? __ldcg(row + j) : -1;
    const unsigned bk = __ballot_sync(FULL, kept), bd = __ballot_sync(FULL, in && !kept);
    const unsigned lt = (1u << lane) - 1u;
    if (lane == 0) {
      sm[warp] = __popc(bk);
      sm[32 + warp] = __popc(bd);
    }
    __syncthreads();
    int bkb = 0, bdb = 0, tk = 0, td = 0;
    for (int w = 0; w < nw; ++w) {
      if (w < warp) {
        bkb += sm[w];
        bdb += sm[32 + w];
      }
      tk += sm[w];
      td += sm[32 + w];
    }
    const int ck = carry[0], cd = carry[1];
    // every old entry of this chunk has been read; a kept page moves to
    // m <= j, so nothing not yet read is overwritten
    __syncthreads();
    if (kept) {
      row[ck + bkb + __popc(bk & lt)] = old;
      K_mine += min(L, (j + 1) * ps) - j * ps;
    } else if (in) {
      drops[cd + bdb + __popc(bd & lt)] = old;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      carry[0] = ck + tk;
      carry[1] = cd + td;
    }
    __syncthreads();
  }
  const int kept_total = carry[0];
  *n_drops = carry[1];
  for (int m = kept_total + threadIdx.x; m < max_pages; m += blockDim.x) row[m] = -1;
  return block_sum_int(K_mine, sm);
}

// Ranks of the candidates j in [c0, c1) under two keys at once (the counting
// definition of rank_of over that range: larger key first, equal keys by the
// lower index); key2[j] = (key a, key b).  n <= 1024.
__device__ void rank_two(const float2* key2, int c0, int c1, uint16_t* ra, uint16_t* rb) {
  const int nc = c1 - c0;
  int tpc = 1;  // lanes per candidate
  while (tpc < 32 && tpc * 2 * nc <= (int)blockDim.x) tpc <<= 1;
  const int per_pass = blockDim.x / tpc, sub = threadIdx.x & (tpc - 1);
  for (int j0 = 0; j0 < nc; j0 += per_pass) {
    const int j = c0 + j0 + (int)threadIdx.x / tpc;
    const bool mine = j < c1;
    int x = 0, y = 0;
    if (mine) {
      const float2 kj = key2[j];
      for (int i = c0 + sub; i < c1; i += tpc) {
        const float2 ki = key2[i];
        x += ki.x > kj.x || (ki.x == kj.x && i < j);
        y += ki.y > kj.y || (ki.y == kj.y && i < j);
      }
    }
    for (int o = tpc >> 1; o; o >>= 1) {
      x += __shfl_xor_sync(FULL, x, o);
      y += __shfl_xor_sync(FULL, y, o);
    }
    if (mine && sub == 0) {
      ra[j] = (uint16_t)x;
      rb[j] = (uint16_t)y;
    }
  }
  __syncthreads();
}

// Boundary selection of row b in one block (as select_row in boundary mode
// for finite keys): writes keep[b], drift[b], grow[b] = 0; returns wants.
// The candidates are the pages between the forced first and last ones.
__device__ int select_boundary_row(const StepArgs& a, int b, int n, float* sm_f, int* red,
                                   int* s_int) {
  uint8_t* keep = a.keep + (size_t)b * a.max_pages;
  if (threadIdx.x == 0) {
    a.grow[b] = 0;
    if (a.drift) a.drift[b] = 0;
  }
  const int c0 = min(a.n_first, n), c1 = max(c0, n - a.n_last);
  const int nc = c1 - c0;
  float2* key2 = reinterpret_cast<float2*>(sm_f);                  // [n] (S_fast, S_slow)
  float* rr = reinterpret_cast<float*>(key2 + n);                  // [n] S_fast + S_slow
  uint8_t* cand = reinterpret_cast<uint8_t*>(rr + n);              // [n] (rows above 1024)
  uint16_t* idx = reinterpret_cast<uint16_t*>(cand + align_up(n, 4));  // [next_pow2(n)]
  int P2 = 1;
  while (P2 < n) P2 <<= 1;
  uint16_t* rank_f = idx + P2;                                     // [n]
  uint16_t* rank_s = rank_f + n;                                   // [n]
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const float2 sc = __ldcg(reinterpret_cast<const float2*>(a.scores + (size_t)b * a.max_pages * 2) + j);
    key2[j] = sc;
    rr[j] = __fadd_rn(sc.x, sc.y);
    cand[j] = j >= c0 && j < c1;
  }
  __syncthreads();
  int wants = 0;
  if (nc == 0) {
    wants = 1;
  } else {
    int w = (int)ceilf(__fmul_rn(a.ws_frac, (float)nc));
    w = max(1, min(w, nc));
    if (n <= 1024) {
      rank_two(key2, c0, c1, rank_f, rank_s);
    } else {
      float* sf = reinterpret_cast<float*>(rank_s + n);  // unpacked keys for the sort
      float* ss = sf + n;
      for (int j = threadIdx.x; j < n; j += blockDim.x) {
        sf[j] = key2[j].x;
        ss[j] = key2[j].y;
      }
      __syncthreads();
      rank_candidates(sf, cand, n, idx, rank_f);
      rank_candidates(ss, cand, n, idx, rank_s);
    }
    int my_d = 0;
    for (int j = c0 + threadIdx.x; j < c1; j += blockDim.x) my_d += rank_f[j] < w && rank_s[j] >= w;
    const int D = block_sum_int(my_d, red);
    wants = (float)D > __fmul_rn(a.delta, (float)w);
    if (threadIdx.x == 0 && a.drift) a.drift[b] = D;
  }
  // keep = forced + the best nc - 1 candidates by R: all candidates but the
  // last in rank order -- the smallest R, the higher index among equal R
  if (threadIdx.x == 0) s_int[0] = -1;
  __syncthreads();
  if (nc > 0) {
    float best = INFINITY;
    int bj = -1;
    for (int j = c0 + threadIdx.x; j < c1; j += blockDim.x) {
      if (bj < 0 || rr[j] < best || (rr[j] == best && j > bj)) {
        best = rr[j];
        bj = j;
      }
    }
    for (int o = 16; o; o >>= 1) {
      const float ob = __shfl_xor_sync(FULL, best, o);
      const int oj = __shfl_xor_sync(FULL, bj, o);
      if (oj >= 0 && (bj < 0 || ob < best || (ob == best && oj > bj))) {
        best = ob;
        bj = oj;
      }
    }
    float* wb = reinterpret_cast<float*>(red);  // [32] values, [32..63] indices
    if ((threadIdx.x & 31) == 0) {
      wb[threadIdx.x >> 5] = best;
      red[32 + (threadIdx.x >> 5)] = bj;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float bb = INFINITY;
      int bjj = -1;
      for (int w2 = 0; w2 < (int)(blockDim.x >> 5); ++w2) {
        const float v = wb[w2];
        const int jj = red[32 + w2];
        if (jj >= 0 && (bjj < 0 || v < bb || (v == bb && jj > bjj))) {
          bb = v;
          bjj = jj;
        }
      }
      s_int[0] = bjj;
    }
  }
  __syncthreads();
  const int drop = s_int[0];
  for (int j = threadIdx.x; j < a.max_pages; j += blockDim.x) keep[j] = j < n && j != drop;
  return wants;
}

template <class T, int CPL>
__global__ void __launch_bounds__(kStepThreads, 1) budget_step_kernel(const StepArgs a) {
  // the token copy that follows may be scheduled early; it waits for this
  // grid to finish before it reads anything (griddepcontrol.wait)
  pdl_launch_dependents();
  extern __shared__ float step_sm[];
  __shared__ int red[64];
  __shared__ int s_carry[4];
  __shared__ int s_int[2];
  __shared__ int s_last;
  constexpr int D = 32 * CPL;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = blockDim.x >> 5;
  const int G = a.Hq / a.Hkv;
  float* ema_s = step_sm;                   // [2][Hkv][D], the updated EMAs of b
  float* sel_sm = step_sm + 2 * a.Hkv * D;  // selection arrays / last block's scratch
  const uint16_t* k16 = reinterpret_cast<const uint16_t*>(a.k_pool);
  bool finisher = false;  // this block finishes the step (the last sequence to arrive)
  __shared__ unsigned s_item;
  __shared__ int s_rows[kStepListMax];  // the sequences at a boundary, ascending
  __shared__ int s_nsc;

  // Work items: (sequence b, split s).  A sequence at a capacity boundary
  // (scored) has S items, any other one item.  Every block lists the scored
  // sequences from the lengths (which no block changes during this kernel:
  // the final lengths go to new_len), so the items can be numbered densely:
  // first the scored sequences' S splits, split-major, then one item per
  // sequence in b order (scored ones skip it).  Above kStepListMax sequences
  // the items are all B x S pairs, split-major, the unscored ones skipped.
  // Blocks take items one at a time from a counter and never wait on one
  // another.
  auto is_scored = [&](int b) {  // as mark_kernel, mode 1, within the table
    const int L = a.seq_lens[b];
    return L > 0 && L % a.ps == 0 && L / a.ps >= a.budget[b] &&
           ceil_div_ll(L, a.ps) <= a.max_pages;
  };
  const bool listed = a.B <= kStepListMax;
  if (tid == 0) s_nsc = 0;
  __syncthreads();
  if (listed)
    for (int base = 0; base < a.B; base += blockDim.x) {
      const int bb = base + tid;
      const bool sc = bb < a.B && is_scored(bb);
      const unsigned bal = __ballot_sync(FULL, sc);
      if (lane == 0) red[warp] = __popc(bal);
      __syncthreads();
      int before = s_nsc;
      for (int i = 0; i < warp; ++i) before += red[i];
      if (sc) s_rows[before + __popc(bal & ((1u << lane) - 1u))] = bb;
      __syncthreads();
      if (tid == 0)
        for (int i = 0; i < nw; ++i) s_nsc += red[i];
      __syncthreads();
    }
  const int nsc = s_nsc;
  const unsigned n_items = listed ? (unsigned)(nsc * a.S + a.B) : (unsigned)a.B * (unsigned)a.S;
  for (;;) {
  __syncthreads();  // the previous item's use of shared memory is over
  if (tid == 0) s_item = atomicAdd(a.grab, 1u);
  __syncthreads();
  const unsigned item = s_item;
  if (item >= n_items) break;
  int s, b;
  if (!listed) {
    s = (int)(item / a.B);
    b = (int)(item - (item / a.B) * a.B);
  } else if (item < (unsigned)(nsc * a.S)) {
    s = (int)(item / nsc);
    b = s_rows[item - (unsigned)s * nsc];
  } else {
    s = 0;
    b = (int)(item - (unsigned)(nsc * a.S));
  }
  // ---- capacity boundary (as mark_kernel, mode 1)
  const int L = a.seq_lens[b];
  const bool act = L > 0 && L % a.ps == 0 && L / a.ps >= a.budget[b];
  const int n = (int)ceil_div_ll(L, a.ps);
  const bool scoring = act && n <= a.max_pages;
  if (!scoring && s != 0) continue;  // one item for a sequence that is not scored
  if (listed && scoring && item >= (unsigned)(nsc * a.S)) continue;  // its items came first
  // ---- query EMAs of b (as ema_kernel, first = 0), into shared memory; the
  // row's last block writes them out once every block has read the old ones
  for (int i = tid; i < a.Hkv * D; i += blockDim.x) {
    const int h = i / D, c = i - h * D;
    float gm = 0.0f;
    if (a.update_ema) {
      float acc = 0.0f;
      for (int g = 0; g < G; ++g)
        acc = __fadd_rn(acc, ld16<T>(a.q, ((size_t)b * a.Hq + (size_t)h * G + g) * D + c));
      gm = __fdiv_rn(acc, (float)G);
    }
    for (int u = 0; u < 2; ++u) {
      const float al = u == 0 ? a.a_fast : a.a_slow;
      float v = __ldcg(a.ema + (((size_t)b * 2 + u) * a.Hkv + h) * D + c);
      if (a.update_ema) v = __fadd_rn(__fmul_rn(al, v), __fmul_rn(__fsub_rn(1.0f, al), gm));
      ema_s[(u * a.Hkv + h) * D + c] = v;
    }
  }
  __syncthreads();
  if (scoring) {
    // ---- summary of the page that just filled (as summary_kernel), by the
    // block that scores it
    const int jl = n - 1;
    if (jl % a.S == s) {
      const int page = a.table[(size_t)b * a.max_pages + jl];
      if (page < 0 || page >= a.num_pages) {
        if (tid == 0) set_status(a.status, KV_EBADPAGE);
      } else {
        for (int i = tid; i < a.Hkv * D; i += blockDim.x) {
          const int h = i / D, c = i - h * D;
          const uint16_t* src = k16 + ((size_t)page * a.Hkv + h) * a.ps * D + c;
          float acc = 0.0f, mn = INFINITY, mx = -INFINITY;
          auto take = [&](float v) {
            acc = __fadd_rn(acc, v);
            mn = v < mn ? v : mn;
            mx = v > mx ? v : mx;
          };
          if (a.ps == 16) {  // the 16 loads in flight together, then the running order
            float x[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) x[t] = ld16<T>(src, (size_t)t * D);
#pragma unroll
            for (int t = 0; t < 16; ++t) take(x[t]);
          } else {
            for (int t = 0; t < a.ps; ++t) take(ld16<T>(src, (size_t)t * D));
          }
          float* sp = a.summ + ((size_t)page * a.Hkv + h) * 3 * D;
          sp[c] = __fdiv_rn(acc, (float)a.ps);
          sp[D + c] = mn;
          sp[2 * D + c] = mx;
        }
      }
      __syncthreads();
    }
    // ---- scores of this block's pages (as score_kernel: one warp per page)
    for (int j = s + a.S * warp; j < a.max_pages; j += a.S * nw) {
      float2* out = reinterpret_cast<float2*>(a.scores + ((size_t)b * a.max_pages + j) * 2);
      if (j >= n) {
        if (lane == 0) *out = make_float2(-INFINITY, -INFINITY);
        continue;
      }
      const int page = a.table[(size_t)b * a.max_pages + j];
      if (page < 0 || page >= a.num_pages) {
        if (lane == 0) set_status(a.status, KV_EBADPAGE);
        continue;
      }
      float af = 0.0f, as = 0.0f;
      const float* smp = a.summ + (size_t)page * a.Hkv * 3 * D + lane * CPL;
#pragma unroll 4
      for (int h = 0; h < a.Hkv; ++h) {
        const float* uf = ema_s + (0 * a.Hkv + h) * D + lane * CPL;
        const float* us = ema_s + (1 * a.Hkv + h) * D + lane * CPL;
        const float* sm = smp + (size_t)h * 3 * D;
        float mu[CPL], mnv[CPL], mxv[CPL];
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          mu[i] = sm[i];
          mnv[i] = sm[D + i];
          mxv[i] = sm[2 * D + i];
        }
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          {
            const float u = uf[i];
            const float ta = __fmul_rn(u, mnv[i]), tb = __fmul_rn(u, mxv[i]);
            af = __fadd_rn(af, __fadd_rn(__fmul_rn(u, mu[i]), ta > tb ? ta : tb));
          }
          {
            const float u = us[i];
            const float ta = __fmul_rn(u, mnv[i]), tb = __fmul_rn(u, mxv[i]);
            as = __fadd_rn(as, __fadd_rn(__fmul_rn(u, mu[i]), ta > tb ? ta : tb));
          }
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        af = __fadd_rn(af, __shfl_xor_sync(FULL, af, o));
        as = __fadd_rn(as, __shfl_xor_sync(FULL, as, o));
      }
      if (lane == 0) *out = make_float2(af, as);
    }
  }
  // ---- the row's last block: EMAs out, selection, compaction
  __threadfence();
  __syncthreads();
  if (tid == 0)
    s_last = atomicAdd(a.row_tk + b, 1) == (scoring ? a.S : 1) - 1;
  __syncthreads();
  if (!s_last) continue;
  __threadfence();
  for (int i = tid; i < 2 * a.Hkv * D; i += blockDim.x) {
    const int u = i / (a.Hkv * D), r = i - u * (a.Hkv * D);
    a.ema[((size_t)b * 2 + u) * a.Hkv * D + r] = ema_s[i];
  }
  int wants = 0, new_len = L, drops = 0;
  uint8_t* keep = a.keep + (size_t)b * a.max_pages;
  if (tid == 0) {
    a.active[b] = act;
    a.row_tk[b] = 0;  // ready for the next call
  }
  if (!act || n > a.max_pages) {
    // as select_row for a row that is not selected: every page kept
    if (n > a.max_pages && tid == 0) set_status(a.status, KV_EINVAL);
    if (tid == 0) {
      a.grow[b] = 0;
      if (a.drift) a.drift[b] = 0;
    }
    for (int j = tid; j < a.max_pages; j += blockDim.x) keep[j] = j < n;
  } else {
    wants = select_boundary_row(a, b, n, sel_sm, red, s_int);
    __threadfence();
    __syncthreads();
    if (!wants)
      new_len = compact_row_pages(a.table + (size_t)b * a.max_pages, keep, n, L, a.ps,
                                  a.max_pages, a.drop_ids + (size_t)b * a.max_pages, &drops, red,
                                  s_carry);
  }
  if (tid == 0) {
    a.wants[b] = act ? wants : 0;
    a.new_len[b] = new_len;
    a.drop_cnt[b] = drops;
  }
  // ---- the last sequence to arrive finishes the step
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.ticket, 1u) == (unsigned)(a.B - 1);
  __syncthreads();
  if (s_last) finisher = true;
  if (finisher) break;  // every sequence has arrived: no item is left to take
  }  // items
  // the last block to stop taking items (the finisher stops after its work)
  // puts the counters back to zero
  auto leave = [&]() {
    if (tid == 0 && atomicAdd(a.exits, 1u) == gridDim.x - 1) {
      *a.grab = 0;
      *a.exits = 0;
    }
  };
  if (!finisher) {
    leave();
    return;
  }
  __syncthreads();
  __threadfence();
  const int free_count = __ldcg(a.free_top);
  int* pend = reinterpret_cast<int*>(sel_sm);  // [B] rows to compact here, then offsets
  int* cnt_s = pend + a.B;                     // [B] pages freed per row
  int* pg_pre = pend + 2 * a.B;                // [B] the token's page of rows needing none new
  int* pops = pend + 3 * a.B;                  // [B] the free-list ids the appends pop
  // A row whose length is not a page multiple was not at a boundary: it keeps
  // its length and table, and its token goes to the page its length ends in.
  // Loaded now, used by the append plan below.
  for (int bb = tid; bb < a.B; bb += blockDim.x) {
    const int Lo = a.seq_lens[bb];
    pg_pre[bb] = Lo > 0 && Lo % a.ps != 0 && Lo / a.ps < a.max_pages
                     ? __ldcg(a.table + (size_t)bb * a.max_pages + Lo / a.ps)
                     : -1;
  }
  // grants in ascending b while free pages last (as select_grant_kernel);
  // rows that wanted a page and got none are compacted here
  if (tid == 0) {
    s_carry[2] = 0;
    s_carry[3] = 0;
  }
  __syncthreads();
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int bb = base + tid;
    const int w = bb < a.B ? __ldcg(a.wants + bb) : 0;
    int x = w;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) red[warp] = x;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += red[i];
    const int carry = s_carry[3];
    const int excl = carry + before + x - w;
    if (bb < a.B && w) {
      if (excl < free_count) {
        a.grow[bb] = 1;
        a.budget[bb] += 1;
        const int nb = (int)ceil_div_ll(__ldcg(a.seq_lens + bb), a.ps);
        uint8_t* kb = a.keep + (size_t)bb * a.max_pages;
        for (int j = 0; j < nb && j < a.max_pages; ++j) kb[j] = 1;
      } else {
        pend[atomicAdd(&s_carry[2], 1)] = bb;
      }
    }
    __syncthreads();
    if (tid == blockDim.x - 1) s_carry[3] = carry + before + x;
    __syncthreads();
  }
  const int npend = s_carry[2];
  for (int i = 0; i < npend; ++i) {
    const int bb = pend[i];
    const int Lb = __ldcg(a.seq_lens + bb);
    int dr = 0;
    __threadfence();
    __syncthreads();
    const int K = compact_row_pages(a.table + (size_t)bb * a.max_pages,
                                    a.keep + (size_t)bb * a.max_pages,
                                    (int)ceil_div_ll(Lb, a.ps), Lb, a.ps, a.max_pages,
                                    a.drop_ids + (size_t)bb * a.max_pages, &dr, red, s_carry);
    if (tid == 0) {
      a.new_len[bb] = K;
      a.drop_cnt[bb] = dr;
    }
    __threadfence();
    __syncthreads();
  }
  // freed pages onto the free list in (b, j) order (no page is popped by a
  // page-granular compaction); one warp per sequence
  int top = free_count;
  {
    if (tid == 0) s_carry[3] = 0;
    __syncthreads();
    for (int base = 0; base < a.B; base += blockDim.x) {
      const int bb = base + tid;
      const int c = bb < a.B ? __ldcg(a.drop_cnt + bb) : 0;
      int x = c;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) red[warp] = x;
      __syncthreads();
      int before = 0;
      for (int i = 0; i < warp; ++i) before += red[i];
      const int carry = s_carry[3];
      if (bb < a.B) {
        pend[bb] = carry + before + x - c;  // exclusive offset of b's pushes
        cnt_s[bb] = c;
      }
      __syncthreads();
      if (tid == blockDim.x - 1) s_carry[3] = carry + before + x;
      __syncthreads();
    }
    const int pushes = s_carry[3];
    for (int bb = warp; bb < a.B; bb += nw) {
      const int c = cnt_s[bb];
      for (int r = lane; r < c; r += 32)
        a.free_list[top + pend[bb] + r] = __ldcg(a.drop_ids + (size_t)bb * a.max_pages + r);
    }
    top += pushes;
  }
  __threadfence();
  __syncthreads();
  // ---- append (as append_plan_kernel + append_copy_kernel, no shared pages).
  // Each sequence's length, its page for the token and the ids to be popped
  // are read once; sequences are taken blockDim at a time.
  int2* dest = reinterpret_cast<int2*>(pend);  // [B] (page, slot)
  if (tid == 0) {
    s_carry[0] = s_carry[1] = 0;
    s_carry[3] = 0;
  }
  __syncthreads();
  int my_need = 0;
  for (int bb = tid; bb < a.B; bb += blockDim.x) {
    const int Lb = __ldcg(a.new_len + bb);
    int pg = -1;
    if (Lb < 0) {
      s_carry[1] = 1;
    } else if (Lb % a.ps == 0) {
      if (Lb / a.ps >= a.max_pages) s_carry[0] = 1;
      ++my_need;
    } else {
      pg = pg_pre[bb];  // Lb is the row's unchanged length here
      if (pg < 0 || pg >= a.num_pages) s_carry[1] = 1;
    }
    dest[bb] = make_int2(pg, Lb);  // (page or -1 for a pop, length) until the pops are known
  }
  const int total = block_sum_int(my_need, red);
  if (total <= top)  // at most one pop per sequence: total <= B
    for (int i = tid; i < total; i += blockDim.x) {
      const int p = __ldcg(a.free_list + (top - 1 - i));
      pops[i] = p;
      if (p < 0 || p >= a.num_pages) s_carry[1] = 1;
    }
  __syncthreads();
  const int err = s_carry[0] ? KV_EFULL : (s_carry[1] ? KV_EBADPAGE : (total > top ? KV_ENOSPACE : 0));
  if (err) {
    // the compaction stands (new_len holds its lengths); the append changes
    // nothing
    if (tid == 0) {
      set_status(a.status, err);
      *a.free_top = top;
      *a.ctl = 1;
      *a.ticket = 0;
    }
    leave();
    return;
  }
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int bb = base + tid;
    const int2 dl = bb < a.B ? dest[bb] : make_int2(0, 1);
    const int Lb = dl.y;
    const bool nd = bb < a.B && Lb % a.ps == 0;
    const unsigned bal = __ballot_sync(FULL, nd);
    const int x = __popc(bal & ((1u << lane) - 1u));
    __syncthreads();
    if (lane == 0) red[warp] = __popc(bal);
    __syncthreads();
    int before = 0;
    for (int i = 0; i < warp; ++i) before += red[i];
    const int carry = s_carry[3];
    if (bb < a.B) {
      int pg = dl.x;
      if (nd) {
        pg = pops[carry + before + x];
        a.table[(size_t)bb * a.max_pages + Lb / a.ps] = pg;
      }
      dest[bb] = make_int2(pg, Lb % a.ps);
      a.new_len[bb] = Lb + 1;  // the final length (all of new_len was read above)
    }
    __syncthreads();
    if (tid == 0) {
      int tot = 0;
      for (int i = 0; i < nw; ++i) tot += red[i];
      s_carry[3] = carry + tot;
    }
    __syncthreads();
  }
  // the copies of the token's K and V rows are step_copy_kernel's
  for (int bb = tid; bb < a.B; bb += blockDim.x) a.dest[bb] = dest[bb];
  if (tid == 0) {
    *a.free_top = top - total;
    *a.ctl = 0;
    *a.ticket = 0;  // ready for the next call
  }
  leave();
}

// The step's token: K and V rows (all heads) of sequence blockIdx.x into the
// (page, slot) the fused step planned (nothing when its append failed), and
// the sequence's final length into seq_lens.
__global__ void __launch_bounds__(128) step_copy_kernel(const StepArgs a) {
  // the decode that follows may be scheduled now (it waits for this grid to
  // finish before it reads anything); this kernel waits for the step's plan
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x;
  if (threadIdx.x == 0) a.seq_lens[b] = a.new_len[b];
  if (*a.ctl) return;
  const int2 dst = a.dest[b];
  const size_t row_bytes = (size_t)a.d * 2;
  const int vec = (int)(row_bytes / 16);
  for (int i = threadIdx.x; i < a.Hkv * vec; i += blockDim.x) {
    const int h = i / vec, v = i - h * vec;
    const size_t so = ((size_t)b * a.Hkv + h) * row_bytes + (size_t)v * 16;
    const size_t dof = (((size_t)dst.x * a.Hkv + h) * a.ps + dst.y) * row_bytes + (size_t)v * 16;
    *reinterpret_cast<uint4*>(a.k_pool + dof) = *reinterpret_cast<const uint4*>(a.k_new + so);
    *reinterpret_cast<uint4*>(a.v_pool + dof) = *reinterpret_cast<const uint4*>(a.v_new + so);
  }
}

bool dtype_ok(int dtype) { return dtype == KV_F16 || dtype == KV_BF16; }

constexpr int kCompactMaxSmem = 200 * 1024;  // shared memory of compact_apply_kernel, at most

size_t ws_take(size_t* off, size_t bytes) {
  size_t o = *off;
  *off = align_up(*off + bytes, 256);
  return o;
}

}  // namespace
}  // namespace kvb

using namespace kvb;

namespace kvb {
namespace {

// Push pool pages [first, first + n) onto the free-list stack, highest id
// first, so the next pops hand them out in ascending order.  One CTA; the
// stack's capacity is checked before anything is written.
__global__ void __launch_bounds__(256) free_push_kernel(int32_t* free_list, int32_t* free_top,
                                                        int capacity, int first, int n,
                                                        int* status) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_top;
  if (threadIdx.x == 0) {
    const int top = *free_top;
    s_top = (top < 0 || (long long)top + n > capacity) ? -1 : top;
    if (s_top < 0) set_status(status, KV_ENOSPACE);
  }
  __syncthreads();
  const int top = s_top;
  if (top < 0) return;
  for (int i = threadIdx.x; i < n; i += blockDim.x) free_list[top + i] = first + n - 1 - i;
  __syncthreads();
  if (threadIdx.x == 0) *free_top = top + n;
}

}  // namespace
}  // namespace kvb

extern "C" {

int kv_update_query_summaries(const void* q, int B, int Hq, int Hkv, int d, int dtype, float a_fast,
                              float a_slow, int first, float* ema, void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || !dtype_ok(dtype)) return KV_EINVAL;
  if (B == 0) return KV_OK;
  if (!q || !ema) return KV_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int threads = d < 128 ? d : 128;
  KV_CUDA_CHECK(launch(dtype == KV_BF16 ? ema_kernel<BF16> : ema_kernel<F16>, dim3(B * Hkv),
                       dim3(threads), 0, s, false, static_cast<const uint16_t*>(q), Hq, Hkv, d,
                       a_fast, a_slow, first, ema));
  return KV_OK;
}

int kv_mark_active(const int32_t* seq_lens, const int32_t* budget, int B, int page_size, int mode,
                   uint8_t* active, void* stream) {
  if (B < 0 || page_size <= 0 || (mode != 0 && mode != 1)) return KV_EINVAL;
  if (B == 0) return KV_OK;
  if (!seq_lens || !budget || !active) return KV_EINVAL;
  KV_CUDA_CHECK(launch(mark_kernel, dim3(ceil_div(B, 256)), dim3(256), 0,
                       static_cast<cudaStream_t>(stream), false, seq_lens, budget, B, page_size,
                       mode, active));
  return KV_OK;
}

static int launch_summaries(const void* k_pool, int num_pages, const int32_t* page_ids, int n,
                            const int32_t* table, int max_pages, const int32_t* seq_lens,
                            const uint8_t* active, int Hkv, int page_size, int d, int dtype,
                            float* summ, void* ws, size_t ws_bytes, void* stream) {
  if (n < 0 || Hkv <= 0 || page_size <= 0 || d <= 0 || num_pages < 0 || !dtype_ok(dtype))
    return KV_EINVAL;
  if (n == 0) return KV_OK;
  if (!k_pool || !summ || !ws || ws_bytes < kHeaderBytes) return KV_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int threads = d < 128 ? d : 128;
  int* status = static_cast<int*>(ws);
  const long long blocks = (long long)n * Hkv;
  if (blocks > 0x7fffffffll) return KV_EINVAL;
  KV_CUDA_CHECK(launch(dtype == KV_BF16 ? summary_kernel<BF16> : summary_kernel<F16>,
                       dim3((unsigned)blocks), dim3(threads), 0, s, false,
                       static_cast<const uint16_t*>(k_pool), num_pages, page_ids, n, table,
                       max_pages, seq_lens, active, Hkv, page_size, d, summ, status));
  return KV_OK;
}

int kv_page_summaries(const void* k_pool, int num_pages, const int32_t* page_ids, int n, int Hkv,
                      int page_size, int d, int dtype, float* summ, void* ws, size_t ws_bytes,
                      void* stream) {
  if (n > 0 && !page_ids) return KV_EINVAL;
  return launch_summaries(k_pool, num_pages, page_ids, n, nullptr, 0, nullptr, nullptr, Hkv,
                          page_size, d, dtype, summ, ws, ws_bytes, stream);
}

int kv_summarize_last_pages(const void* k_pool, int num_pages, const int32_t* block_table,
                            int max_pages, const int32_t* seq_lens, const uint8_t* active, int B,
                            int Hkv, int page_size, int d, int dtype, float* summ, void* ws,
                            size_t ws_bytes, void* stream) {
  if (B > 0 && (!block_table || !seq_lens)) return KV_EINVAL;
  if (max_pages < 0) return KV_EINVAL;
  return launch_summaries(k_pool, num_pages, nullptr, B, block_table, max_pages, seq_lens, active,
                          Hkv, page_size, d, dtype, summ, ws, ws_bytes, stream);
}

int kv_score_pages(const float* query_summaries, const float* page_key_summaries, int num_pages,
                   const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                   const uint8_t* active, int B, int Hkv, int d, int page_size, float* scores,
                   void* ws, size_t ws_bytes, void* stream) {
  if (B < 0 || Hkv <= 0 || page_size <= 0 || max_pages < 0 || (d != 64 && d != 128)) return KV_EINVAL;
  if (B == 0 || max_pages == 0) return KV_OK;
  if (!query_summaries || !page_key_summaries || !block_table || !seq_lens || !scores || !ws ||
      ws_bytes < kHeaderBytes)
    return KV_EINVAL;
  const long long warps = (long long)B * max_pages;
  const int wpb = 8;
  const long long blocks = ceil_div_ll(warps, wpb);
  if (blocks > 0x7fffffffll) return KV_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(ws);
  KV_CUDA_CHECK(launch(d == 128 ? score_kernel<4> : score_kernel<2>, dim3((unsigned)blocks),
                       dim3(wpb * 32), 0, s, false, query_summaries, page_key_summaries, num_pages,
                       block_table, max_pages, seq_lens, active, B, Hkv, page_size, scores,
                       status));
  return KV_OK;
}

size_t kv_select_workspace_size(int B, int max_pages) {
  (void)max_pages;
  size_t off = kHeaderBytes;
  ws_take(&off, (size_t)(B > 0 ? B : 1) * 4);
  return off;
}

// Shared memory of select_rank_kernel for rows of max_pages pages: three
// float keys, the sort's index array (next power of two), ranks, two flags.
static size_t select_smem(int max_pages) {
  size_t p2 = 1;
  while (p2 < (size_t)max_pages) p2 <<= 1;
  return (size_t)max_pages * (3 * sizeof(float) + 2 + 2) + p2 * 2 + 16;
}

int kv_select_pages(const float* scores, const int32_t* seq_lens, const uint8_t* active,
                    int32_t* budget, int B, int max_pages, int page_size, int n_first, int n_last,
                    float delta, float ws_frac, int mode, const int32_t* free_top,
                    uint8_t* keep_mask, uint8_t* grow, int32_t* drift, void* ws, size_t ws_bytes,
                    void* stream) {
  if (B < 0 || max_pages < 0 || page_size <= 0 || n_first < 0 || n_last < 0) return KV_EINVAL;
  if (mode != KV_SELECT_TOPK && mode != KV_SELECT_BOUNDARY) return KV_EINVAL;
  if (max_pages > kMaxSelectPages) return KV_EINVAL;
  if (B == 0) return KV_OK;
  if (!scores || !seq_lens || !budget || !keep_mask || !grow || !ws) return KV_EINVAL;
  if (mode == KV_SELECT_BOUNDARY && !free_top) return KV_EINVAL;
  if (ws_bytes < kv_select_workspace_size(B, max_pages)) return KV_EWORKSPACE;
  SelectArgs a{};
  a.scores = scores;
  a.seq_lens = seq_lens;
  a.active = active;
  a.budget = budget;
  a.B = B;
  a.max_pages = max_pages;
  a.ps = page_size;
  a.n_first = n_first;
  a.n_last = n_last;
  a.mode = mode;
  a.delta = delta;
  a.ws_frac = ws_frac;
  a.keep = keep_mask;
  a.grow = grow;
  a.drift = drift;
  a.status = static_cast<int*>(ws);
  a.wants = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + kHeaderBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t smem = select_smem(max_pages);
  KV_CUDA_CHECK(cudaFuncSetAttribute(select_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)select_smem(kMaxSelectPages)));
  KV_CUDA_CHECK(launch(select_rank_kernel, dim3(B), dim3(kSelThreads), smem, s, false, a));
  if (mode == KV_SELECT_BOUNDARY)
    KV_CUDA_CHECK(launch(select_grant_kernel, dim3(1), dim3(1024), 0, s, false, a, free_top));
  return KV_OK;
}

struct CompactLayout {
  size_t new_len, pop, push, ctl, fresh, freed_flag, page_cnt, page_key, total;
  long long max_fresh;
};
static CompactLayout compact_layout(int B, int max_pages, int num_pages) {
  CompactLayout L{};
  size_t off = kHeaderBytes;
  const size_t nb = (size_t)(B > 0 ? B : 1);
  L.new_len = ws_take(&off, nb * 4);
  L.pop = ws_take(&off, nb * 4);
  L.push = ws_take(&off, nb * 4);
  L.ctl = ws_take(&off, 16);
  L.max_fresh = (long long)nb * (max_pages > 0 ? max_pages : 1);
  L.fresh = ws_take(&off, (size_t)L.max_fresh * 4);
  // shared pages only (num_pages > 0)
  L.freed_flag = ws_take(&off, num_pages > 0 ? (size_t)L.max_fresh : 0);
  L.page_cnt = ws_take(&off, (size_t)(num_pages > 0 ? num_pages : 0) * 4);
  L.page_key = ws_take(&off, (size_t)(num_pages > 0 ? num_pages : 0) * 4);
  L.total = off;
  return L;
}

size_t kv_compact_workspace_size(int B, int max_pages, int num_pages, int token_granular) {
  (void)token_granular;
  return compact_layout(B, max_pages, num_pages).total;
}

int kv_compact(int32_t* block_table, int max_pages, int32_t* seq_lens, const uint8_t* keep_mask,
               int token_granular, void* k_pool, void* v_pool, int num_pages, int32_t* free_list,
               int32_t* free_top, int32_t* refcnt, int B, int Hkv, int d, int page_size,
               int dtype, void* ws, size_t ws_bytes, void* stream) {
  if (B < 0 || max_pages < 0 || Hkv <= 0 || page_size <= 0 || (d % 8) || d <= 0 || !dtype_ok(dtype))
    return KV_EINVAL;
  if (B == 0) return KV_OK;
  if (!block_table || !seq_lens || !keep_mask || !free_list || !free_top || !ws) return KV_EINVAL;
  if (token_granular && (!k_pool || !v_pool || ((uintptr_t)k_pool & 15) || ((uintptr_t)v_pool & 15)))
    return KV_EINVAL;
  const size_t smem = (size_t)3 * max_pages * 4;
  if (smem > (size_t)kCompactMaxSmem) return KV_EINVAL;
  if (refcnt && num_pages < 1) return KV_EINVAL;
  const CompactLayout CL = compact_layout(B, max_pages, refcnt ? num_pages : 0);
  if (ws_bytes < CL.total) return KV_EWORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  CompactArgs a{};
  a.table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.keep = keep_mask;
  a.token_granular = token_granular ? 1 : 0;
  a.k_pool = static_cast<uint8_t*>(k_pool);
  a.v_pool = static_cast<uint8_t*>(v_pool);
  a.num_pages = num_pages;
  a.free_list = free_list;
  a.free_top = free_top;
  a.B = B;
  a.Hkv = Hkv;
  a.d = d;
  a.ps = page_size;
  a.new_len = reinterpret_cast<int32_t*>(w + CL.new_len);
  a.pop_base = reinterpret_cast<int32_t*>(w + CL.pop);
  a.push_base = reinterpret_cast<int32_t*>(w + CL.push);
  a.ctl = reinterpret_cast<int32_t*>(w + CL.ctl);
  a.fresh_ids = reinterpret_cast<int32_t*>(w + CL.fresh);
  a.max_fresh = CL.max_fresh;
  a.status = reinterpret_cast<int*>(w);
  a.refcnt = refcnt;
  a.freed_flag = w + CL.freed_flag;
  a.page_cnt = reinterpret_cast<int32_t*>(w + CL.page_cnt);
  a.page_key = reinterpret_cast<int32_t*>(w + CL.page_key);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (refcnt) {
    const long long blocks = std::min<long long>(1024, ((long long)num_pages + 255) / 256);
    KV_CUDA_CHECK(launch(compact_clear_kernel, dim3((unsigned)blocks), dim3(256), 0, s, false, a));
  }
  KV_CUDA_CHECK(launch(compact_count_kernel, dim3(B), dim3(kCountThreads), 0, s, false, a));
  if (refcnt)
    KV_CUDA_CHECK(launch(compact_free_kernel, dim3(B), dim3(kCountThreads), 0, s, false, a));
  KV_CUDA_CHECK(launch(compact_scan_kernel, dim3(1), dim3(1024), 0, s, false, a));
  if (smem > 48 * 1024)  // one fixed limit for every call (the attribute is per function)
    KV_CUDA_CHECK(cudaFuncSetAttribute(compact_apply_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kCompactMaxSmem));
  KV_CUDA_CHECK(launch(compact_apply_kernel, dim3(B), dim3(kApplyThreads), smem, s, false, a));
  return KV_OK;
}

struct StepLayout {
  size_t wants, new_len, drop_cnt, row_tk, dest, drop_ids, total;
};
static StepLayout step_layout(int B, int max_pages) {
  StepLayout L{};
  size_t off = kHeaderBytes;
  const size_t nb = (size_t)(B > 0 ? B : 1);
  L.wants = ws_take(&off, nb * 4);
  L.new_len = ws_take(&off, nb * 4);
  L.drop_cnt = ws_take(&off, nb * 4);
  L.row_tk = ws_take(&off, nb * 4);
  L.dest = ws_take(&off, nb * 8);
  L.drop_ids = ws_take(&off, nb * (size_t)(max_pages > 0 ? max_pages : 1) * 4);
  L.total = off;
  return L;
}

// Dynamic shared memory of budget_step_kernel: the row's EMAs, then the
// larger of the selection's arrays (three keys, the sort's index array above
// 1024 pages, two ranks, the candidate flags) and the last block's per-row
// scratch.
static size_t step_smem(int B, int Hkv, int d, int max_pages) {
  size_t p2 = 1;
  while (p2 < (size_t)max_pages) p2 <<= 1;
  // packed keys, R, flags, ranks (two), unpacked keys above 1024 pages
  const size_t sel = (size_t)max_pages * (8 + 4 + 1 + 2 + 2 + 8) + p2 * 2 + 32;
  return (size_t)2 * Hkv * d * 4 + std::max(align_up(sel, 16), (size_t)B * 16);
}

size_t kv_budget_step_workspace_size(int B, int max_pages) { return step_layout(B, max_pages).total; }

int kv_budget_step(const void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                   int num_pages, int32_t* block_table, int max_pages, int32_t* seq_lens,
                   int32_t* budget, int B, int Hq, int Hkv, int d, int page_size, int dtype,
                   float a_fast, float a_slow, int update_ema, int n_first, int n_last, float delta,
                   float ws_frac, float* ema, float* summ, float* scores, uint8_t* active,
                   uint8_t* keep_mask, uint8_t* grow, int32_t* drift, int32_t* free_list,
                   int32_t* free_top, void* ws, size_t ws_bytes, void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || (d != 64 && d != 128) || page_size <= 0 ||
      max_pages < 1 || max_pages > kMaxSelectPages || n_first < 0 || n_last < 0 || num_pages < 1 ||
      !dtype_ok(dtype))
    return KV_EINVAL;
  if (B == 0) return KV_OK;
  if (!q || !k_new || !v_new || !k_pool || !v_pool || !block_table || !seq_lens || !budget ||
      !ema || !summ || !scores || !active || !keep_mask || !grow || !free_list || !free_top || !ws)
    return KV_EINVAL;
  if (((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)k_pool | (uintptr_t)v_pool) & 15)
    return KV_EINVAL;
  const StepLayout L = step_layout(B, max_pages);
  if (ws_bytes < L.total) return KV_EWORKSPACE;
  const size_t smem = step_smem(B, Hkv, d, max_pages);
  int dev = 0, optin = 0;
  KV_CUDA_CHECK(cudaGetDevice(&dev));
  KV_CUDA_CHECK(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
  uint8_t* w = static_cast<uint8_t*>(ws);
  StepArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.k_new = static_cast<const uint8_t*>(k_new);
  a.v_new = static_cast<const uint8_t*>(v_new);
  a.k_pool = static_cast<uint8_t*>(k_pool);
  a.v_pool = static_cast<uint8_t*>(v_pool);
  a.num_pages = num_pages;
  a.table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.budget = budget;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.ps = page_size;
  a.a_fast = a_fast;
  a.a_slow = a_slow;
  a.n_first = n_first;
  a.n_last = n_last;
  a.delta = delta;
  a.ws_frac = ws_frac;
  a.update_ema = update_ema ? 1 : 0;
  a.ema = ema;
  a.summ = summ;
  a.scores = scores;
  a.active = active;
  a.keep = keep_mask;
  a.grow = grow;
  a.drift = drift;
  a.free_list = free_list;
  a.free_top = free_top;
  a.wants = reinterpret_cast<int32_t*>(w + L.wants);
  a.new_len = reinterpret_cast<int32_t*>(w + L.new_len);
  a.drop_cnt = reinterpret_cast<int32_t*>(w + L.drop_cnt);
  a.drop_ids = reinterpret_cast<int32_t*>(w + L.drop_ids);
  a.row_tk = reinterpret_cast<int32_t*>(w + L.row_tk);
  a.dest = reinterpret_cast<int2*>(w + L.dest);
  a.S = kStepSplit;
  a.ticket = reinterpret_cast<unsigned*>(w + kStepTicketOffset);
  a.grab = reinterpret_cast<unsigned*>(w + kStepGrabOffset);
  a.exits = reinterpret_cast<unsigned*>(w + kStepExitOffset);
  a.ctl = reinterpret_cast<int*>(w + kStepCtlOffset);
  a.status = reinterpret_cast<int*>(w);
  using StepFn = void (*)(const StepArgs);
  StepFn fn = dtype == KV_BF16 ? (d == 128 ? budget_step_kernel<BF16, 4> : budget_step_kernel<BF16, 2>)
                               : (d == 128 ? budget_step_kernel<F16, 4> : budget_step_kernel<F16, 2>);
  cudaFuncAttributes fa{};
  KV_CUDA_CHECK(cudaFuncGetAttributes(&fa, fn));
  if (smem + fa.sharedSizeBytes > (size_t)optin) return KV_EINVAL;  // rows too wide for one block
  KV_CUDA_CHECK(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  // a resident grid: every block is scheduled at once and takes items
  // (sequence, split) in turn
  int sms = 0, per_sm = 0;
  KV_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  KV_CUDA_CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kStepThreads, smem));
  if (per_sm < 1) return cuda_failed(cudaErrorInvalidConfiguration, "budget step occupancy");
  const long long grid = std::min<long long>((long long)B * kStepSplit, (long long)sms * per_sm);
  KV_CUDA_CHECK(launch(fn, dim3((unsigned)grid), dim3(kStepThreads), smem,
                       static_cast<cudaStream_t>(stream), false, a));
  KV_CUDA_CHECK(launch(step_copy_kernel, dim3(B), dim3(128), 0, static_cast<cudaStream_t>(stream),
                       true, a));
  return KV_OK;
}

int kv_free_list_push(int first_page, int n, int32_t* free_list, int capacity, int32_t* free_top,
                      void* ws, void* stream) {
  if (first_page < 0 || n < 0 || capacity < 0 || (long long)first_page + n > 0x7fffffffll)
    return KV_EINVAL;
  if (n == 0) return KV_OK;
  if (!free_list || !free_top || !ws) return KV_EINVAL;
  KV_CUDA_CHECK(launch(free_push_kernel, dim3(1), dim3(256), 0, static_cast<cudaStream_t>(stream),
                       true, free_list, free_top, capacity, first_page, n, static_cast<int*>(ws)));
  return KV_OK;
}

size_t kv_append_workspace_size(int B) {
  size_t off = kHeaderBytes;
  const size_t nb = (size_t)(B > 0 ? B : 1);
  ws_take(&off, nb * 8);   // dest
  ws_take(&off, 16);       // ctl
  ws_take(&off, nb * 4);   // cand
  ws_take(&off, nb * 4);   // cow_src
  return off;
}

int kv_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool, int num_pages,
              int32_t* block_table, int max_pages, int32_t* seq_lens, int32_t* free_list,
              int32_t* free_top, int32_t* refcnt, int B, int Hkv, int d, int page_size, int dtype,
              void* ws, size_t ws_bytes, void* stream) {
  if (B < 0 || max_pages < 0 || Hkv <= 0 || page_size <= 0 || d <= 0 || (d % 8) || !dtype_ok(dtype))
    return KV_EINVAL;
  if (B == 0) return KV_OK;
  if (!k_new || !v_new || !k_pool || !v_pool || !block_table || !seq_lens || !free_list ||
      !free_top || !ws)
    return KV_EINVAL;
  if (((uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)k_pool | (uintptr_t)v_pool) & 15)
    return KV_EINVAL;
  if (ws_bytes < kv_append_workspace_size(B)) return KV_EWORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  size_t off = kHeaderBytes;
  const size_t o_dest = ws_take(&off, (size_t)B * 8);
  const size_t o_ctl = ws_take(&off, 16);
  const size_t o_cand = ws_take(&off, (size_t)B * 4);
  const size_t o_cow = ws_take(&off, (size_t)B * 4);
  AppendArgs a{};
  a.k_new = static_cast<const uint8_t*>(k_new);
  a.v_new = static_cast<const uint8_t*>(v_new);
  a.k_pool = static_cast<uint8_t*>(k_pool);
  a.v_pool = static_cast<uint8_t*>(v_pool);
  a.num_pages = num_pages;
  a.table = block_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.free_list = free_list;
  a.free_top = free_top;
  a.B = B;
  a.Hkv = Hkv;
  a.d = d;
  a.ps = page_size;
  a.dest = reinterpret_cast<int2*>(w + o_dest);
  a.ctl = reinterpret_cast<int32_t*>(w + o_ctl);
  a.status = reinterpret_cast<int*>(w);
  a.refcnt = refcnt;
  a.cand = reinterpret_cast<int32_t*>(w + o_cand);
  a.cow_src = reinterpret_cast<int32_t*>(w + o_cow);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  KV_CUDA_CHECK(launch(append_plan_kernel, dim3(1), dim3(1024), 0, s, false, a));
  if (refcnt) KV_CUDA_CHECK(launch(append_cow_kernel, dim3(B), dim3(128), 0, s, false, a));
  KV_CUDA_CHECK(launch(append_copy_kernel, dim3(B), dim3(128), 0, s, false, a));
  return KV_OK;
}

}  // extern "C"
