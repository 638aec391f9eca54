// Split-KV GQA decode over a paged KV cache, with the split merge fused in.
//
// What is computed (PersistentKV, aissential.tech -- Summary, Method): for each
// sequence and query head, softmax attention of the one new query over the
// sequence's tokens, read through its block table; the K/V tile of each
// (page, KV head) is loaded once and used for all G query heads of that KV
// head; the work is a compact list of non-empty (sequence, KV head, split)
// tasks, and the splits of a sequence are recombined exactly by their
// log-sum-exp.
//
// How (this library's design for sm_103a), one launch per decode step:
//  * Prologue (every CTA): page offsets O_b of the batch by a block-wide scan
//    of seq_lens into shared memory (batches above kFusedMaxB read them from
//    a small offsets kernel instead), the chunk size, and out = 0 /
//    lse = -inf for sequences without tokens.
//  * One persistent CTA per SM slot walks chunks c = blockIdx.x, + gridDim.x,
//    ...; the non-empty splits of chunk c are the sequences whose page range
//    meets it (found by binary search on O), i.e. the CTA builds the slice of
//    the workqueue it executes.  A CTA has one producer warp and one consumer
//    warp per KV head.  A "stage" is one logical page of one sequence for all
//    KV heads: the page's K block [Hkv][16][d] and V block are each one
//    contiguous run in the pool, fetched by two cp.async.bulk copies (plus
//    the sequence's q on its first page) that complete on the stage's
//    mbarrier.  Stages form a ring of S slots; the consumers release a slot
//    through a second mbarrier.
//  * Consumer warp h computes its head's tile: q.k for 16 tokens x G query
//    heads with 8 lanes per token row (16-byte shared loads, partial dots
//    reduce-scattered over the 8 lanes), an online softmax in base 2, and
//    p.v with each lane owning d/32 output channels of all G heads.
//  * A sequence with one split writes out/lse directly.  Otherwise each split
//    writes its normalised partial (o, base-2 lse) to one of two slots of its
//    chunk (slot 2c + 1: the split that starts in chunk c and continues past
//    it; slot 2c: the split that began in an earlier chunk), then takes a
//    ticket on a counter; the split that draws the last ticket merges the
//    partials (lse = log-sum-exp of the parts, out = the lse-weighted sum)
//    and puts the counter back to zero.  Up to 8 splits are merged at once;
//    a longer sequence's splits are merged in groups of about sqrt(splits)
//    and then the groups, which spreads the merge traffic over the SMs that
//    finish each group.  No CTA ever waits on another.
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "kv_internal.h"

namespace kvb {
namespace {

constexpr int PS = 16;                      // tokens per page
constexpr unsigned FULL = 0xffffffffu;
constexpr int kFirst = 1, kLast = 2, kSingle = 4, kDone = 8;
constexpr int kMaxStages = 8;
constexpr int kHeaderStageBytes = 16;
constexpr int kDecodeThreadsMax = 32 * 9;
constexpr int kDirectMerge = 8;  // splits merged in one pass; more go through groups
// shared memory header: barriers, abort flag, chunk parameters, scan scratch
constexpr int kSmemAbort = 16 * kMaxStages;       // int
constexpr int kSmemParams = kSmemAbort + 16;      // long long chunk, nchunks, W
constexpr int kSmemScan = kSmemParams + 32;       // long long [32]
constexpr int kSmemDead = kSmemScan + 32 * 8;     // mbarrier nothing completes (test mode)
constexpr int kSmemHeader = 1024;
static_assert(kSmemDead + 8 <= kSmemHeader, "shared header");

struct DecodeParams {
  const uint8_t* q;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const int32_t* table;
  const int32_t* seq_lens;
  const int32_t* page_off;  // [B + 1] from the offsets kernel, or NULL (computed here)
  float* out;
  float* lse;
  float* part_o;            // [slots][Hkv][G][D]
  float* part_lse;          // [slots][Hkv][G], base 2
  int32_t* row_done;        // [B][Hkv] merge tickets (zero between calls)
  int32_t* group_done;      // [slots][Hkv] group-merge tickets (zero between calls)
  int* status;
  long long chunk_req;      // > 0: pages per chunk; 0: automatic
  long long max_slots;      // partial slots the workspace holds
  int B, num_pages, max_pages, Hq, Hkv, stages, min_chunk;
  float scale_log2;         // softmax scale * log2(e)
  uint32_t kv_bytes;        // one page, all KV heads: Hkv * 16 * d * 2
  uint32_t q_bytes;         // one sequence's q: Hq * d * 2
  uint32_t stage_bytes;     // K + V + q + header, 128-byte multiple
  uint32_t off_pbuf, off_offsets, off_stages;
  unsigned long long test_wait_ns;  // > 0: failure-path test mode (see test_consumer_wait_ns)
};

__host__ __device__ constexpr uint32_t stage_header_offset(uint32_t kv_bytes, uint32_t q_bytes) {
  return 2 * kv_bytes + q_bytes;
}

template <int D, int G, class T>
__global__ void __launch_bounds__(kDecodeThreadsMax, 1) decode_kernel(const DecodeParams p) {
  constexpr int CH = D / 8;                 // q.k channels per lane (8 lanes per row)
  constexpr int CPL = D / 32;               // p.v output channels per lane
  constexpr int NV = G >= 2 ? G / 2 : 1;    // scores a lane holds after the reduction
  static_assert(D == 64 || D == 128, "d");
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "G");

  extern __shared__ __align__(1024) uint8_t smem[];
  const int S = p.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[S], empty[S]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemAbort);
  long long* params = reinterpret_cast<long long*>(smem + kSmemParams);
  long long* scan_sm = reinterpret_cast<long long*>(smem + kSmemScan);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x, nth = blockDim.x;
  const int B = p.B;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[kMaxStages + s]), p.Hkv);
    }
    mbar_init(smem_u32(smem + kSmemDead), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Inputs (seq_lens, tables, pools, offsets) may come from the previous
  // kernel on the stream: wait for it before reading any of them.
  pdl_wait();
  pdl_launch_dependents();

  // ---- prologue: page offsets, chunk size, outputs of empty sequences
  // Every producer reads block-table entries right after the offsets: have
  // the table on its way to L2 meanwhile (spread over all CTAs).
  {
    const size_t lines = ((size_t)B * p.max_pages * 4 + 127) / 128;
    const char* tb = reinterpret_cast<const char*>(p.table);
    for (size_t i = (size_t)blockIdx.x * nth + tid; i < lines && i < (1u << 20);
         i += (size_t)gridDim.x * nth)
      prefetch_l2(tb + i * 128);
  }
  const int32_t* O;
  if (p.page_off) {
    O = p.page_off;
  } else {
    int32_t* Os = reinterpret_cast<int32_t*>(smem + p.off_offsets);
    const int per = ceil_div(B, nth);
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    long long mine = 0;
    bool bad = false;
    for (int b = b0; b < b1; ++b) {
      const int L = __ldg(p.seq_lens + b);
      long long np = L > 0 ? ceil_div_ll(L, PS) : 0;
      if (L < 0 || np > p.max_pages) {
        bad = true;
        np = 0;
      }
      Os[b] = (int32_t)np;
      mine += np;
    }
    long long off;
    const long long W = block_exclusive_scan(mine, &off, scan_sm);
    const bool overflow = W > 0x7fffffffll;
    if ((bad || overflow) && blockIdx.x == 0) set_status(p.status, KV_EINVAL);
    for (int b = b0; b < b1; ++b) {
      const int np = Os[b];
      Os[b] = overflow ? 0 : (int32_t)off;
      off += np;
    }
    if (tid == 0) Os[B] = overflow ? 0 : (int32_t)W;
    __syncthreads();
    O = Os;
  }
  if (tid == 0) {
    const long long W = O[B];
    const long long chunk = p.chunk_req > 0 ? p.chunk_req : auto_chunk(W, gridDim.x, p.min_chunk);
    long long nchunks = W > 0 ? ceil_div_ll(W, chunk) : 0;
    if (2 * nchunks > p.max_slots) {
      if (blockIdx.x == 0) set_status(p.status, KV_EWORKSPACE);
      nchunks = -1;  // nothing is decoded; every output row is written empty
    }
    params[0] = chunk;
    params[1] = nchunks;
  }
  __syncthreads();
  const long long chunk = params[0];
  const bool overflow = params[1] < 0;
  const long long nchunks = overflow ? 0 : params[1];
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    if (O[b + 1] > O[b] && !overflow) continue;
    float* ob = p.out + (size_t)b * p.Hq * D;
    for (int i = tid; i < p.Hq * D; i += nth) ob[i] = 0.f;
    for (int i = tid; i < p.Hq; i += nth) p.lse[(size_t)b * p.Hq + i] = -INFINITY;
  }

  const uint32_t hdr_off = stage_header_offset(p.kv_bytes, p.q_bytes);
  uint8_t* stages = smem + p.off_stages;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_evict_first();
    int slot = 0, round = 0;
    bool aborted = false;
    for (long long c = blockIdx.x; c < nchunks && !aborted; c += gridDim.x) {
      const long long c0 = c * chunk, c1 = min((long long)O[B], c0 + chunk);
      for (int b = seq_at(O, B, c0); b < B && O[b] < c1 && !aborted; ++b) {
        const long long Ob = O[b], np = O[b + 1] - Ob;
        if (np == 0) continue;
        const long long ns = split_count(Ob, np, chunk);
        const long long s = c - Ob / chunk;
        long long lo, hi;
        split_range(Ob, np, chunk, c, &lo, &hi);
        const int p0 = (int)lo, p1 = (int)hi;
        const int slot_id = ns == 1 ? -1 : (int)(2 * c + (s == 0 ? 1 : 0));
        const int L = __ldg(p.seq_lens + b);
        const int32_t* trow = p.table + (size_t)b * p.max_pages;
        for (int jw = p0; jw < p1 && !aborted; jw += 32) {
          const int j = jw + lane;
          int id = 0;
          if (j < p1) {
            id = __ldg(trow + j);
            if (id < 0 || id >= p.num_pages) {
              set_status(p.status, KV_EBADPAGE);
              id = 0;
            }
          }
          const int n = min(32, p1 - jw);
          for (int i = 0; i < n; ++i) {
            const int pid = __shfl_sync(FULL, id, i);
            if (lane == 0) {
              bool ok = true;
              if (round > 0)
                ok = mbar_wait(smem_u32(&bars[kMaxStages + slot]), (round - 1) & 1, kWaitLimitNs,
                               abort_flag);
              if (!ok) {
                set_status(p.status, KV_ETIMEOUT);  // no-op when a consumer already set it
                *abort_flag = 1;
                aborted = true;
              } else {
                const int jj = jw + i;
                const int flags = (jj == p0 ? kFirst : 0) | (jj == p1 - 1 ? kLast : 0) |
                                  (ns == 1 ? kSingle : 0);
                const int nvalid = min(PS, L - jj * PS);
                uint8_t* st = stages + (size_t)slot * p.stage_bytes;
                *reinterpret_cast<int4*>(st + hdr_off) = make_int4(b, flags, nvalid, slot_id);
                const uint32_t bar = smem_u32(&bars[slot]);
                mbar_arrive_expect_tx(bar, 2 * p.kv_bytes + ((flags & kFirst) ? p.q_bytes : 0));
                bulk_g2s(smem_u32(st), p.k_pool + (size_t)pid * p.kv_bytes, p.kv_bytes, bar, pol);
                bulk_g2s(smem_u32(st + p.kv_bytes), p.v_pool + (size_t)pid * p.kv_bytes,
                         p.kv_bytes, bar, pol);
                if (flags & kFirst)
                  bulk_g2s(smem_u32(st + 2 * p.kv_bytes), p.q + (size_t)b * p.q_bytes, p.q_bytes,
                           bar, pol);
              }
            }
            aborted = __shfl_sync(FULL, aborted, 0);
            if (aborted) break;
            if (++slot == S) { slot = 0; ++round; }
          }
        }
      }
    }
    if (lane == 0) {
      if (!aborted) {
        // end-of-stream marker: a stage with no data
        bool ok = true;
        if (round > 0)
          ok = mbar_wait(smem_u32(&bars[kMaxStages + slot]), (round - 1) & 1, kWaitLimitNs,
                         abort_flag);
        if (ok) {
          uint8_t* st = stages + (size_t)slot * p.stage_bytes;
          *reinterpret_cast<int4*>(st + hdr_off) = make_int4(0, kDone, 0, -1);
          mbar_arrive(smem_u32(&bars[slot]));
        } else {
          set_status(p.status, KV_ETIMEOUT);
          *abort_flag = 1;
          aborted = true;
        }
      }
      if (aborted) {
        // Let copies already issued land before the CTA's shared memory goes
        // away: the last phase issued on each slot (bounded waits).
        for (int s = 0; s < S; ++s) {
          const int issued = s < slot ? round + 1 : round;
          if (issued > 0) mbar_wait(smem_u32(&bars[s]), (issued - 1) & 1);
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int h = warp - 1;
  const int tq = lane >> 3, c8 = lane & 7;
  const int bit2 = (c8 >> 2) & 1, bit1 = (c8 >> 1) & 1, bit0 = c8 & 1;
  const int my_t = 4 * (2 * bit2 + bit1) + tq;   // token whose scores this lane ends with
  const int rot = (CH == 16) ? bit2 : 0;         // 16-byte chunk order (bank spread)
  float* pbuf = reinterpret_cast<float*>(smem + p.off_pbuf) + h * PS * G;
  auto part_index = [&](long long slot) { return (size_t)slot * p.Hkv + h; };

  // Ticket on a completion counter of n arrivals: true for the last one.
  // The warp's partial writes are ordered before the ticket by the warp
  // barrier and published by the atomic's release; the winner's acquire
  // orders its reads of the other splits' partials after it.
  auto ticket = [&](int32_t* ctr, int n) -> bool {
    __syncwarp();
    int prev = 0;
    if (lane == 0) prev = atom_add_acq_rel_gpu(ctr, 1);
    prev = __shfl_sync(FULL, prev, 0);
    __syncwarp();
    if (prev >= n) {  // the counter did not start at zero
      if (lane == 0) set_status(p.status, KV_EWORKSPACE);
      return false;
    }
    return prev == n - 1;
  };
  // Merge n partials of this head (partial i in slot slot_of(i)):
  //   L = log2 sum_i 2^{lse_i},  o = sum_i 2^{lse_i - L} o_i
  // into the final out/lse of sequence b (natural-log lse) or into the
  // partial slot dst_slot (normalised o, base-2 lse).  Up to 32 parts: lane
  // i reads part i's lse once and holds its weights, which the accumulation
  // takes by shuffle while it keeps four parts' loads in flight.
  auto merge = [&](int n, auto slot_of, int b, long long dst_slot) {
    float acc[G][CPL];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[g][c] = 0.f;
    float L2[G];
    auto accumulate = [&](int i, const float* w) {
      const float* po = p.part_o + part_index(slot_of(i)) * G * D + lane * CPL;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if constexpr (CPL == 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(po + (size_t)g * D));
          acc[g][0] = fmaf(w[g], v.x, acc[g][0]);
          acc[g][1] = fmaf(w[g], v.y, acc[g][1]);
          acc[g][2] = fmaf(w[g], v.z, acc[g][2]);
          acc[g][3] = fmaf(w[g], v.w, acc[g][3]);
        } else {
          const float2 v = __ldcg(reinterpret_cast<const float2*>(po + (size_t)g * D));
          acc[g][0] = fmaf(w[g], v.x, acc[g][0]);
          acc[g][1] = fmaf(w[g], v.y, acc[g][1]);
        }
      }
    };
    if (n <= 32) {
      float lv[G], wl[G];
#pragma unroll
      for (int g = 0; g < G; ++g) lv[g] = -INFINITY;
      if (lane < n) {
        const float* pl = p.part_lse + part_index(slot_of(lane)) * G;
#pragma unroll
        for (int g = 0; g < G; ++g) lv[g] = __ldcg(pl + g);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mx = lv[g];
#pragma unroll
        for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, off));
        float e = lane < n ? ex2(lv[g] - mx) : 0.f;
        float sum = e;
#pragma unroll
        for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(FULL, sum, off);
        L2[g] = mx + log2f(sum);
        wl[g] = lane < n ? ex2(lv[g] - L2[g]) : 0.f;
      }
      int i = 0;
      for (; i + 4 <= n; i += 4) {
        float w[4][G];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int g = 0; g < G; ++g) w[j][g] = __shfl_sync(FULL, wl[g], i + j);
#pragma unroll
        for (int j = 0; j < 4; ++j) accumulate(i + j, w[j]);
      }
      for (; i < n; ++i) {
        float w[G];
#pragma unroll
        for (int g = 0; g < G; ++g) w[g] = __shfl_sync(FULL, wl[g], i);
        accumulate(i, w);
      }
    } else {
      float mx[G], sum[G];
#pragma unroll
      for (int g = 0; g < G; ++g) { mx[g] = -INFINITY; sum[g] = 0.f; }
      for (int i = lane; i < n; i += 32) {
        const float* pl = p.part_lse + part_index(slot_of(i)) * G;
#pragma unroll
        for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], __ldcg(pl + g));
      }
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int off = 16; off; off >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(FULL, mx[g], off));
      for (int i = lane; i < n; i += 32) {
        const float* pl = p.part_lse + part_index(slot_of(i)) * G;
#pragma unroll
        for (int g = 0; g < G; ++g) sum[g] += ex2(__ldcg(pl + g) - mx[g]);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int off = 16; off; off >>= 1) sum[g] += __shfl_xor_sync(FULL, sum[g], off);
        L2[g] = mx[g] + log2f(sum[g]);
      }
#pragma unroll 2
      for (int i = 0; i < n; ++i) {
        const float* pl = p.part_lse + part_index(slot_of(i)) * G;
        float w[G];
#pragma unroll
        for (int g = 0; g < G; ++g) w[g] = ex2(__ldcg(pl + g) - L2[g]);
        accumulate(i, w);
      }
    }
    __syncwarp();  // every lane has read the sources before any overwrite
    const bool final_out = dst_slot < 0;
    float* dst_o = final_out ? p.out + ((size_t)b * p.Hq + (size_t)h * G) * D
                             : p.part_o + part_index(dst_slot) * G * D;
    float* dst_l = final_out ? p.lse + (size_t)b * p.Hq + (size_t)h * G
                             : p.part_lse + part_index(dst_slot) * G;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* d = dst_o + (size_t)g * D + lane * CPL;
      if constexpr (CPL == 4)
        *reinterpret_cast<float4*>(d) = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
      else
        *reinterpret_cast<float2*>(d) = make_float2(acc[g][0], acc[g][1]);
      if (lane == g) dst_l[g] = final_out ? L2[g] * 0.6931471805599453f : L2[g];
    }
  };

  // test mode: a bounded wait on a barrier nothing completes runs out here,
  // and the warp takes the same way out as any wait that runs out
  if (p.test_wait_ns && !mbar_wait(smem_u32(smem + kSmemDead), 0, p.test_wait_ns)) {
    set_status(p.status, KV_ETIMEOUT);
    *abort_flag = 1;
    return;
  }
  int slot = 0, round = 0;
  for (;;) {  // one task (sequence, KV head h, split) per iteration
    if (!mbar_wait(smem_u32(&bars[slot]), round & 1)) {
      set_status(p.status, KV_ETIMEOUT);
      *abort_flag = 1;
      break;
    }
    const uint8_t* st = stages + (size_t)slot * p.stage_bytes;
    int4 hdr = *reinterpret_cast<const int4*>(st + hdr_off);
    if (hdr.y & kDone) break;
    // the first page of a task carries q: rows h*G .. h*G+G-1 of the
    // sequence, this lane's 8-lane slice, rotated like K
    float qr[G][CH];
    {
      const uint8_t* qs = st + 2 * p.kv_bytes + (size_t)h * G * D * 2;
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int half = 0; half < CH / 8; ++half) {
          const int chunk8 = half ^ rot;
          const uint4 v = *reinterpret_cast<const uint4*>(qs + ((size_t)g * D + c8 * CH + chunk8 * 8) * 2);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = T::to_f2(w[e]);
            qr[g][half * 8 + 2 * e] = f.x * p.scale_log2;
            qr[g][half * 8 + 2 * e + 1] = f.y * p.scale_log2;
          }
        }
      }
    }
    float o[G][CPL];
    float m_run[G];
    float l_part[NV];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -INFINITY;
#pragma unroll
      for (int c = 0; c < CPL; ++c) o[g][c] = 0.f;
    }
#pragma unroll
    for (int n = 0; n < NV; ++n) l_part[n] = 0.f;

    bool timed_out = false;
    for (;;) {  // the task's pages
      const int nvalid = hdr.z;
      // ---- scores: 4 token rows per step, 8 lanes per row
      const uint8_t* Kt = st + (size_t)h * PS * D * 2;
      float acc[4 * G];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = 4 * i + tq;
        float kf[CH];
#pragma unroll
        for (int half = 0; half < CH / 8; ++half) {
          const int chunk8 = half ^ rot;
          const uint4 v = *reinterpret_cast<const uint4*>(Kt + ((size_t)t * D + c8 * CH + chunk8 * 8) * 2);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = T::to_f2(w[e]);
            kf[half * 8 + 2 * e] = f.x;
            kf[half * 8 + 2 * e + 1] = f.y;
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float s = 0.f;
#pragma unroll
          for (int e = 0; e < CH; ++e) s = fmaf(qr[g][e], kf[e], s);
          acc[i * G + g] = s;
        }
      }
      // reduce-scatter over the 8 lanes of a row: xor 4, 2, 1
      float r1[2 * G];
#pragma unroll
      for (int n = 0; n < 2 * G; ++n) {
        const float keep = bit2 ? acc[2 * G + n] : acc[n];
        const float send = bit2 ? acc[n] : acc[2 * G + n];
        r1[n] = keep + __shfl_xor_sync(FULL, send, 4);
      }
      float r2[G];
#pragma unroll
      for (int n = 0; n < G; ++n) {
        const float keep = bit1 ? r1[G + n] : r1[n];
        const float send = bit1 ? r1[n] : r1[G + n];
        r2[n] = keep + __shfl_xor_sync(FULL, send, 2);
      }
      float sc[NV];
      if constexpr (G >= 2) {
#pragma unroll
        for (int n = 0; n < NV; ++n) {
          const float keep = bit0 ? r2[NV + n] : r2[n];
          const float send = bit0 ? r2[n] : r2[NV + n];
          sc[n] = keep + __shfl_xor_sync(FULL, send, 1);
        }
      } else {
        sc[0] = r2[0] + __shfl_xor_sync(FULL, r2[0], 1);
      }
      const bool valid = my_t < nvalid;
#pragma unroll
      for (int n = 0; n < NV; ++n) sc[n] = valid ? sc[n] : -INFINITY;

      // ---- online softmax (base 2)
      float mx[NV];
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        float x = sc[n];
        x = fmaxf(x, __shfl_xor_sync(FULL, x, 2));
        x = fmaxf(x, __shfl_xor_sync(FULL, x, 4));
        x = fmaxf(x, __shfl_xor_sync(FULL, x, 8));
        x = fmaxf(x, __shfl_xor_sync(FULL, x, 16));
        mx[n] = x;
      }
      float m_page[G];
      if constexpr (G >= 2) {
#pragma unroll
        for (int n = 0; n < NV; ++n) {
          const float other = __shfl_xor_sync(FULL, mx[n], 1);
          m_page[n] = bit0 ? other : mx[n];
          m_page[NV + n] = bit0 ? mx[n] : other;
        }
      } else {
        m_page[0] = mx[0];
      }
      float alpha[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mn = fmaxf(m_run[g], m_page[g]);
        alpha[g] = ex2(m_run[g] - mn);
        m_run[g] = mn;
      }
      float pv[NV];
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        const float mg = (G >= 2 && bit0) ? m_run[NV + n] : m_run[n];
        const float ag = (G >= 2 && bit0) ? alpha[NV + n] : alpha[n];
        pv[n] = ex2(sc[n] - mg);
        l_part[n] = l_part[n] * ag + pv[n];
      }
      {
        float* dst = pbuf + my_t * G + (G >= 2 ? bit0 * NV : 0);
        if constexpr (NV == 4) {
          *reinterpret_cast<float4*>(dst) = make_float4(pv[0], pv[1], pv[2], pv[3]);
        } else if constexpr (NV == 2) {
          *reinterpret_cast<float2*>(dst) = make_float2(pv[0], pv[1]);
        } else {
          if (G >= 2 || bit0 == 0) dst[0] = pv[0];
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < CPL; ++c) o[g][c] *= alpha[g];
      __syncwarp();

      // ---- o += p v, lane owns channels lane*CPL .. +CPL
      const uint8_t* Vt = st + p.kv_bytes + (size_t)h * PS * D * 2;
      auto pv_row = [&](int t) {
        float vf[CPL];
        if constexpr (CPL == 4) {
          const uint2 v = *reinterpret_cast<const uint2*>(Vt + ((size_t)t * D + lane * 4) * 2);
          const float2 a0 = T::to_f2(v.x), a1 = T::to_f2(v.y);
          vf[0] = a0.x; vf[1] = a0.y; vf[2] = a1.x; vf[3] = a1.y;
        } else {
          const uint32_t v = *reinterpret_cast<const uint32_t*>(Vt + ((size_t)t * D + lane * 2) * 2);
          const float2 a0 = T::to_f2(v);
          vf[0] = a0.x; vf[1] = a0.y;
        }
        float pg[G];
        if constexpr (G == 8) {
          const float4 x = *reinterpret_cast<const float4*>(pbuf + t * G);
          const float4 y = *reinterpret_cast<const float4*>(pbuf + t * G + 4);
          pg[0] = x.x; pg[1] = x.y; pg[2] = x.z; pg[3] = x.w;
          pg[4] = y.x; pg[5] = y.y; pg[6] = y.z; pg[7] = y.w;
        } else if constexpr (G == 4) {
          const float4 x = *reinterpret_cast<const float4*>(pbuf + t * G);
          pg[0] = x.x; pg[1] = x.y; pg[2] = x.z; pg[3] = x.w;
        } else if constexpr (G == 2) {
          const float2 x = *reinterpret_cast<const float2*>(pbuf + t * G);
          pg[0] = x.x; pg[1] = x.y;
        } else {
          pg[0] = pbuf[t];
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int c = 0; c < CPL; ++c) o[g][c] = fmaf(pg[g], vf[c], o[g][c]);
      };
      if (nvalid == PS) {
#pragma unroll
        for (int t = 0; t < PS; ++t) pv_row(t);
      } else {
#pragma unroll 1
        for (int t = 0; t < nvalid; ++t) pv_row(t);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[kMaxStages + slot]));

      if (++slot == S) { slot = 0; ++round; }
      if (hdr.y & kLast) break;
      if (!mbar_wait(smem_u32(&bars[slot]), round & 1)) {
        set_status(p.status, KV_ETIMEOUT);
        *abort_flag = 1;
        timed_out = true;
        break;
      }
      st = stages + (size_t)slot * p.stage_bytes;
      hdr = *reinterpret_cast<const int4*>(st + hdr_off);
    }
    if (timed_out) break;

    // ---- finish the task: total l per head, then the output or a partial
    float lt[G];
#pragma unroll
    for (int n = 0; n < NV; ++n) {
      float x = l_part[n];
      x += __shfl_xor_sync(FULL, x, 2);
      x += __shfl_xor_sync(FULL, x, 4);
      x += __shfl_xor_sync(FULL, x, 8);
      x += __shfl_xor_sync(FULL, x, 16);
      if constexpr (G >= 2) {
        const float other = __shfl_xor_sync(FULL, x, 1);
        lt[n] = bit0 ? other : x;
        lt[NV + n] = bit0 ? x : other;
      } else {
        lt[0] = x;
      }
    }
    const int b = hdr.x;
    const bool single = (hdr.y & kSingle) != 0;
    float* dst_o = single ? p.out + ((size_t)b * p.Hq + (size_t)h * G) * D
                          : p.part_o + part_index(hdr.w) * G * D;
    float* dst_l = single ? p.lse + (size_t)b * p.Hq + (size_t)h * G
                          : p.part_lse + part_index(hdr.w) * G;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float inv = 1.0f / lt[g];
      if constexpr (CPL == 4) {
        *reinterpret_cast<float4*>(dst_o + (size_t)g * D + lane * 4) =
            make_float4(o[g][0] * inv, o[g][1] * inv, o[g][2] * inv, o[g][3] * inv);
      } else {
        *reinterpret_cast<float2*>(dst_o + (size_t)g * D + lane * 2) =
            make_float2(o[g][0] * inv, o[g][1] * inv);
      }
      const float l2 = m_run[g] + log2f(lt[g]);
      if (lane == g) dst_l[g] = single ? l2 * 0.6931471805599453f : l2;
    }
    if (single) continue;

    // ---- split merge.  Split s of b (chunk cf + s) sits in slot 2(cf + s),
    // or 2cf + 1 for s = 0.  Up to kDirectMerge splits are merged at once by
    // the last to finish; more are merged in groups of GS = ceil(sqrt(ns))
    // consecutive splits (the last of each group merges it into the group's
    // first slot), then the groups (the last group merger).
    const long long Ob = O[b];
    const int ns = (int)split_count(Ob, O[b + 1] - Ob, chunk);
    const long long cf = Ob / chunk;
    const int s = (hdr.w & 1) ? 0 : (int)(hdr.w / 2 - cf);
    auto slot_of = [&](int i) -> long long { return i == 0 ? 2 * cf + 1 : 2 * (cf + i); };
    int32_t* row_ticket = p.row_done + (size_t)b * p.Hkv + h;
    if (ns <= kDirectMerge) {
      if (ticket(row_ticket, ns)) {
        merge(ns, slot_of, b, -1);
        if (lane == 0) *row_ticket = 0;  // ready for the next call
      }
    } else {
      int GS = (int)ceilf(sqrtf((float)ns));
      while (GS * GS < ns) ++GS;
      while ((GS - 1) * (GS - 1) >= ns) --GS;
      const int ng = (ns + GS - 1) / GS;
      const int first = (s / GS) * GS;
      const int nk = min(ns, first + GS) - first;
      int32_t* group_ticket = p.group_done + part_index(slot_of(first));
      if (ticket(group_ticket, nk)) {
        merge(nk, [&](int i) { return slot_of(first + i); }, b, slot_of(first));
        if (lane == 0) *group_ticket = 0;
        if (ticket(row_ticket, ng)) {
          merge(ng, [&](int i) { return slot_of(i * GS); }, b, -1);
          if (lane == 0) *row_ticket = 0;
        }
      }
    }
  }
}

using DecodeFn = void (*)(const DecodeParams);

DecodeFn pick_decode(int d, int G, int dtype) {
#define KVB_CASE(DD, GG)                                                            \
  if (d == DD && G == GG)                                                           \
    return dtype == KV_BF16 ? decode_kernel<DD, GG, BF16> : decode_kernel<DD, GG, F16>;
  KVB_CASE(64, 1) KVB_CASE(64, 2) KVB_CASE(64, 4) KVB_CASE(64, 8)
  KVB_CASE(128, 1) KVB_CASE(128, 2) KVB_CASE(128, 4) KVB_CASE(128, 8)
#undef KVB_CASE
  return nullptr;
}

struct KernelConfig {
  int stages = 0, blocks_per_sm = 0, num_sms = 0, threads = 0;
  uint32_t kv_bytes = 0, q_bytes = 0, stage_bytes = 0, off_pbuf = 0, off_offsets = 0,
           off_stages = 0;
  size_t smem = 0;
  DecodeFn fn = nullptr;
};

// Launch shape for a decode shape on the current device (cached).
int kernel_config(int Hq, int Hkv, int d, int dtype, KernelConfig* out) {
  static std::mutex mu;
  static std::unordered_map<long long, KernelConfig> cache;
  int dev = 0;
  KV_CUDA_CHECK(cudaGetDevice(&dev));
  const long long key = ((((long long)dev * 64 + Hq) * 32 + Hkv) * 512 + d) * 4 + dtype;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return KV_OK;
  }
  KernelConfig k;
  const int G = Hq / Hkv;
  k.fn = pick_decode(d, G, dtype);
  if (!k.fn) return KV_EINVAL;
  int optin = 0;
  KV_CUDA_CHECK(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
  KV_CUDA_CHECK(cudaDeviceGetAttribute(&k.num_sms, cudaDevAttrMultiProcessorCount, dev));
  k.kv_bytes = (uint32_t)(Hkv * PS * d * 2);
  k.q_bytes = (uint32_t)(Hq * d * 2);
  k.stage_bytes = (uint32_t)align_up(stage_header_offset(k.kv_bytes, k.q_bytes) + kHeaderStageBytes, 128);
  k.off_pbuf = kSmemHeader;
  k.off_offsets = (uint32_t)align_up(k.off_pbuf + (size_t)Hkv * PS * G * 4, 16);
  k.off_stages = (uint32_t)align_up(k.off_offsets + (size_t)(kFusedMaxB + 1) * 4, 1024);
  const size_t fixed = k.off_stages;
  const size_t budget = (size_t)optin - 1024;  // margin below the opt-in limit
  long long S = budget > fixed ? (long long)((budget - fixed) / k.stage_bytes) : 0;
  S = std::min<long long>(S, kMaxStages);
  if (S < 2) return KV_EINVAL;
  k.stages = (int)S;
  k.smem = fixed + (size_t)k.stages * k.stage_bytes;
  k.threads = 32 * (1 + Hkv);
  // The limit belongs to the kernel function, which several shapes share:
  // always the device maximum, so no shape's setting undercuts another's.
  KV_CUDA_CHECK(cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin));
  KV_CUDA_CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k.blocks_per_sm, k.fn, k.threads, k.smem));
  if (k.blocks_per_sm < 1) return cuda_failed(cudaErrorInvalidConfiguration, "decode occupancy is 0");
  cache[key] = k;
  *out = k;
  return KV_OK;
}

bool shape_ok(int page_size, int Hq, int Hkv, int d, int dtype) {
  if (page_size != PS || Hq <= 0 || Hkv <= 0 || Hkv > 8 || Hq % Hkv) return false;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  if (d != 64 && d != 128) return false;
  return dtype == KV_F16 || dtype == KV_BF16;
}

}  // namespace

namespace {
thread_local cudaEvent_t t_ev_before = nullptr, t_ev_after = nullptr;
std::atomic<unsigned long long> g_test_wait_ns{0};
}
unsigned long long test_consumer_wait_ns() { return g_test_wait_ns.load(std::memory_order_relaxed); }
void set_test_consumer_wait_ns(unsigned long long ns) { g_test_wait_ns.store(ns); }
void set_profile_events(cudaEvent_t before, cudaEvent_t after) {
  t_ev_before = before;
  t_ev_after = after;
}
void take_profile_events(cudaEvent_t* before, cudaEvent_t* after) {
  *before = t_ev_before;
  *after = t_ev_after;
  t_ev_before = t_ev_after = nullptr;
}

int decode_num_workers(int Hq, int Hkv, int d, int page_size, int dtype) {
  if (!shape_ok(page_size, Hq, Hkv, d, dtype)) return KV_EINVAL;
  KernelConfig k;
  int rc = kernel_config(Hq, Hkv, d, dtype, &k);
  if (rc) return rc;
  return k.num_sms * k.blocks_per_sm;
}

DecodeLayout decode_layout(int B, int Hq, int Hkv, int d, int max_pages, int page_size,
                           int pages_per_split, long long n_workers) {
  DecodeLayout L{};
  const int G = Hq / Hkv;
  if (pages_per_split > 0)
    L.max_chunks = ceil_div_ll((long long)B * max_pages, pages_per_split);
  else
    L.max_chunks = n_workers;  // the automatic chunk never yields more chunks than workers
  L.max_slots = 2 * L.max_chunks;
  size_t off = kHeaderBytes;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.row_done = take((size_t)B * Hkv * 4);
  L.group_done = take((size_t)L.max_slots * Hkv * 4);
  L.page_off = take(B > kFusedMaxB ? (size_t)(B + 1) * 4 : 0);
  L.part_o = take((size_t)L.max_slots * Hkv * G * d * 4);
  L.part_lse = take((size_t)L.max_slots * Hkv * G * 4);
  L.total = off;
  (void)page_size;
  return L;
}

int decode_launch(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                  const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                  int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                  int pages_per_split, float* out, float* lse, void* ws, size_t ws_bytes,
                  cudaStream_t stream) {
  if (!shape_ok(page_size, Hq, Hkv, d, dtype)) return KV_EINVAL;
  if (B < 0 || num_pages < 0 || max_pages < 0 || pages_per_split < 0) return KV_EINVAL;
  if (B == 0) return KV_OK;
  if (num_pages < 1) return KV_EINVAL;  // page 0 stands in for bad ids: the pool must hold one
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out || !lse || !ws) return KV_EINVAL;
  if (((uintptr_t)q | (uintptr_t)k_pool | (uintptr_t)v_pool) & 15) return KV_EINVAL;
  if (((uintptr_t)out & 15) || ((uintptr_t)ws & 255)) return KV_EINVAL;
  KernelConfig k;
  int rc = kernel_config(Hq, Hkv, d, dtype, &k);
  if (rc) return rc;
  const long long n_workers = (long long)k.num_sms * k.blocks_per_sm;
  const DecodeLayout L = decode_layout(B, Hq, Hkv, d, max_pages, page_size, pages_per_split, n_workers);
  if (ws_bytes < L.total) return KV_EWORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* status = reinterpret_cast<int*>(w);

  cudaEvent_t ev_before = nullptr, ev_after = nullptr;
  take_profile_events(&ev_before, &ev_after);
  if (ev_before) KV_CUDA_CHECK(cudaEventRecord(ev_before, stream));

  DecodeParams dp{};
  dp.page_off = nullptr;
  if (B > kFusedMaxB) {
    OffsetsArgs oa{};
    oa.seq_lens = seq_lens;
    oa.B = B;
    oa.page_size = page_size;
    oa.max_pages = max_pages;
    oa.page_off = reinterpret_cast<int32_t*>(w + L.page_off);
    oa.status = status;
    KV_CUDA_CHECK(launch_page_offsets(oa, stream));
    dp.page_off = oa.page_off;
  }
  dp.q = static_cast<const uint8_t*>(q);
  dp.k_pool = static_cast<const uint8_t*>(k_pool);
  dp.v_pool = static_cast<const uint8_t*>(v_pool);
  dp.table = block_table;
  dp.seq_lens = seq_lens;
  dp.out = out;
  dp.lse = lse;
  dp.part_o = reinterpret_cast<float*>(w + L.part_o);
  dp.part_lse = reinterpret_cast<float*>(w + L.part_lse);
  dp.row_done = reinterpret_cast<int32_t*>(w + L.row_done);
  dp.group_done = reinterpret_cast<int32_t*>(w + L.group_done);
  dp.status = status;
  dp.chunk_req = pages_per_split;
  dp.max_slots = L.max_slots;
  dp.B = B;
  dp.num_pages = num_pages;
  dp.max_pages = max_pages;
  dp.Hq = Hq;
  dp.Hkv = Hkv;
  dp.stages = k.stages;
  dp.min_chunk = kMinChunk;
  dp.scale_log2 = scale * 1.4426950408889634f;
  dp.kv_bytes = k.kv_bytes;
  dp.q_bytes = k.q_bytes;
  dp.stage_bytes = k.stage_bytes;
  dp.off_pbuf = k.off_pbuf;
  dp.off_offsets = k.off_offsets;
  dp.off_stages = k.off_stages;
  dp.test_wait_ns = test_consumer_wait_ns();
  KV_CUDA_CHECK(launch(k.fn, dim3((unsigned)n_workers), dim3((unsigned)k.threads), k.smem, stream,
                       true, dp));
  if (ev_after) KV_CUDA_CHECK(cudaEventRecord(ev_after, stream));
  return KV_OK;
}

}  // namespace kvb

// ---------------------------------------------------------------------------
// Decode for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers: a host
// framework that plans and owns every device allocation itself, or a
// plugin interface whose contract forbids allocating on the hot path (where
// cudaMalloc's implicit synchronisation would stall the whole device).  They
// cannot provide kv_decode's workspace, so this variant keeps its scratch
// (merge tickets, partial results, page offsets) in one file-scope device
// array instead.  Every device that loads the library holds the array until
// the process exits; all calls share it.
// ---------------------------------------------------------------------------
namespace kvb {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};
unsigned long long g_noalloc_ctx[kNoAllocMaxDevices] = {};

// Unique id of the calling thread's current CUDA context (never reused, so
// a context destroyed by cudaDeviceReset and created anew gets a new one);
// 0 when no context is current yet.
int current_context_id(unsigned long long* id) {
  using CtxGetCurrent = CUresult (*)(CUcontext*);
  using CtxGetId = CUresult (*)(CUcontext, unsigned long long*);
  static CtxGetCurrent get_current = nullptr;
  static CtxGetId get_id = nullptr;
  if (!get_current || !get_id) {
    void* f0 = nullptr;
    void* f1 = nullptr;
    cudaDriverEntryPointQueryResult q0, q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000, cudaEnableDefault, &q0) !=
            cudaSuccess ||
        q0 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || !f0 || !f1)
      return cuda_failed(cudaErrorNotSupported, "cuCtxGetCurrent / cuCtxGetId entry points");
    get_current = reinterpret_cast<CtxGetCurrent>(f0);
    get_id = reinterpret_cast<CtxGetId>(f1);
  }
  CUcontext ctx = nullptr;
  *id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS)
    return cuda_failed(cudaErrorUnknown, "cuCtxGetCurrent");
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return cuda_failed(cudaErrorUnknown, "cuCtxGetId");
  return KV_OK;
}

// Device address of the scratch array on the current device (the host-side
// name of the array is not a device address).  Looked up once per device and
// context: a context reset (cudaDeviceReset) makes the next call look it up
// again.  The lookup itself makes the device's primary context current.
int noalloc_scratch(void** out) {
  int dev = 0;
  KV_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kNoAllocMaxDevices) return KV_EINVAL;
  unsigned long long ctx = 0;
  int rc = current_context_id(&ctx);
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!ctx || !g_noalloc_addr[dev] || g_noalloc_ctx[dev] != ctx) {
    void* ptr = nullptr;
    KV_CUDA_CHECK(cudaGetSymbolAddress(&ptr, g_noalloc_scratch));
    rc = current_context_id(&ctx);
    if (rc) return rc;
    g_noalloc_addr[dev] = ptr;
    g_noalloc_ctx[dev] = ctx;
  }
  *out = g_noalloc_addr[dev];
  return KV_OK;
}

int decode_noalloc(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                   const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                   int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                   int pages_per_split, float* out, float* lse, int32_t* status,
                   cudaStream_t stream) {
  if (!shape_ok(page_size, Hq, Hkv, d, dtype)) return KV_EINVAL;
  if (B < 0 || num_pages < 0 || max_pages < 0 || pages_per_split < 0) return KV_EINVAL;
  if (!status) return KV_EINVAL;
  if ((uintptr_t)status & 3) return KV_EINVAL;
  if (B == 0) {
    KV_CUDA_CHECK(cudaMemsetAsync(status, 0, sizeof(int32_t), stream));
    return KV_OK;
  }
  if (num_pages < 1) return KV_EINVAL;
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out || !lse) return KV_EINVAL;
  if (((uintptr_t)q | (uintptr_t)k_pool | (uintptr_t)v_pool | (uintptr_t)out) & 15) return KV_EINVAL;
  KernelConfig k;
  int rc = kernel_config(Hq, Hkv, d, dtype, &k);
  if (rc) return rc;
  const long long n_workers = (long long)k.num_sms * k.blocks_per_sm;
  const DecodeLayout L = decode_layout(B, Hq, Hkv, d, max_pages, page_size, pages_per_split, n_workers);
  if (L.total > kNoAllocScratchBytes) return KV_EWORKSPACE;  // beyond the fixed scratch
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  uint8_t* w = static_cast<uint8_t*>(scratch);
  // The array keeps the previous call's contents: zero the tickets (and
  // offsets) this call relies on, and the caller's status word.
  KV_CUDA_CHECK(cudaMemsetAsync(w, 0, L.part_o, stream));
  KV_CUDA_CHECK(cudaMemsetAsync(status, 0, sizeof(int32_t), stream));

  DecodeParams dp{};
  dp.page_off = nullptr;
  if (B > kFusedMaxB) {
    OffsetsArgs oa{};
    oa.seq_lens = seq_lens;
    oa.B = B;
    oa.page_size = page_size;
    oa.max_pages = max_pages;
    oa.page_off = reinterpret_cast<int32_t*>(w + L.page_off);
    oa.status = status;
    KV_CUDA_CHECK(launch_page_offsets(oa, stream));
    dp.page_off = oa.page_off;
  }
  dp.q = static_cast<const uint8_t*>(q);
  dp.k_pool = static_cast<const uint8_t*>(k_pool);
  dp.v_pool = static_cast<const uint8_t*>(v_pool);
  dp.table = block_table;
  dp.seq_lens = seq_lens;
  dp.out = out;
  dp.lse = lse;
  dp.part_o = reinterpret_cast<float*>(w + L.part_o);
  dp.part_lse = reinterpret_cast<float*>(w + L.part_lse);
  dp.row_done = reinterpret_cast<int32_t*>(w + L.row_done);
  dp.group_done = reinterpret_cast<int32_t*>(w + L.group_done);
  dp.status = status;
  dp.chunk_req = pages_per_split;
  dp.max_slots = L.max_slots;
  dp.B = B;
  dp.num_pages = num_pages;
  dp.max_pages = max_pages;
  dp.Hq = Hq;
  dp.Hkv = Hkv;
  dp.stages = k.stages;
  dp.min_chunk = kMinChunk;
  dp.scale_log2 = scale * 1.4426950408889634f;
  dp.kv_bytes = k.kv_bytes;
  dp.q_bytes = k.q_bytes;
  dp.stage_bytes = k.stage_bytes;
  dp.off_pbuf = k.off_pbuf;
  dp.off_offsets = k.off_offsets;
  dp.off_stages = k.off_stages;
  dp.test_wait_ns = test_consumer_wait_ns();
  KV_CUDA_CHECK(launch(k.fn, dim3((unsigned)n_workers), dim3((unsigned)k.threads), k.smem, stream,
                       true, dp));
  return KV_OK;
}

}  // namespace
}  // namespace kvb

extern "C" int kv_decode_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                 int num_pages, const int32_t* block_table, int max_pages,
                                 const int32_t* seq_lens, int B, int page_size, int Hq, int Hkv,
                                 int d, int dtype, float scale, int pages_per_split, float* out,
                                 float* lse, int32_t* status, void* stream) {
  return kvb::decode_noalloc(q, k_pool, v_pool, num_pages, block_table, max_pages, seq_lens, B,
                             page_size, Hq, Hkv, d, dtype, scale, pages_per_split, out, lse, status,
                             static_cast<cudaStream_t>(stream));
}
