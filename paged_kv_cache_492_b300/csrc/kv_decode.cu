// Split-KV GQA decode over a paged KV cache, and the log-sum-exp split merge.
//
// What is computed (PersistentKV, aissential.tech -- Summary, Method): for each
// sequence and query head, softmax attention of the one new query over the
// sequence's tokens, read through its block table; the K/V tile of each
// (page, KV head) is loaded once and used for all G query heads of that KV
// head; the work is a compact list of non-empty (sequence, KV head, split)
// tasks, and the splits of a sequence are recombined exactly by their
// log-sum-exp.
//
// How (this library's design for sm_103a):
//  * One persistent CTA per SM slot walks the pages of its chunk(s).  A CTA has
//    one producer warp and one consumer warp per KV head.  A "stage" is one
//    logical page of one sequence for all KV heads: the page's K block
//    [Hkv][16][d] and V block are each one contiguous run in the pool, fetched
//    by two cp.async.bulk copies (plus the sequence's q on its first page) that
//    complete on the stage's mbarrier.  Stages form a ring of S slots; the
//    consumers release a slot through a second mbarrier.
//  * Consumer warp h computes its head's tile: q.k for 16 tokens x G query
//    heads with 8 lanes per token row (16-byte shared loads, partial dots
//    reduce-scattered over the 8 lanes), an online softmax in base 2, and
//    p.v with each lane owning d/32 output channels of all G heads.
//  * A sequence with one split writes out/lse directly; otherwise each task
//    writes its normalised partial (o, lse) and the merge kernel combines them.
#include <math.h>

#include <algorithm>
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

struct DecodeParams {
  const uint8_t* q;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const int32_t* table;
  float* out;
  float* lse;
  float* part_o;
  float* part_lse;
  const int32_t* tasks;
  const int32_t* chunk_begin;
  const int32_t* meta;
  int* status;
  int num_pages, max_pages, Hq, Hkv, stages;
  float scale_log2;       // softmax scale * log2(e)
  uint32_t kv_bytes;      // one page, all KV heads: Hkv * 16 * d * 2
  uint32_t q_bytes;       // one sequence's q: Hq * d * 2
  uint32_t stage_bytes;   // K + V + q + header, 128-byte multiple
  uint32_t off_pbuf, off_stages;
};

__host__ __device__ constexpr uint32_t stage_header_offset(uint32_t kv_bytes, uint32_t q_bytes) {
  return 2 * kv_bytes + q_bytes;
}

template <int D, int G, class T>
__global__ void __launch_bounds__(32 * 9, 1) decode_kernel(const DecodeParams p) {
  constexpr int CH = D / 8;                 // q.k channels per lane (8 lanes per row)
  constexpr int CPL = D / 32;               // p.v output channels per lane
  constexpr int NV = G >= 2 ? G / 2 : 1;    // scores a lane holds after the reduction
  static_assert(D == 64 || D == 128, "d");
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "G");

  extern __shared__ __align__(1024) uint8_t smem[];
  const int S = p.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[S], empty[S]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kMaxStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_consumers = p.Hkv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[kMaxStages + s]), n_consumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Everything below reads the workqueue or writes outputs: wait for the
  // grids this launch depends on.
  pdl_wait();
  pdl_launch_dependents();

  const uint32_t hdr_off = stage_header_offset(p.kv_bytes, p.q_bytes);
  uint8_t* stages = smem + p.off_stages;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_evict_first();
    int slot = 0, round = 0;
    bool aborted = false;
    const int nchunks = p.meta[3];
    for (int c = blockIdx.x; c < nchunks && !aborted; c += gridDim.x) {
      const int g0 = p.chunk_begin[c], g1 = p.chunk_begin[c + 1];
      for (int gi = g0; gi < g1 && !aborted; ++gi) {
        const int4* rec = reinterpret_cast<const int4*>(p.tasks + (size_t)gi * p.Hkv * 8);
        const int4 r0 = rec[0], r1 = rec[1];
        const int b = r0.x, nsplit = r0.w, p0 = r1.x, p1 = r1.y, L = r1.w;
        const int32_t* trow = p.table + (size_t)b * p.max_pages;
        for (int jw = p0; jw < p1 && !aborted; jw += 32) {
          const int j = jw + lane;
          int id = 0;
          if (j < p1) {
            id = trow[j];
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
              if (round > 0) ok = mbar_wait(smem_u32(&bars[kMaxStages + slot]), (round - 1) & 1);
              if (!ok) {
                set_status(p.status, KV_ETIMEOUT);
                *abort_flag = 1;
                aborted = true;
              } else {
                const int jj = jw + i;
                const int flags = (jj == p0 ? kFirst : 0) | (jj == p1 - 1 ? kLast : 0) |
                                  (nsplit == 1 ? kSingle : 0);
                const int nvalid = min(PS, L - jj * PS);
                uint8_t* st = stages + (size_t)slot * p.stage_bytes;
                *reinterpret_cast<int4*>(st + hdr_off) = make_int4(gi, b, flags, nvalid);
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
        if (round > 0) ok = mbar_wait(smem_u32(&bars[kMaxStages + slot]), (round - 1) & 1);
        if (ok) {
          uint8_t* st = stages + (size_t)slot * p.stage_bytes;
          *reinterpret_cast<int4*>(st + hdr_off) = make_int4(0, 0, kDone, 0);
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

  float qr[G][CH];
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

  int slot = 0, round = 0;
  for (;;) {
    const uint32_t full_bar = smem_u32(&bars[slot]);
    if (!mbar_wait(full_bar, round & 1)) {
      set_status(p.status, KV_ETIMEOUT);
      *abort_flag = 1;
      break;
    }
    const uint8_t* st = stages + (size_t)slot * p.stage_bytes;
    const int4 hdr = *reinterpret_cast<const int4*>(st + hdr_off);
    const int flags = hdr.z;
    if (flags & kDone) break;
    const int nvalid = hdr.w;

    if (flags & kFirst) {
      // q rows h*G .. h*G+G-1 of this sequence, my 8-lane slice, rotated like K
      const uint8_t* qs = st + 2 * p.kv_bytes + (size_t)h * G * D * 2;
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int half = 0; half < CH / 8; ++half) {
          const int chunk = half ^ rot;
          const uint4 v = *reinterpret_cast<const uint4*>(qs + ((size_t)g * D + c8 * CH + chunk * 8) * 2);
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

    // ---- scores: 4 token rows per step, 8 lanes per row
    const uint8_t* Kt = st + (size_t)h * PS * D * 2;
    float acc[4 * G];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * i + tq;
      float kf[CH];
#pragma unroll
      for (int half = 0; half < CH / 8; ++half) {
        const int chunk = half ^ rot;
        const uint4 v = *reinterpret_cast<const uint4*>(Kt + ((size_t)t * D + c8 * CH + chunk * 8) * 2);
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

    if (flags & kLast) {
      // ---- finish the task: total l per head, normalise, write
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
      const int gi = hdr.x, b = hdr.y;
      float* dst_o;
      float* dst_l;
      if (flags & kSingle) {
        dst_o = p.out + ((size_t)b * p.Hq + (size_t)h * G) * D;
        dst_l = p.lse + (size_t)b * p.Hq + (size_t)h * G;
      } else {
        const size_t task = (size_t)gi * p.Hkv + h;
        dst_o = p.part_o + task * G * D;
        dst_l = p.part_lse + task * G;
      }
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
        if (lane == g) dst_l[g] = (m_run[g] + log2f(lt[g])) * 0.6931471805599453f;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
#pragma unroll
        for (int c = 0; c < CPL; ++c) o[g][c] = 0.f;
      }
#pragma unroll
      for (int n = 0; n < NV; ++n) l_part[n] = 0.f;
    }
    if (++slot == S) { slot = 0; ++round; }
  }
}

// Combine the splits of each (sequence, KV head), all G query heads at once:
//   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) out_s.
// One CTA per (sequence, KV head).  Sequences with one split were written by
// the decode kernel and empty ones by the workqueue builder; both are skipped.
// Threads are (split group, float4 of the G x d outputs): each sums every
// NSG-th split with independent loads, then the groups are added in shared
// memory.  The per-split weights are computed once into shared memory.
constexpr int kMergeThreads = 512;
constexpr int kMergeMaxWeights = 4096;  // G * splits held in shared memory

struct MergeParams {
  const int32_t* seq_lens;
  const int32_t* seq_group_begin;
  const int32_t* seq_nsplit;
  const float* part_o;
  const float* part_lse;
  float* out;
  float* lse;
  int Hq, Hkv, G, d;
};

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
  __shared__ float w_sm[kMergeMaxWeights];
  __shared__ float lse_sm[8];
  __shared__ float4 red[kMergeThreads];
  pdl_wait();
  const int row = blockIdx.x;
  const int b = row / p.Hkv, h = row - b * p.Hkv;
  const int ns = p.seq_nsplit[b];
  if (p.seq_lens[b] <= 0 || ns <= 1) return;
  const int G = p.G, d = p.d;
  const size_t base = p.seq_group_begin[b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto task = [&](int s) { return (base + s) * p.Hkv + h; };
  // per query head of the group: the merged log-sum-exp
  if (warp < G) {
    const int g = warp;
    float mx = -INFINITY;
    for (int s = lane; s < ns; s += 32) mx = fmaxf(mx, __ldcg(p.part_lse + task(s) * G + g));
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
    float sum = 0.f;
    for (int s = lane; s < ns; s += 32) sum += expf(__ldcg(p.part_lse + task(s) * G + g) - mx);
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
    const float l = mx + logf(sum);
    if (lane == 0) {
      lse_sm[g] = l;
      p.lse[(size_t)b * p.Hq + (size_t)h * G + g] = l;
    }
  }
  __syncthreads();
  const bool cached = ns * G <= kMergeMaxWeights;
  if (cached)
    for (int i = threadIdx.x; i < ns * G; i += blockDim.x) {
      const int s = i / G, g = i - s * G;
      w_sm[i] = expf(__ldcg(p.part_lse + task(s) * G + g) - lse_sm[g]);
    }
  __syncthreads();
  const int F4 = G * d / 4;              // float4s per split
  const int NSG = blockDim.x / F4;       // split groups
  const int f = threadIdx.x % F4, sg = threadIdx.x / F4;
  const int g = f / (d / 4);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (sg < NSG) {
#pragma unroll 4
    for (int s = sg; s < ns; s += NSG) {
      const float w = cached ? w_sm[s * G + g]
                             : expf(__ldcg(p.part_lse + task(s) * G + g) - lse_sm[g]);
      const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + task(s) * G * d) + f);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  if (sg == 0) {
    for (int k = 1; k < NSG; ++k) {
      const float4 v = red[k * F4 + f];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    reinterpret_cast<float4*>(p.out + ((size_t)b * p.Hq + (size_t)h * G) * d)[f] = acc;
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
  uint32_t kv_bytes = 0, q_bytes = 0, stage_bytes = 0, off_pbuf = 0, off_stages = 0;
  size_t smem = 0;
  DecodeFn fn = nullptr;
};

// Launch shape for a decode shape on the current device (cached).
int kernel_config(int Hq, int Hkv, int d, int dtype, KernelConfig* out) {
  static std::mutex mu;
  static std::unordered_map<long long, KernelConfig> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KV_ECUDA;
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
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&k.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KV_ECUDA;
  k.kv_bytes = (uint32_t)(Hkv * PS * d * 2);
  k.q_bytes = (uint32_t)(Hq * d * 2);
  k.stage_bytes = (uint32_t)align_up(stage_header_offset(k.kv_bytes, k.q_bytes) + kHeaderStageBytes, 128);
  k.off_pbuf = 1024;
  k.off_stages = (uint32_t)align_up(k.off_pbuf + (size_t)Hkv * PS * G * 4, 1024);
  const size_t fixed = k.off_stages;
  const size_t budget = (size_t)optin - 1024;  // leave room for static/reserved smem
  long long S = budget > fixed ? (long long)((budget - fixed) / k.stage_bytes) : 0;
  S = std::min<long long>(S, kMaxStages);
  if (S < 2) return KV_EINVAL;
  k.stages = (int)S;
  k.smem = fixed + (size_t)k.stages * k.stage_bytes;
  k.threads = 32 * (1 + Hkv);
  if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)k.smem) != cudaSuccess)
    return KV_ECUDA;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&k.blocks_per_sm, k.fn, k.threads, k.smem) !=
          cudaSuccess ||
      k.blocks_per_sm < 1)
    return KV_ECUDA;
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
}
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
    L.max_chunks = ceil_div_ll((long long)B * max_pages, pages_per_split) + 1;
  else
    L.max_chunks = n_workers + 1;
  L.max_tasks = (long long)Hkv * (B + L.max_chunks);
  size_t off = kHeaderBytes;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.tasks = take((size_t)L.max_tasks * 32);
  L.chunk_begin = take((size_t)L.max_chunks * 4);
  L.seq_group_begin = take((size_t)B * 4);
  L.seq_nsplit = take((size_t)B * 4);
  L.seq_page_off = take((size_t)B * 8);
  L.scratch_np = take((size_t)B * 4);
  L.meta = take(64);
  L.part_o = take((size_t)L.max_tasks * G * d * 4);
  L.part_lse = take((size_t)L.max_tasks * G * 4);
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

  WorkqueueArgs wa{};
  wa.seq_lens = seq_lens;
  wa.B = B;
  wa.Hkv = Hkv;
  wa.page_size = page_size;
  wa.max_pages = max_pages;
  wa.chunk_req = pages_per_split;
  wa.n_workers = n_workers;
  wa.min_chunk = kMinChunk;
  wa.tasks = reinterpret_cast<int32_t*>(w + L.tasks);
  wa.max_tasks = L.max_tasks;
  wa.chunk_begin = reinterpret_cast<int32_t*>(w + L.chunk_begin);
  wa.max_chunks = L.max_chunks;
  wa.seq_group_begin = reinterpret_cast<int32_t*>(w + L.seq_group_begin);
  wa.seq_nsplit = reinterpret_cast<int32_t*>(w + L.seq_nsplit);
  wa.seq_page_off = reinterpret_cast<long long*>(w + L.seq_page_off);
  wa.scratch_np = reinterpret_cast<int32_t*>(w + L.scratch_np);
  wa.meta = reinterpret_cast<int32_t*>(w + L.meta);
  wa.status = status;
  wa.out = out;
  wa.lse = lse;
  wa.Hq = Hq;
  wa.d = d;
  if (launch_build_workqueue(wa, stream) != cudaSuccess) return KV_ECUDA;

  DecodeParams dp{};
  dp.q = static_cast<const uint8_t*>(q);
  dp.k_pool = static_cast<const uint8_t*>(k_pool);
  dp.v_pool = static_cast<const uint8_t*>(v_pool);
  dp.table = block_table;
  dp.out = out;
  dp.lse = lse;
  dp.part_o = reinterpret_cast<float*>(w + L.part_o);
  dp.part_lse = reinterpret_cast<float*>(w + L.part_lse);
  dp.tasks = wa.tasks;
  dp.chunk_begin = wa.chunk_begin;
  dp.meta = wa.meta;
  dp.status = status;
  dp.num_pages = num_pages;
  dp.max_pages = max_pages;
  dp.Hq = Hq;
  dp.Hkv = Hkv;
  dp.stages = k.stages;
  dp.scale_log2 = scale * 1.4426950408889634f;
  dp.kv_bytes = k.kv_bytes;
  dp.q_bytes = k.q_bytes;
  dp.stage_bytes = k.stage_bytes;
  dp.off_pbuf = k.off_pbuf;
  dp.off_stages = k.off_stages;

  cudaEvent_t ev_before = nullptr, ev_after = nullptr;
  take_profile_events(&ev_before, &ev_after);
  if (ev_before && cudaEventRecord(ev_before, stream) != cudaSuccess) return KV_ECUDA;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)n_workers);
  cfg.blockDim = dim3((unsigned)k.threads);
  cfg.dynamicSmemBytes = k.smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k.fn, dp) != cudaSuccess) return KV_ECUDA;
  if (ev_after && cudaEventRecord(ev_after, stream) != cudaSuccess) return KV_ECUDA;

  MergeParams mp{};
  mp.seq_lens = seq_lens;
  mp.seq_group_begin = wa.seq_group_begin;
  mp.seq_nsplit = wa.seq_nsplit;
  mp.part_o = dp.part_o;
  mp.part_lse = dp.part_lse;
  mp.out = out;
  mp.lse = lse;
  mp.Hq = Hq;
  mp.Hkv = Hkv;
  mp.G = Hq / Hkv;
  mp.d = d;
  cudaLaunchConfig_t mcfg{};
  mcfg.gridDim = dim3((unsigned)((long long)B * Hkv));
  mcfg.blockDim = dim3(kMergeThreads);
  mcfg.stream = stream;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&mcfg, merge_kernel, mp) != cudaSuccess) return KV_ECUDA;
  return KV_OK;
}

}  // namespace kvb
