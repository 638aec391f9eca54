// Attention of up to 64 query rows per KV head over the paged cache on the
// tensor cores: T query tokens x G grouped heads (T * G <= 64), so one page
// tile read from HBM serves every row.  Used for several query tokens per
// sequence (the step before decode: a prefill chunk or drafted tokens being
// verified; the T queries are the sequence's last T tokens, causal) and for
// wide GQA groups.  What is computed is the same softmax attention as the
// decode step (PersistentKV, aissential.tech -- Summary, Method: block-table
// GQA attention, K/V tiles reused across the query heads of a group, a
// compact queue of non-empty (sequence, KV head, split) tasks).
//
// Design (sm_103a):
//  * The batch's non-empty pages, laid end to end, are cut into equal chunks
//    (the split rule of the decode workqueue, kv_common.cuh); one CTA per
//    chunk (and block of up to 8 KV heads) derives its own (sequence, split)
//    tasks from a scan of the lengths and streams exactly its chunk's pages,
//    so every CTA moves the same number of bytes whatever the length mix.
//  * A producer warp reads the block table 32 entries at a time and issues
//    TMA tensor copies (cp.async.bulk.tensor, a 5-D view of the pool:
//    64 channels, channel half, slot, head, page) with the 128-byte swizzle
//    into a ring of stages (full/empty mbarriers).  One stage is one page of
//    every head of the block.
//  * One consumer warp per KV head and block of 16 query rows (at most 8
//    per CTA; a ring deep enough for ~192 KB in flight whatever the head
//    block): S = Q K^T and O += P V are mma.sync m16n8k16 (fp32
//    accumulation) with the warp's 16 query rows as M, K/V fragments
//    from ldmatrix on the swizzled tiles (conflict-free), P taken from the
//    score fragments straight into the A fragments of P V.  bf16
//    probabilities are split into a high and a low bf16 part (two MMAs) so
//    their rounding stays far below the output tolerance.
//  * The online softmax runs on the fragments (base 2, scale folded in).  A
//    split of a sequence writes its normalised partial (o, natural-log lse)
//    to a slot named by its chunk (2c + 1 for a sequence's first split, 2c
//    for a continuation: a chunk holds at most one of each), and a merge
//    kernel combines the splits.
#include <cuda.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <array>
#include <mutex>

#include "kv_internal.h"

namespace kvb {
namespace {

// head dimension d: 64 or 128 (one or two 64-channel halves of 128 bytes)
constexpr int kMmaRows = 16;            // query rows of one m16 tile (one consumer warp)
constexpr int kMaxRowBlocks = 4;        // up to 64 query rows per KV head
constexpr int kMaxStages = 12;          // pages in flight per CTA (3 at 8 heads .. 12)
constexpr int kRingBytes = 192 * 1024;  // shared memory for the ring
constexpr int kMaxHeadBlock = 8;        // KV heads (consumer warps) per CTA
constexpr int kHalfTile = 16 * 64 * 2;  // 16 tokens x 64 channels, bytes
constexpr int kBarBytes = 256;          // full[kMaxStages], empty[kMaxStages], dead, abort
constexpr int kDeadBar = 2 * kMaxStages;  // mbarrier nothing completes (test mode)
constexpr int kAbortWord = 2 * kMaxStages + 1;  // 8-byte slot of the abort flag
static_assert((kAbortWord + 1) * 8 <= kBarBytes, "barrier area");
constexpr unsigned FULLM = 0xffffffffu;

struct MmaParams {
  const uint16_t* q;          // [B][Tstride][Hq][128], this call's first token at row 0
  const int32_t* table;
  const int32_t* seq_lens;
  const int32_t* page_off_in; // [B + 1] page offsets (large batches), else null
  int32_t* page_off_out;      // [B + 1] written by CTA 0 for the merge (small batches)
  int32_t* chunk_out;         // [1] the chunk size, written by CTA 0
  float* out;                 // [B][Tstride][Hq][128], as q
  float* lse;                 // [B][Tstride][Hq]
  float* part_o;              // [slot][Hkv][16][128]
  float* part_lse;            // [slot][Hkv][16]
  int* status;
  int B, num_pages, max_pages, Hq, Hkv, G, Tq, rows, rows_pad, rb, hb, nhb, chunk_req, stages;
  int Tstride;                // query tokens per sequence in q/out/lse (>= Tq)
  int len_shift;              // this call's tokens see max(0, L - len_shift) cached tokens
  long long n_chunks;         // chunks of the automatic split (CTAs per head block)
  float scale_log2;
  unsigned long long test_wait_ns;  // > 0: failure-path test mode (see test_consumer_wait_ns)
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <class T>
__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<F16>(float* d, const uint32_t* a, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<BF16>(float* d, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 values as one register of the element type (x in the low half).
template <class T>
__device__ __forceinline__ uint32_t pack2(float x, float y);
template <>
__device__ __forceinline__ uint32_t pack2<F16>(float x, float y) {
  __half2 h = __floats2half2_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<BF16>(float x, float y) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<uint32_t*>(&h);
}

// TMA tensor copy of a 5-D box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const void* tmap, int c0, int c1, int c2,
                                            int c3, int c4, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar), "l"(policy)
      : "memory");
}

// The cached tokens a call's queries see: max(0, L - shift); a negative
// length stays negative, so it is still reported.
__device__ __forceinline__ int shifted_len(int L, int shift) {
  return L < 0 ? L : max(0, L - shift);
}

// Stage layout: K then V; each is [channel half][head of the block][token]
// rows of 128 bytes (64 channels), i.e. a (half, head) sub-tile of 2 KiB; a
// head has d / 64 halves.  The 128-byte swizzle stores logical 16-byte chunk
// c of a row at chunk c ^ (token % 8), so the eight rows one ldmatrix reads
// fall in eight different bank groups.  Offset of logical chunk `chunk`
// (0 .. d/8 - 1 over the d channels) of token `t` within one head's tile:
__device__ __forceinline__ uint32_t tile_off(int t, int chunk, uint32_t half_stride) {
  return (uint32_t)(chunk >> 3) * half_stride + (uint32_t)(t * 128 + (((chunk & 7) ^ (t & 7)) << 4));
}

template <class T, int D>
__global__ void __launch_bounds__(32 * (1 + kMaxHeadBlock), 1)
    mma_attend_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const MmaParams p) {
  constexpr int kHalves = D / 64;  // 64-channel halves of a head's row (one 128-byte atom each)
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[S], empty[S]
  const uint32_t raw = smem_u32(smem);
  uint8_t* stages = smem + (((raw + kBarBytes + 1023) & ~1023u) - raw);  // 1024-aligned
  const uint32_t half_stride = (uint32_t)p.hb * kHalfTile;
  const uint32_t stage_bytes = 2 * kHalves * half_stride;  // K and V, kHalves halves each
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x / p.nhb, hblk = blockIdx.x - (blockIdx.x / p.nhb) * p.nhb;

  __shared__ int32_t s_off[kFusedMaxB + 1];
  __shared__ long long s_scan[32];
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&bars[kAbortWord]);
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[kMaxStages + s]), p.hb * p.rb);
    }
    mbar_init(smem_u32(&bars[kDeadBar]), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  pdl_wait();  // lengths and page offsets may come from the previous kernel
  pdl_launch_dependents();
  // Every producer reads block-table entries right after the offsets: have
  // the table on its way to L2 meanwhile (spread over all CTAs).
  {
    const size_t lines = ((size_t)p.B * p.max_pages * 4 + 127) / 128;
    const char* tb = reinterpret_cast<const char*>(p.table);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < lines && i < (1u << 20);
         i += (size_t)gridDim.x * blockDim.x)
      prefetch_l2(tb + i * 128);
  }
  // page offsets O[b] of the batch (sum of ceil(L/16) before b)
  const int32_t* O = p.page_off_in;
  if (!O) {
    const int nth = blockDim.x, per = ceil_div(p.B, nth);
    const int b0 = min(p.B, (int)threadIdx.x * per), b1 = min(p.B, b0 + per);
    long long mine = 0;
    bool bad = false;
    for (int b = b0; b < b1; ++b) {
      const int L = shifted_len(__ldg(p.seq_lens + b), p.len_shift);
      const long long np = L > 0 ? ceil_div_ll(L, 16) : 0;
      if (L < 0 || np > p.max_pages) bad = true; else mine += np;
    }
    if (bad && blockIdx.x == 0) set_status(p.status, KV_EINVAL);
    long long off;
    const long long W = block_exclusive_scan(mine, &off, s_scan);  // <= B * max_pages < 2^31
    for (int b = b0; b < b1; ++b) {
      s_off[b] = (int32_t)off;
      const int L = shifted_len(__ldg(p.seq_lens + b), p.len_shift);
      const long long np = L > 0 ? ceil_div_ll(L, 16) : 0;
      if (L >= 0 && np <= p.max_pages) off += np;
    }
    if (threadIdx.x == 0) s_off[p.B] = (int32_t)W;
    O = s_off;
  }
  __syncthreads();
  const long long W = O[p.B];
  const long long chunk = p.chunk_req > 0 ? p.chunk_req : auto_chunk(W, p.n_chunks, kMinChunk);
  const long long nchunks = W > 0 ? ceil_div_ll(W, chunk) : 0;
  if (blockIdx.x == 0) {
    if (p.page_off_out)
      for (int b = threadIdx.x; b <= p.B; b += blockDim.x) p.page_off_out[b] = O[b];
    if (threadIdx.x == 0) *p.chunk_out = (int32_t)chunk;
  }
  if (c >= nchunks) return;
  const long long c0 = (long long)c * chunk, c1 = min(W, c0 + chunk);
  const int b_first = seq_at(O, p.B, c0);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_evict_first();
    const int h0 = hblk * p.hb;
    int slot = 0, round = 0;
    bool aborted = false;
    for (int b = b_first; b < p.B && O[b] < c1 && !aborted; ++b) {
      const long long Ob = O[b], np = O[b + 1] - Ob;
      if (np == 0) continue;
      long long lo, hi;
      split_range(Ob, np, chunk, c, &lo, &hi);
      const int p0 = (int)lo, p1 = (int)hi;
      const int32_t* trow = p.table + (size_t)b * p.max_pages;
      for (int jw = p0; jw < p1 && !aborted; jw += 32) {
        int id = 0;
        if (jw + lane < p1) {
          id = __ldg(trow + jw + lane);
          if (id < 0 || id >= p.num_pages) {
            set_status(p.status, KV_EBADPAGE);
            id = 0;
          }
        }
        const int n = min(32, p1 - jw);
        for (int i = 0; i < n; ++i) {
          const int pid = __shfl_sync(FULLM, id, i);
          if (lane == 0) {
            bool ok = true;
            if (round > 0)
              ok = mbar_wait(smem_u32(&bars[kMaxStages + slot]), (round - 1) & 1, kWaitLimitNs,
                             abort_flag);
            if (!ok) {
              set_status(p.status, KV_ETIMEOUT);  // no-op when a consumer already set it
              aborted = true;
            } else {
              const uint32_t bar = smem_u32(&bars[slot]);
              const uint32_t st = smem_u32(stages) + (uint32_t)slot * stage_bytes;
              mbar_arrive_expect_tx(bar, stage_bytes);
#pragma unroll
              for (int half = 0; half < kHalves; ++half) {
                tma_load_5d(st + half * half_stride, &tmk, 0, half, 0, h0, pid, bar, pol);
                tma_load_5d(st + (kHalves + half) * half_stride, &tmv, 0, half, 0, h0, pid, bar,
                            pol);
              }
            }
          }
          aborted = __shfl_sync(FULLM, aborted, 0);
          if (aborted) break;
          if (++slot == p.stages) {
            slot = 0;
            ++round;
          }
        }
      }
    }
    if (aborted && lane == 0) {
      // let the copies already issued land before the CTA's shared memory
      // goes away: the last phase issued on each slot (bounded waits)
      for (int s = 0; s < p.stages; ++s) {
        const int issued = s < slot ? round + 1 : round;
        if (issued > 0) mbar_wait(smem_u32(&bars[s]), (issued - 1) & 1);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // consumer warp c: head hw of the block, rows [16 rbi, 16 rbi + 16)
  const int cw = warp - 1, hw = cw / p.rb, rbi = cw - (cw / p.rb) * p.rb;
  const int h = hblk * p.hb + hw;
  const int qr0 = rbi * kMmaRows + (lane >> 2), qr1 = qr0 + 8, qc = (lane & 3) * 2;
  const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: matrix mi, row mr
  // test mode: a bounded wait on a barrier nothing completes runs out here,
  // and the warp takes the same way out as any wait that runs out
  if (p.test_wait_ns && !__all_sync(FULLM, mbar_wait(smem_u32(&bars[kDeadBar]), 0, p.test_wait_ns))) {
    if (lane == 0) set_status(p.status, KV_ETIMEOUT);
    *abort_flag = 1;
    return;
  }
  int slot = 0, round = 0;
  for (int b = b_first; b < p.B && O[b] < c1; ++b) {
    const long long Ob = O[b], np = O[b + 1] - Ob;
    if (np == 0) continue;
    long long lo, hi;
    split_range(Ob, np, chunk, c, &lo, &hi);
    const int p0 = (int)lo, p1 = (int)hi;
    const bool single = split_count(Ob, np, chunk) == 1;
    const long long slot_id = 2ll * c + (c == Ob / chunk ? 1 : 0);
    const int L = shifted_len(__ldg(p.seq_lens + b), p.len_shift);

    // Q fragments; row r = i * G + g is query token i, head h * G + g
    auto qrow = [&](int r) -> const uint16_t* {
      if (r >= p.rows) return nullptr;
      const int i = r / p.G, g = r - (r / p.G) * p.G;
      return p.q + (((size_t)b * p.Tstride + i) * p.Hq + (size_t)h * p.G + g) * D;
    };
    const uint16_t* q0 = qrow(qr0);
    const uint16_t* q1 = qrow(qr1);
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int cc = kk * 16 + qc;
      qa[kk][0] = q0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + cc)) : 0u;
      qa[kk][1] = q1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + cc)) : 0u;
      qa[kk][2] = q0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + cc + 8)) : 0u;
      qa[kk][3] = q1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + cc + 8)) : 0u;
    }
    // causal limit of each row: tokens [0, L - Tq + 1 + i)
    const int lim0 = qr0 < p.rows ? L - p.Tq + 1 + qr0 / p.G : 0;
    const int lim1 = qr1 < p.rows ? L - p.Tq + 1 + qr1 / p.G : 0;

    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int j = p0; j < p1; ++j) {
      if (!__all_sync(FULLM, mbar_wait(smem_u32(&bars[slot]), round & 1))) {
        if (lane == 0) set_status(p.status, KV_ETIMEOUT);
        *abort_flag = 1;
        return;
      }
      const uint32_t kt = smem_u32(stages) + (uint32_t)slot * stage_bytes + hw * kHalfTile;
      const uint32_t vt = kt + kHalves * half_stride;
      // ---- S = Q K^T: two n-tiles of 8 tokens, eight k-steps of 16 channels
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        // matrices: (tokens 0-7, ch lo), (0-7, ch hi), (8-15, lo), (8-15, hi)
        const int t = (mi >> 1) * 8 + mr, chunk = kk * 2 + (mi & 1);
        uint32_t b00, b01, b10, b11;
        ldsm_x4(kt + tile_off(t, chunk, half_stride), b00, b01, b10, b11);
        mma16816<T>(s[0], qa[kk], b00, b01);
        mma16816<T>(s[1], qa[kk], b10, b11);
      }
      // ---- masks (partial last page, causal limit), scale to base 2
      const int base = j * 16;
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pos = base + nt * 8 + qc + e;
          s[nt][e] = pos < lim0 ? s[nt][e] * p.scale_log2 : -INFINITY;
          s[nt][2 + e] = pos < lim1 ? s[nt][2 + e] * p.scale_log2 : -INFINITY;
          mx0 = fmaxf(mx0, s[nt][e]);
          mx1 = fmaxf(mx1, s[nt][2 + e]);
        }
#pragma unroll
      for (int off = 1; off <= 2; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(FULLM, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(FULLM, mx1, off));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      // a row with nothing valid yet keeps factor 1 and adds nothing
      const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = ex2(m0 - ms0), al1 = ex2(m1 - ms1);
      m0 = mn0;
      m1 = mn1;
      float pr[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        pr[nt][0] = ex2(s[nt][0] - ms0);
        pr[nt][1] = ex2(s[nt][1] - ms0);
        pr[nt][2] = ex2(s[nt][2] - ms1);
        pr[nt][3] = ex2(s[nt][3] - ms1);
      }
      l0 = l0 * al0 + pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
      l1 = l1 * al1 + pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
      }
      // ---- O += P V: P as A fragments (k = 16 tokens), V by transposed ldmatrix
      uint32_t pa[4], pl[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        pa[k] = pack2<T>(pr[k >> 1][(k & 1) * 2], pr[k >> 1][(k & 1) * 2 + 1]);
      if constexpr (T::code == KV_BF16) {
        // low part: what the bf16 rounding of P dropped (exact in fp32)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 hi = T::to_f2(pa[k]);
          pl[k] = pack2<T>(pr[k >> 1][(k & 1) * 2] - hi.x, pr[k >> 1][(k & 1) * 2 + 1] - hi.y);
        }
      }
#pragma unroll
      for (int n2 = 0; n2 < D / 16; ++n2) {
        // matrices: (tokens 0-7, ch tile 2n2), (8-15, 2n2), (0-7, 2n2+1), (8-15, 2n2+1)
        const int t = (mi & 1) * 8 + mr, chunk = n2 * 2 + (mi >> 1);
        uint32_t v00, v01, v10, v11;
        ldsm_x4_t(vt + tile_off(t, chunk, half_stride), v00, v01, v10, v11);
        mma16816<T>(o[2 * n2], pa, v00, v01);
        mma16816<T>(o[2 * n2 + 1], pa, v10, v11);
        if constexpr (T::code == KV_BF16) {
          mma16816<T>(o[2 * n2], pl, v00, v01);
          mma16816<T>(o[2 * n2 + 1], pl, v10, v11);
        }
      }
      // this warp is done with the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars[kMaxStages + slot]));
      if (++slot == p.stages) {
        slot = 0;
        ++round;
      }
    }

    // ---- finish the split: row sums, normalise, write the output or partial
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      l0 += __shfl_xor_sync(FULLM, l0, off);
      l1 += __shfl_xor_sync(FULLM, l1, off);
    }
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const float ls0 = l0 > 0.f ? (m0 + log2f(l0)) * 0.6931471805599453f : -INFINITY;
    const float ls1 = l1 > 0.f ? (m1 + log2f(l1)) * 0.6931471805599453f : -INFINITY;
    auto dst_row = [&](int r, float** o_ptr, float** l_ptr) {
      if (single) {
        const int i = r / p.G, g = r - (r / p.G) * p.G;
        const size_t row = ((size_t)b * p.Tstride + i) * p.Hq + (size_t)h * p.G + g;
        *o_ptr = p.out + row * D;
        *l_ptr = p.lse + row;
      } else {
        const size_t part = (size_t)slot_id * p.Hkv + h;
        *o_ptr = p.part_o + (part * p.rows_pad + r) * D;
        *l_ptr = p.part_lse + part * p.rows_pad + r;
      }
    };
    if (qr0 < p.rows) {
      float *po, *pl;
      dst_row(qr0, &po, &pl);
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<float2*>(po + n * 8 + qc) = make_float2(o[n][0] * inv0, o[n][1] * inv0);
      if ((lane & 3) == 0) *pl = ls0;
    }
    if (qr1 < p.rows) {
      float *po, *pl;
      dst_row(qr1, &po, &pl);
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<float2*>(po + n * 8 + qc) = make_float2(o[n][2] * inv1, o[n][3] * inv1);
      if ((lane & 3) == 0) *pl = ls1;
    }
  }
}

using AttendFn = void (*)(const CUtensorMap, const CUtensorMap, const MmaParams);

// Combine the splits of each (sequence, KV head): per row
// lse = ln sum_s e^{lse_s}, out = sum_s e^{lse_s - lse} out_s (parts with
// lse_s = -inf add nothing; all of them -inf gives out = 0, lse = -inf).
// Split s of a sequence whose pages start in chunk c_0 is in slot 2 c_0 + 1
// (s = 0) or 2 (c_0 + s).  One CTA per (sequence, KV head, row); its warps
// take an equal share of the splits each and merge them online, 32 at a time
// (lane i holds split i's lse; the 16-partial batches are loaded before they
// are needed, so a batch costs one memory round trip), then combine through
// shared memory.  16 warps when the grid fits the SMs once (few sequences,
// each split over many chunks: one batch per warp), else 4 (many small CTAs
// that schedule quickly and can wait beside the attention kernel's CTAs).  Single-split sequences were written by the
// attention kernel; sequences without pages get out = 0, lse = -inf here.
struct MmaMergeParams {
  const int32_t* page_off;  // [B + 1]
  const int32_t* chunk;     // [1]
  const float* part_o;
  const float* part_lse;
  float* out;
  float* lse;
  int B, Hq, Hkv, G, Tstride, rows, rows_pad;
};

// CPL consecutive fp32 channels of one lane (4 at d = 128, 2 at d = 64).
template <int CPL>
struct Chans {
  float v[CPL];
};
template <int CPL>
__device__ __forceinline__ Chans<CPL> ldcg_chans(const float* p) {
  Chans<CPL> r;
  if constexpr (CPL == 4) {
    const float4 x = __ldcg(reinterpret_cast<const float4*>(p));
    r.v[0] = x.x, r.v[1] = x.y, r.v[2] = x.z, r.v[3] = x.w;
  } else {
    const float2 x = __ldcg(reinterpret_cast<const float2*>(p));
    r.v[0] = x.x, r.v[1] = x.y;
  }
  return r;
}
template <int CPL>
__device__ __forceinline__ void st_chans(float* p, const Chans<CPL>& c) {
  if constexpr (CPL == 4)
    *reinterpret_cast<float4*>(p) = make_float4(c.v[0], c.v[1], c.v[2], c.v[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(c.v[0], c.v[1]);
}

template <int kMergeWarps, int D>
__global__ void __launch_bounds__(kMergeWarps * 32, 1) mma_merge_kernel(const MmaMergeParams p) {
  constexpr int CPL = D / 32;  // channels per lane
  __shared__ float sm_m[kMergeWarps], sm_l[kMergeWarps];
  __shared__ Chans<CPL> sm_acc[kMergeWarps][32];
  pdl_wait();
  const int b = blockIdx.x / p.Hkv, h = blockIdx.x - (blockIdx.x / p.Hkv) * p.Hkv;
  const int r = blockIdx.y;
  const long long Ob = p.page_off[b], np = p.page_off[b + 1] - Ob, chunk = *p.chunk;
  const long long ns = split_count(Ob, np, chunk);
  if (ns == 1 || r >= p.rows) return;
  const int i = r / p.G, g = r - (r / p.G) * p.G;
  const size_t row = ((size_t)b * p.Tstride + i) * p.Hq + (size_t)h * p.G + g;
  if (ns == 0) {
    if (threadIdx.x < D) p.out[row * D + threadIdx.x] = 0.f;
    if (threadIdx.x == 0) p.lse[row] = -INFINITY;
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, c0 = lane * CPL;
  const long long cf = Ob / chunk;
  auto part = [&](long long s) {
    return ((size_t)(s == 0 ? 2 * cf + 1 : 2 * (cf + s)) * p.Hkv + h) * p.rows_pad + r;
  };
  auto load_o = [&](long long s) { return ldcg_chans<CPL>(p.part_o + part(s) * D + c0); };
  const long long q = (ns + kMergeWarps - 1) / kMergeWarps;
  const long long sa = min(ns, warp * q), sb = min(ns, sa + q);
  float m = -INFINITY, l = 0.f;
  Chans<CPL> acc;
#pragma unroll
  for (int e = 0; e < CPL; ++e) acc.v[e] = 0.f;
  Chans<CPL> zero;
#pragma unroll
  for (int e = 0; e < CPL; ++e) zero.v[e] = 0.f;
  for (long long s0 = sa; s0 < sb; s0 += 32) {
    const int n = (int)min(32ll, sb - s0);
    const float ls = lane < n ? __ldcg(p.part_lse + part(s0 + lane)) : -INFINITY;
    Chans<CPL> v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = k < n ? load_o(s0 + k) : zero;
    float mb = ls;
#pragma unroll
    for (int off = 16; off; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(FULLM, mb, off));
    if (mb == -INFINITY) continue;  // nothing in this batch
    const float mn = fmaxf(m, mb);
    const float keep = m == -INFINITY ? 0.f : expf(m - mn);
    m = mn;
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc.v[e] *= keep;
    const float w_mine = ls == -INFINITY ? 0.f : expf(ls - m);
    float wsum = w_mine;
#pragma unroll
    for (int off = 16; off; off >>= 1) wsum += __shfl_xor_sync(FULLM, wsum, off);
    l = l * keep + wsum;
    auto add = [&](const Chans<CPL>& x, float w) {
#pragma unroll
      for (int e = 0; e < CPL; ++e) acc.v[e] = fmaf(w, x.v[e], acc.v[e]);
    };
#pragma unroll
    for (int k = 0; k < 16; ++k) add(v[k], __shfl_sync(FULLM, w_mine, k));
    if (n > 16) {
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = 16 + k < n ? load_o(s0 + 16 + k) : zero;
#pragma unroll
      for (int k = 0; k < 16; ++k) add(v[k], __shfl_sync(FULLM, w_mine, 16 + k));
    }
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
  sm_acc[warp][lane] = acc;
  __syncthreads();
  if (warp != 0) return;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, sm_m[w]);
  Chans<CPL> o = zero;
  float Lr = -INFINITY;
  if (M > -INFINITY) {
    float L = 0.f;
    float sc[kMergeWarps];
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      sc[w] = sm_m[w] == -INFINITY ? 0.f : expf(sm_m[w] - M);
      L += sm_l[w] * sc[w];
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      const Chans<CPL> a = sm_acc[w][lane];
      const float f = sc[w] * inv;
#pragma unroll
      for (int e = 0; e < CPL; ++e) o.v[e] = fmaf(f, a.v[e], o.v[e]);
    }
    Lr = M + logf(L);
  }
  st_chans<CPL>(p.out + row * D + c0, o);
  if (lane == 0) p.lse[row] = Lr;
}

// ---- tensor maps -------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int encode_fn(EncodeTiledFn* out) {
  static std::mutex mu;
  static EncodeTiledFn fn = nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
      return cuda_failed(cudaErrorNotSupported, "cuTensorMapEncodeTiled entry point");
    fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  *out = fn;
  return KV_OK;
}

// Pool [P][Hkv][16][d] seen as 5-D (64 channels, channel half, slot, head,
// page; d / 64 halves); one box is one channel half of `hb` heads of one
// page: hb x 16 rows of 128 bytes, 128-byte swizzled.  A map depends only on
// these arguments, so the last few are kept and reused (encoding is host
// work on every call otherwise).
int encode_pool_map_uncached(CUtensorMap* m, const void* pool, int num_pages, int Hkv, int hb,
                             int dtype, int d);
int encode_pool_map(CUtensorMap* m, const void* pool, int num_pages, int Hkv, int hb, int dtype,
                    int d) {
  struct Entry {
    const void* pool;
    int num_pages, Hkv, hb, dtype, d;
    CUtensorMap map;
  };
  constexpr int kEntries = 8;
  static std::mutex mu;
  static Entry cache[kEntries];
  static int used = 0, next = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i) {
      const Entry& e = cache[i];
      if (e.pool == pool && e.num_pages == num_pages && e.Hkv == Hkv && e.hb == hb &&
          e.dtype == dtype && e.d == d) {
        *m = e.map;
        return KV_OK;
      }
    }
  }
  const int rc = encode_pool_map_uncached(m, pool, num_pages, Hkv, hb, dtype, d);
  if (rc) return rc;
  std::lock_guard<std::mutex> lk(mu);
  Entry& e = cache[next];
  e = Entry{pool, num_pages, Hkv, hb, dtype, d, *m};
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  return KV_OK;
}

int encode_pool_map_uncached(CUtensorMap* m, const void* pool, int num_pages, int Hkv, int hb,
                             int dtype, int d) {
  EncodeTiledFn fn;
  int rc = encode_fn(&fn);
  if (rc) return rc;
  const cuuint64_t row = (cuuint64_t)d * 2;  // bytes of one token's head row
  const cuuint64_t dims[5] = {64, (cuuint64_t)d / 64, 16, (cuuint64_t)Hkv, (cuuint64_t)num_pages};
  const cuuint64_t strides[4] = {128, row, 16 * row, (cuuint64_t)Hkv * 16 * row};
  const cuuint32_t box[5] = {64, 1, 16, (cuuint32_t)hb, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(m, dtype == KV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        5, const_cast<void*>(pool), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[64];
    snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled returned %d", (int)r);
    return cuda_failed(cudaErrorInvalidValue, msg);
  }
  return KV_OK;
}

// Row blocks of 16 query rows per KV head.
int row_blocks(int rows) { return (rows + kMmaRows - 1) / kMmaRows; }
// Heads per CTA: the largest divisor of Hkv with at most 8 consumer warps
// (one per head and row block).
int head_block(int Hkv, int rb) {
  for (int hb = kMaxHeadBlock / rb; hb > 1; --hb)
    if (Hkv % hb == 0) return hb;
  return 1;
}
// Ring depth: about kRingBytes in flight whatever the head block (a stage is
// one page of hb heads, K and V, d / 64 halves each).
int ring_stages(int hb, int d) {
  const int s = kRingBytes / (2 * (d / 64) * hb * kHalfTile);
  return s < 3 ? 3 : (s > kMaxStages ? kMaxStages : s);
}
size_t mma_smem(int hb, int d) {
  return kBarBytes + 1024 + (size_t)ring_stages(hb, d) * 2 * (d / 64) * hb * kHalfTile;
}

struct MmaLayout {
  size_t page_off, chunk, part_o, part_lse, total;
  long long max_chunks;
};

MmaLayout mma_layout(int B, int Hkv, int rows, int d, int max_pages, int pages_per_split,
                     long long n_chunks, size_t region) {
  const size_t rows_pad = (size_t)row_blocks(rows) * kMmaRows;
  MmaLayout L{};
  L.max_chunks = pages_per_split > 0 ? ceil_div_ll((long long)B * max_pages, pages_per_split)
                                     : n_chunks;
  if (L.max_chunks < 1) L.max_chunks = 1;
  const long long slots = 2 * L.max_chunks;
  size_t off = align_up(region < kHeaderBytes ? kHeaderBytes : region, 256);
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.page_off = take((size_t)(B + 1) * 4);
  L.chunk = take(4);
  L.part_o = take((size_t)slots * Hkv * rows_pad * d * 4);
  L.part_lse = take((size_t)slots * Hkv * rows_pad * 4);
  L.total = off;
  return L;
}

// Chunks of the automatic split: one per CTA that fits on the device at once.
int mma_chunks(int Hkv, int rows, int d, long long* out) {
  static std::mutex mu;
  static int cached[64][2][kMaxHeadBlock + 1][kMaxRowBlocks + 1] = {};
  int dev = 0;
  KV_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return KV_EINVAL;
  const int rb = row_blocks(rows);
  if (rb < 1 || rb > kMaxRowBlocks) return KV_EINVAL;
  const int hb = head_block(Hkv, rb), di = d == 64 ? 0 : 1;
  std::lock_guard<std::mutex> lk(mu);
  if (!cached[dev][di][hb][rb]) {
    int sms = 0, per = 0;
    KV_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const auto fns = d == 64 ? std::array<AttendFn, 2>{mma_attend_kernel<F16, 64>,
                                                       mma_attend_kernel<BF16, 64>}
                             : std::array<AttendFn, 2>{mma_attend_kernel<F16, 128>,
                                                       mma_attend_kernel<BF16, 128>};
    for (auto fn : fns) {
      KV_CUDA_CHECK(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)mma_smem(kMaxHeadBlock, d)));
      int n = 0;
      KV_CUDA_CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, 32 * (1 + hb * rb),
                                                                  mma_smem(hb, d)));
      per = per == 0 ? n : min(per, n);
    }
    if (per < 1) return cuda_failed(cudaErrorInvalidConfiguration, "tensor-core attend occupancy");
    cached[dev][di][hb][rb] = sms * per;
  }
  const int nhb = Hkv / hb;
  *out = (cached[dev][di][hb][rb] + nhb - 1) / nhb;
  return KV_OK;
}

}  // namespace

int mma_attend_max_tokens(int Hq, int Hkv, int d) {
  if ((d != 64 && d != 128) || Hkv <= 0 || Hq <= 0 || Hq % Hkv) return 0;
  return kMmaRows * kMaxRowBlocks / (Hq / Hkv);  // 0 when G > 64
}

bool mma_attend_supported(int Hq, int Hkv, int d, int Tq) {
  return (d == 64 || d == 128) && Hkv > 0 && Hq % Hkv == 0 && Tq >= 1 &&
         (long long)(Hq / Hkv) * Tq <= (long long)kMmaRows * kMaxRowBlocks;
}

size_t mma_attend_workspace_size(int B, int Hkv, int rows, int d, int max_pages,
                                 int pages_per_split, size_t region) {
  long long chunks = 0;
  if (B < 0 || Hkv < 1 || rows < 1 || rows > kMmaRows * kMaxRowBlocks || max_pages < 0 ||
      pages_per_split < 0 || (d != 64 && d != 128) || mma_chunks(Hkv, rows, d, &chunks))
    return 0;
  return mma_layout(B, Hkv, rows, d, max_pages, pages_per_split, chunks, region).total;
}

int mma_attend_launch(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                      int Tq, int Tstride, int len_shift, int Hq, int Hkv, int d, int dtype,
                      float scale, int pages_per_split, float* out, float* lse, void* ws,
                      size_t ws_bytes, size_t region, cudaStream_t stream) {
  if (!mma_attend_supported(Hq, Hkv, d, Tq) || (dtype != KV_F16 && dtype != KV_BF16))
    return KV_EINVAL;
  if (Tstride < Tq || len_shift < 0) return KV_EINVAL;
  if (B < 0 || num_pages < 1 || max_pages < 0 || pages_per_split < 0) return KV_EINVAL;
  if (B == 0) return KV_OK;
  if ((long long)B * max_pages > 0x7fffffffll) return KV_EINVAL;  // page offsets are int32
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out || !lse || !ws)
    return KV_EINVAL;
  if (((uintptr_t)q & 3) || ((uintptr_t)k_pool & 15) || ((uintptr_t)v_pool & 15) ||
      ((uintptr_t)out & 15) || ((uintptr_t)ws & 255))
    return KV_EINVAL;
  long long chunks = 0;
  const int rows = (Hq / Hkv) * Tq, rb = row_blocks(rows);
  int rc = mma_chunks(Hkv, rows, d, &chunks);
  if (rc) return rc;
  const MmaLayout L = mma_layout(B, Hkv, rows, d, max_pages, pages_per_split, chunks, region);
  if (ws_bytes < L.total) return KV_EWORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int hb = head_block(Hkv, rb), nhb = Hkv / hb;
  CUtensorMap tmk, tmv;
  rc = encode_pool_map(&tmk, k_pool, num_pages, Hkv, hb, dtype, d);
  if (rc) return rc;
  rc = encode_pool_map(&tmv, v_pool, num_pages, Hkv, hb, dtype, d);
  if (rc) return rc;

  int* status = reinterpret_cast<int*>(w);
  int32_t* page_off = reinterpret_cast<int32_t*>(w + L.page_off);

  const bool fused_offsets = B <= kFusedMaxB;
  if (!fused_offsets) {
    OffsetsArgs oa{};
    oa.seq_lens = seq_lens;
    oa.B = B;
    oa.page_size = 16;
    oa.max_pages = max_pages;
    oa.len_shift = len_shift;
    oa.page_off = page_off;
    oa.status = status;
    KV_CUDA_CHECK(launch_page_offsets(oa, stream));
  }

  MmaParams mp{};
  mp.q = static_cast<const uint16_t*>(q);
  mp.table = block_table;
  mp.seq_lens = seq_lens;
  mp.page_off_in = fused_offsets ? nullptr : page_off;
  mp.page_off_out = fused_offsets ? page_off : nullptr;
  mp.chunk_out = reinterpret_cast<int32_t*>(w + L.chunk);
  mp.out = out;
  mp.lse = lse;
  mp.part_o = reinterpret_cast<float*>(w + L.part_o);
  mp.part_lse = reinterpret_cast<float*>(w + L.part_lse);
  mp.status = status;
  mp.B = B;
  mp.num_pages = num_pages;
  mp.max_pages = max_pages;
  mp.Hq = Hq;
  mp.Hkv = Hkv;
  mp.G = Hq / Hkv;
  mp.Tq = Tq;
  mp.Tstride = Tstride;
  mp.len_shift = len_shift;
  mp.rows = rows;
  mp.rows_pad = rb * kMmaRows;
  mp.stages = ring_stages(hb, d);
  mp.rb = rb;
  mp.hb = hb;
  mp.nhb = nhb;
  mp.chunk_req = pages_per_split;
  mp.n_chunks = chunks;
  mp.scale_log2 = scale * 1.4426950408889634f;
  mp.test_wait_ns = test_consumer_wait_ns();
  // one CTA per (chunk, head block); chunks beyond the batch's count exit
  const long long grid = L.max_chunks * nhb;
  if (grid > 0x7fffffffll) return KV_EINVAL;
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;
  take_profile_events(&ev_before, &ev_after);
  if (ev_before) KV_CUDA_CHECK(cudaEventRecord(ev_before, stream));
  const dim3 block(32 * (1 + hb * rb));
  const AttendFn kernel = dtype == KV_BF16
                              ? (d == 64 ? mma_attend_kernel<BF16, 64> : mma_attend_kernel<BF16, 128>)
                              : (d == 64 ? mma_attend_kernel<F16, 64> : mma_attend_kernel<F16, 128>);
  KV_CUDA_CHECK(launch(kernel, dim3((unsigned)grid), block, mma_smem(hb, d), stream, true, tmk, tmv,
                       mp));
  if (ev_after) KV_CUDA_CHECK(cudaEventRecord(ev_after, stream));  // the attention kernel alone
  MmaMergeParams gp{};
  gp.page_off = page_off;
  gp.chunk = mp.chunk_out;
  gp.part_o = mp.part_o;
  gp.part_lse = mp.part_lse;
  gp.out = out;
  gp.lse = lse;
  gp.B = B;
  gp.Hq = Hq;
  gp.Hkv = Hkv;
  gp.G = mp.G;
  gp.Tstride = Tstride;
  gp.rows = mp.rows;
  gp.rows_pad = mp.rows_pad;
  const dim3 mgrid((unsigned)((long long)B * Hkv), (unsigned)mp.rows);
  int dev = 0, sms = 0;
  KV_CUDA_CHECK(cudaGetDevice(&dev));
  KV_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const bool wide = (long long)B * Hkv * mp.rows <= sms;  // 16 warps per row, else 4
  if (d == 64)
    KV_CUDA_CHECK(launch(wide ? mma_merge_kernel<16, 64> : mma_merge_kernel<4, 64>, mgrid,
                         dim3((wide ? 16 : 4) * 32), 0, stream, true, gp));
  else
    KV_CUDA_CHECK(launch(wide ? mma_merge_kernel<16, 128> : mma_merge_kernel<4, 128>, mgrid,
                         dim3((wide ? 16 : 4) * 32), 0, stream, true, gp));
  return KV_OK;
}

}  // namespace kvb
