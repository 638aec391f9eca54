// Device-side helpers shared by the library's kernels: status word, mbarrier
// and bulk-copy wrappers (inline PTX for sm_103a), bounded waits, 16-bit
// conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kv.h"

namespace kvb {

// The first 256 bytes of every workspace: the device status word.
constexpr size_t kHeaderBytes = 256;
// Bounded waits give up after this long (a decode step takes well under 1 ms).
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Record the first device-side error of a call sequence (0 = none yet).
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier (shared::cta) --------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase with the given parity to complete; false after
// `limit_ns`, or as soon as *abort (shared memory, optional) is non-zero.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs,
                                          const volatile int* abort = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort && *abort) return false;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// ---- bulk copies (TMA, non-tensor) ----------------------------------------
// L2 policy for data read exactly once (K/V pages).
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// global -> shared bulk copy; `bytes` and both addresses are 16-byte multiples.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// ---- memory ordering / prefetch ----------------------------------------------
// Atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* addr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v)
               : "memory");
  return old;
}
// Start bringing a global line into L2 (no register result, never faults on
// an address inside a live allocation).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---- programmatic dependent launch ------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- fast exp2 (MUFU) -------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- 16-bit element types ----------------------------------------------------
struct F16 {
  static constexpr int code = KV_F16;
  __device__ __forceinline__ static float2 to_f2(uint32_t v) {
    __half2 h = *reinterpret_cast<__half2*>(&v);
    return __half22float2(h);
  }
  __device__ __forceinline__ static float to_f(uint16_t v) {
    return __half2float(*reinterpret_cast<__half*>(&v));
  }
};
struct BF16 {
  static constexpr int code = KV_BF16;
  // bf16 is the upper half of an fp32: widening is a shift.
  __device__ __forceinline__ static float2 to_f2(uint32_t v) {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
  }
  __device__ __forceinline__ static float to_f(uint16_t v) {
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
  }
};

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr long long ceil_div_ll(long long a, long long b) {
  return (a + b - 1) / b;
}

// ---- the split rule --------------------------------------------------------
// The non-empty pages of a batch, laid end to end (sequence b owns pages
// [O_b, O_b + np_b) of the flattened range), are cut into chunks of `chunk`
// pages; every non-empty (sequence, chunk) intersection is one split of that
// sequence.  The workqueue builder and the decode kernel both use these.

// Automatic chunk: the W pages spread over n_workers, never below min_chunk.
__host__ __device__ inline long long auto_chunk(long long W, long long n_workers, int min_chunk) {
  long long c = n_workers > 0 ? ceil_div_ll(W, n_workers) : W;
  if (c < min_chunk) c = min_chunk;
  return c < 1 ? 1 : c;
}
// Splits of a sequence with np > 0 pages starting at flattened page O.
__host__ __device__ inline long long split_count(long long O, long long np, long long chunk) {
  return np > 0 ? (O + np - 1) / chunk - O / chunk + 1 : 0;
}
// Pages [lo, hi) of the sequence (its own numbering) that fall in chunk c.
__host__ __device__ inline void split_range(long long O, long long np, long long chunk, long long c,
                                            long long* lo, long long* hi) {
  const long long a = c * chunk > O ? c * chunk : O;
  const long long e = (c + 1) * chunk < O + np ? (c + 1) * chunk : O + np;
  *lo = a - O;
  *hi = e - O;
}

// Largest b in [0, B) with O[b] <= x (O nondecreasing, O[0] = 0 <= x): the
// sequence that owns flattened page x.
__device__ __forceinline__ int seq_at(const int32_t* O, int B, long long x) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (O[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Exclusive block-wide scan of one value per thread (blockDim a multiple of
// 32, at most 1024); returns the total.  `sm` holds 32 values.
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* out_excl, long long* sm) {
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

}  // namespace kvb
