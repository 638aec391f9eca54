// Attention of several new query tokens per sequence over the paged cache --
// the step before decode (a prefill chunk, or the verification of drafted
// tokens), over the same pool and block table.  The T query tokens of
// sequence b are its last T cached tokens (their K/V already appended), and
// query i attends causally to tokens [0, L_b - T + 1 + i).
//
// Two forms.  With d = 128 and page size 16 the tensor-core kernel
// (kv_mma.cu) takes up to 64 rows per KV head (T * G) in one pass over the
// pages; more query tokens are served in ceil(T * G / 64) passes over chunks
// of at most 64 / G tokens, as even as possible (chunk [t0, t0 + Tc) sees
// L_b - (T - t0 - Tc) cached tokens, and the usual causal rule within the
// chunk then gives every token its own limit), so each page is streamed
// ceil(T * G / 64) times.  Otherwise (d = 64) the
// decode kernel runs unchanged on B*T virtual sequences: virtual sequence
// b*T + i has length max(0, L_b - T + 1 + i), reads block-table row b, query
// row q[b][i] and output row out[b][i], so each page is streamed once per
// query token.
#include "kv_internal.h"

namespace kvb {
namespace {

struct MultiLensArgs {
  const int32_t* seq_lens;
  int B, T;
  int32_t* lens_v;  // [B * T]
};

__global__ void multi_lens_kernel(const MultiLensArgs a) {
  pdl_wait();  // seq_lens may come from the previous kernel on the stream
  pdl_launch_dependents();
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < (long long)a.B * a.T;
       v += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(v / a.T), i = (int)(v - (long long)b * a.T);
    const int L = a.seq_lens[b];
    // a negative length stays negative so the decode reports it
    a.lens_v[v] = L < 0 ? L : max(0, L - a.T + 1 + i);
  }
}

size_t lens_offset(size_t decode_bytes) { return align_up(decode_bytes, 256); }

// The tensor-core form wherever it applies (at T = 1 it is the tensor-core
// decode engine); tokens per pass: as many as fit in 64 rows per KV head.
int mma_chunk_tokens(int page_size, int Hq, int Hkv, int d, int T) {
  if (page_size != 16) return 0;
  const int most = mma_attend_max_tokens(Hq, Hkv, d);
  return most < T ? most : T;
}

}  // namespace
}  // namespace kvb

using namespace kvb;

extern "C" {

size_t kv_attend_multi_workspace_size(int B, int T, int Hq, int Hkv, int d, int max_pages,
                                      int page_size, int pages_per_split) {
  if (B < 0 || T < 1) return 0;
  if (const int tc = mma_chunk_tokens(page_size, Hq, Hkv, d, T))
    return mma_attend_workspace_size(B, Hkv, (Hq / Hkv) * tc, max_pages, pages_per_split,
                                     kHeaderBytes);
  const size_t base = kv_decode_workspace_size(B * T, Hq, Hkv, d, max_pages, page_size,
                                               pages_per_split);
  if (!base) return 0;
  return lens_offset(base) + align_up((size_t)(B > 0 ? B : 1) * T * 4, 256);
}

int kv_attend_multi(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                    const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                    int T, int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                    int pages_per_split, float* out, float* lse, void* ws, size_t ws_bytes,
                    void* stream) {
  if (B < 0 || T < 1 || (long long)B * T > 0x7fffffffll) return KV_EINVAL;
  if (B == 0) return KV_OK;
  if (!seq_lens || !ws) return KV_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (const int tc = mma_chunk_tokens(page_size, Hq, Hkv, d, T)) {
    // the fewest passes of at most tc tokens, as even as possible (a pass's
    // time grows with its rows), in order on the stream (one workspace)
    const int passes = (T + tc - 1) / tc, per = (T + passes - 1) / passes;
    const size_t qrow = (size_t)Hq * d * 2;  // bytes of one query token's heads
    for (int t0 = 0; t0 < T; t0 += per) {
      const int n = T - t0 < per ? T - t0 : per;
      const int rc = mma_attend_launch(
          q ? static_cast<const uint8_t*>(q) + (size_t)t0 * qrow : nullptr, k_pool, v_pool,
          num_pages, block_table, max_pages, seq_lens, B, n, T, T - t0 - n, Hq, Hkv, dtype, scale,
          pages_per_split, out ? out + (size_t)t0 * Hq * d : nullptr, lse ? lse + (size_t)t0 * Hq : nullptr,
          ws, ws_bytes, kHeaderBytes, s);
      if (rc) return rc;
    }
    return KV_OK;
  }
  const size_t base = kv_decode_workspace_size(B * T, Hq, Hkv, d, max_pages, page_size,
                                               pages_per_split);
  if (!base) return KV_EINVAL;
  if (ws_bytes < kv_attend_multi_workspace_size(B, T, Hq, Hkv, d, max_pages, page_size,
                                                pages_per_split))
    return KV_EWORKSPACE;
  MultiLensArgs a{};
  a.seq_lens = seq_lens;
  a.B = B;
  a.T = T;
  a.lens_v = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + lens_offset(base));
  const long long n = (long long)B * T;
  const unsigned blocks = (unsigned)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  KV_CUDA_CHECK(launch(multi_lens_kernel, dim3(blocks), dim3(256), 0, s, true, a));
  return decode_launch(q, k_pool, v_pool, num_pages, block_table, max_pages, a.lens_v, B * T,
                       page_size, Hq, Hkv, d, dtype, scale, pages_per_split, out, lse, ws, base, s,
                       T);
}

}  // extern "C"
