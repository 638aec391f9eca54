// Attention of several new query tokens per sequence over the paged cache --
// the step before decode (a prefill chunk, or the verification of drafted
// tokens), over the same pool and block table.  The T query tokens of
// sequence b are its last T cached tokens (their K/V already appended), and
// query i attends causally to tokens [0, L_b - T + 1 + i).
//
// The tensor-core kernel (kv_mma.cu, d = 64 or 128, page size 16) takes up
// to 64 rows per KV head (T * G) in one pass over the pages.  More query
// tokens are served in the fewest passes that fit: chunk [t0, t0 + Tc) sees
// L_b - (T - t0 - Tc) cached tokens, and the usual causal rule within the
// chunk then gives every token its own limit.  Each page is streamed once per
// pass.  A pass's time grows with its 16-row blocks (one consumer warp each),
// so the chunks use as few blocks as the T tokens need, spread evenly: where
// G divides 16, the ceil(T * G / 16) blocks are dealt out over the passes
// (larger shares first, the last pass taking the remaining tokens); otherwise
// every pass but the last is full.
#include "kv_internal.h"

namespace kvb {
namespace {

// Query tokens per pass (as many as fit in 64 rows per KV head); 0 where the
// tensor-core kernel does not apply.
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
  const int tc = mma_chunk_tokens(page_size, Hq, Hkv, d, T);
  if (!tc) return 0;
  return mma_attend_workspace_size(B, Hkv, (Hq / Hkv) * tc, d, max_pages, pages_per_split,
                                   kHeaderBytes);
}

int kv_attend_multi(const void* q, const void* k_pool, const void* v_pool, int num_pages,
                    const int32_t* block_table, int max_pages, const int32_t* seq_lens, int B,
                    int T, int page_size, int Hq, int Hkv, int d, int dtype, float scale,
                    int pages_per_split, float* out, float* lse, void* ws, size_t ws_bytes,
                    void* stream) {
  if (B < 0 || T < 1 || (long long)B * T > 0x7fffffffll) return KV_EINVAL;
  if (B == 0) return KV_OK;
  if (!seq_lens || !ws) return KV_EINVAL;
  const int tc = mma_chunk_tokens(page_size, Hq, Hkv, d, T);
  if (!tc) return KV_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the fewest passes of at most tc tokens, in order on the stream (one
  // workspace); tokens per pass from the row-block plan above
  const int G = Hq / Hkv, passes = (T + tc - 1) / tc;
  const int tpb = 16 % G == 0 ? 16 / G : 0;  // tokens per 16-row block
  const int blocks = tpb ? (T + tpb - 1) / tpb : 0;
  const size_t qrow = (size_t)Hq * d * 2;  // bytes of one query token's heads
  int t0 = 0;
  for (int pass = 0; pass < passes; ++pass) {
    int n = tpb ? (blocks / passes + (pass < blocks % passes ? 1 : 0)) * tpb : tc;
    if (n > T - t0) n = T - t0;
    const int rc = mma_attend_launch(
        q ? static_cast<const uint8_t*>(q) + (size_t)t0 * qrow : nullptr, k_pool, v_pool,
        num_pages, block_table, max_pages, seq_lens, B, n, T, T - t0 - n, Hq, Hkv, d, dtype,
        scale, pages_per_split, out ? out + (size_t)t0 * Hq * d : nullptr,
        lse ? lse + (size_t)t0 * Hq : nullptr, ws, ws_bytes, kHeaderBytes, s);
    if (rc) return rc;
    t0 += n;
  }
  return KV_OK;
}

}  // extern "C"
