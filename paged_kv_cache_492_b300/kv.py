"""Python binding of the C ABI in include/kv.h (ctypes).

Argument marshalling only: every function here forwards to the CUDA library
libkv.so with the same name; all computation happens in its kernels.  Tensors
are torch tensors (device memory and streams come from torch); raw integers
are accepted wherever a pointer is expected.  A missing or unloadable
library raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
import re
import threading
from typing import Optional

import torch

from . import build as _build

KV_OK, KV_EINVAL, KV_EBADPAGE, KV_ENOSPACE, KV_EWORKSPACE, KV_ECUDA, KV_EFULL, KV_ETIMEOUT = (
    0, -1, -2, -3, -4, -5, -6, -7)
KV_F16, KV_BF16 = 0, 1
# pages_per_split value selecting the tensor-core decode engine
KV_DECODE_TENSOR_CORE = -1
KV_SELECT_TOPK, KV_SELECT_BOUNDARY = 0, 1

HEADER = os.path.join(_build.INCLUDE, "kv.h")
_lock = threading.Lock()
_lib = None


class KVError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        msg = status_string(code) if _lib is not None else str(code)
        if code == KV_ECUDA and _lib is not None:
            msg += f" [{last_error()}]"
        super().__init__(f"{what}: {msg} ({code})" if what else f"{msg} ({code})")
        self.code = code


def declared_functions() -> list:
    """Names of the functions include/kv.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_[a-z0-9_]+)\s*\(", text)))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if _build.stale():
                _build.build()
            if not os.path.exists(path):
                raise ImportError(f"CUDA library {path} is missing; run paged_kv_cache_492_b300.build")
            _lib = C.CDLL(path)
            _declare(_lib)
    return _lib


P, I, SZ, F = C.c_void_p, C.c_int, C.c_size_t, C.c_float

_SIGS = {
    "kv_status_string": ([I], C.c_char_p),
    "kv_last_error": ([], C.c_char_p),
    "kv_status_workspace_size": ([], SZ),
    "kv_workspace_reset": ([P, SZ, P], I),
    "kv_get_status": ([P, P], I),
    "kv_decode_num_workers": ([I, I, I, I, I], I),
    "kv_decode_workspace_size": ([I, I, I, I, I, I, I], SZ),
    "kv_decode": ([P, P, P, I, P, I, P, I, I, I, I, I, I, F, I, P, P, P, SZ, P], I),
    "kv_decode_noalloc": ([P, P, P, I, P, I, P, I, I, I, I, I, I, F, I, P, P, P, P], I),
    "kv_decode_hostio_workspace_size": ([I, I, I, I, I, I, I], SZ),
    "kv_decode_hostio": ([P, P, P, I, P, I, P, I, I, I, I, I, I, F, I, P, P, P, SZ, P], I),
    "kv_workqueue_workspace_size": ([I], SZ),
    "kv_profile_next_decode": ([P, P], I),
    "kv_test_consumer_timeout": ([C.c_ulonglong], I),
    "kv_attend_multi_workspace_size": ([I, I, I, I, I, I, I, I], SZ),
    "kv_attend_multi": ([P, P, P, I, P, I, P, I, I, I, I, I, I, I, F, I, P, P, P, SZ, P], I),
    "kv_decode_tune": ([P, P, P, I, P, I, P, I, I, I, I, I, I, F, P, I, I, P, P, P, P, P, SZ, P,
                        SZ, P], I),
    "kv_build_workqueue": ([P, I, I, I, I, I, I, P, I, P, I, P, P, P, P, P], I),
    "kv_update_query_summaries": ([P, I, I, I, I, I, F, F, I, P, P], I),
    "kv_mark_active": ([P, P, I, I, I, P, P], I),
    "kv_page_summaries": ([P, I, P, I, I, I, I, I, P, P, SZ, P], I),
    "kv_summarize_last_pages": ([P, I, P, I, P, P, I, I, I, I, I, P, P, SZ, P], I),
    "kv_score_pages": ([P, P, I, P, I, P, P, I, I, I, I, P, P, SZ, P], I),
    "kv_select_workspace_size": ([I, I], SZ),
    "kv_select_pages": ([P, P, P, P, I, I, I, I, I, F, F, I, P, P, P, P, P, SZ, P], I),
    "kv_compact_workspace_size": ([I, I, I, I], SZ),
    "kv_compact": ([P, I, P, P, I, P, P, I, P, P, P, I, I, I, I, I, P, SZ, P], I),
    "kv_append_workspace_size": ([I], SZ),
    "kv_free_list_push": ([I, I, P, I, P, P, P], I),
    "kv_budget_step_workspace_size": ([I, I], SZ),
    "kv_budget_step": ([P, P, P, P, P, I, P, I, P, P, I, I, I, I, I, I, F, F, I, I, I, F, F, P, P, P,
                        P, P, P, P, P, P, P, SZ, P], I),
    "kv_vmm_pool_create": ([I, SZ, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                            C.POINTER(C.c_size_t)], I),
    "kv_vmm_pool_resize": ([P, SZ, C.POINTER(C.c_size_t)], I),
    "kv_vmm_pool_mapped": ([P], SZ),
    "kv_vmm_pool_destroy": ([P], I),
    "kv_append": ([P, P, P, P, I, P, I, P, P, P, P, I, I, I, I, I, P, SZ, P], I),
}


def _declare(L):
    for name, (args, res) in _SIGS.items():
        fn = getattr(L, name, None)
        if fn is None:
            continue
        fn.argtypes = args
        fn.restype = res


def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    raise TypeError(f"expected a tensor or an address, got {type(x)}")


def _s(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc, what):
    if rc != KV_OK:
        raise KVError(rc, what)


def dtype_code(t) -> int:
    dt = t.dtype if isinstance(t, torch.Tensor) else t
    if dt == torch.float16:
        return KV_F16
    if dt == torch.bfloat16:
        return KV_BF16
    raise TypeError(f"unsupported element type {dt}")


def status_string(code: int) -> str:
    return lib().kv_status_string(int(code)).decode()


def last_error() -> str:
    """The failing CUDA runtime call behind the last KV_ECUDA on this thread."""
    return lib().kv_last_error().decode()


# ---------------------------------------------------------------- workspace
def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zeroed device buffer usable as a workspace (torch allocations are
    at least 256-byte aligned)."""
    ws = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    return ws


def kv_status_workspace_size() -> int:
    return lib().kv_status_workspace_size()


def kv_workspace_reset(ws, stream=None):
    _check(lib().kv_workspace_reset(_p(ws), ws.numel(), _s(stream)), "kv_workspace_reset")


def kv_get_status(ws, stream=None) -> int:
    return lib().kv_get_status(_p(ws), _s(stream))


def check_status(ws, stream=None, what="device"):
    rc = kv_get_status(ws, stream)
    _check(rc, what)


# ---------------------------------------------------------------- decode
def kv_decode_num_workers(Hq, Hkv, d, page_size=16, dtype=KV_F16) -> int:
    n = lib().kv_decode_num_workers(Hq, Hkv, d, page_size, dtype)
    if n < 0:
        raise KVError(n, "kv_decode_num_workers")
    return n


def kv_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size=16, pages_per_split=0) -> int:
    return lib().kv_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size, pages_per_split)


def kv_decode(q, k_pool, v_pool, block_table, seq_lens, scale, out, lse, ws,
              pages_per_split=0, stream=None, *, num_pages=None, dtype=None):
    """q [B,Hq,d], pools [P,Hkv,16,d] (f16/bf16), block_table [B,maxP] int32,
    seq_lens [B] int32, out [B,Hq,d] f32, lse [B,Hq] f32, ws from
    alloc_workspace(kv_decode_workspace_size(...))."""
    B, Hq, d = q.shape
    P_, Hkv, ps, _ = k_pool.shape
    rc = lib().kv_decode(_p(q), _p(k_pool), _p(v_pool), int(num_pages if num_pages is not None else P_),
                         _p(block_table), block_table.shape[1], _p(seq_lens), B, ps, Hq, Hkv, d,
                         dtype_code(q) if dtype is None else dtype, float(scale),
                         int(pages_per_split), _p(out), _p(lse), _p(ws), ws.numel(), _s(stream))
    _check(rc, "kv_decode")


def prepare_decode(q, k_pool, v_pool, block_table, seq_lens, scale, out, lse, ws,
                   pages_per_split=0, stream=None):
    """kv_decode with its arguments marshalled once: returns a callable that
    issues the same C call again (returning the status code) -- for loops
    that replay one step and should not pay the marshalling each time."""
    B, Hq, d = q.shape
    P_, Hkv, ps, _ = k_pool.shape
    fn = lib().kv_decode
    args = (_p(q), _p(k_pool), _p(v_pool), P_, _p(block_table), block_table.shape[1],
            _p(seq_lens), B, ps, Hq, Hkv, d, dtype_code(q), float(scale), int(pages_per_split),
            _p(out), _p(lse), _p(ws), ws.numel(), _s(stream))
    cargs = [t(a) if a is not None else None for t, a in zip(fn.argtypes, args)]

    def call() -> int:
        return fn(*cargs)

    return call


def kv_decode_noalloc(q, k_pool, v_pool, block_table, seq_lens, scale, out, lse, status,
                      pages_per_split=0, stream=None):
    """kv_decode without a workspace, for callers that cannot allocate device
    memory: scratch lives in the library's fixed 16 MiB device array.
    `status` is a 1-element int32 device tensor that receives the first
    device-side error code (0 if none).  Calls that overlap on the GPU race
    on the shared scratch."""
    B, Hq, d = q.shape
    P_, Hkv, ps, _ = k_pool.shape
    rc = lib().kv_decode_noalloc(_p(q), _p(k_pool), _p(v_pool), P_, _p(block_table),
                                 block_table.shape[1], _p(seq_lens), B, ps, Hq, Hkv, d,
                                 dtype_code(q), float(scale), int(pages_per_split), _p(out),
                                 _p(lse), _p(status), _s(stream))
    _check(rc, "kv_decode_noalloc")


def kv_decode_hostio_workspace_size(B, Hq, Hkv, d, max_pages, page_size=16, pages_per_split=0):
    return lib().kv_decode_hostio_workspace_size(B, Hq, Hkv, d, max_pages, page_size,
                                                 pages_per_split)


def kv_decode_hostio(h_q, k_pool, v_pool, h_block_table, h_seq_lens, scale, h_out, h_lse, ws,
                     pages_per_split=0, stream=None):
    """Like kv_decode with q, block_table, seq_lens, out and lse in (pinned) host memory."""
    B, Hq, d = h_q.shape
    P_, Hkv, ps, _ = k_pool.shape
    rc = lib().kv_decode_hostio(_p(h_q), _p(k_pool), _p(v_pool), P_, _p(h_block_table),
                                h_block_table.shape[1], _p(h_seq_lens), B, ps, Hq, Hkv, d,
                                dtype_code(k_pool), float(scale), int(pages_per_split), _p(h_out),
                                _p(h_lse), _p(ws), ws.numel(), _s(stream))
    _check(rc, "kv_decode_hostio")


def kv_attend_multi_workspace_size(B, T, Hq, Hkv, d, max_pages, page_size=16,
                                   pages_per_split=0) -> int:
    return lib().kv_attend_multi_workspace_size(B, T, Hq, Hkv, d, max_pages, page_size,
                                                pages_per_split)


def kv_attend_multi(q, k_pool, v_pool, block_table, seq_lens, scale, out, lse, ws,
                    pages_per_split=0, stream=None):
    """q [B, T, Hq, d] (the last T tokens of each sequence, causal), out
    [B, T, Hq, d] f32, lse [B, T, Hq] f32."""
    B, T, Hq, d = q.shape
    P_, Hkv, ps, _ = k_pool.shape
    rc = lib().kv_attend_multi(_p(q), _p(k_pool), _p(v_pool), P_, _p(block_table),
                               block_table.shape[1], _p(seq_lens), B, T, ps, Hq, Hkv, d,
                               dtype_code(q), float(scale), int(pages_per_split), _p(out), _p(lse),
                               _p(ws), ws.numel(), _s(stream))
    _check(rc, "kv_attend_multi")


def kv_decode_tune(q, k_pool, v_pool, block_table, seq_lens, scale, out, lse, ws, candidates,
                   reps=5, stream=None, flush=None):
    """Time kv_decode for each candidate pages_per_split (0 = automatic,
    KV_DECODE_TENSOR_CORE = the tensor-core engine) on these inputs ->
    (best candidate, [us per candidate, the mean of the middle half of its
    reps]).  flush: a device buffer more than twice the L2 size, overwritten
    and half read back before every timed call so L2 holds none of the inputs
    and no dirty lines (None: timed warm)."""
    B, Hq, d = q.shape
    P_, Hkv, ps, _ = k_pool.shape
    cand = (C.c_int32 * len(candidates))(*[int(c) for c in candidates])
    us = (C.c_float * len(candidates))()
    best = C.c_int32()
    rc = lib().kv_decode_tune(_p(q), _p(k_pool), _p(v_pool), P_, _p(block_table),
                              block_table.shape[1], _p(seq_lens), B, ps, Hq, Hkv, d,
                              dtype_code(q), float(scale), cand, len(candidates), int(reps),
                              _p(out), _p(lse), us, C.byref(best), _p(ws), ws.numel(),
                              _p(flush) if flush is not None else None,
                              flush.numel() * flush.element_size() if flush is not None else 0,
                              _s(stream))
    _check(rc, "kv_decode_tune")
    return int(best.value), [float(u) for u in us]


class DecodePolicy:
    """Per-workload choice of the decode engine and split size, calibrated on
    first sight (PersistentKV's adaptive policy, aissential.tech, Summary,
    restated among this library's own variants: the fused kernel's split
    sizes and the tensor-core engine).  A workload's signature is its batch
    size, log2 of its page count and its long-to-mean length ratio (rounded);
    the first batch with a new signature is timed with kv_decode_tune and the
    fastest variant is reused for every later batch with that signature.  The
    workspace must be sized for every candidate (workspace_size).  With
    `flush` (a device buffer more than twice the L2 size) the candidates are
    timed with L2 flushed before each call, as a step that follows other work
    runs."""

    def __init__(self, candidates=(0, 8, 16, 32, 64, 128, KV_DECODE_TENSOR_CORE), reps=5,
                 flush=None):
        self.candidates = tuple(int(c) for c in candidates)
        self.reps = reps
        self.flush = flush
        self.table = {}

    def usable(self, B, Hq, Hkv, d, max_pages, page_size=16):
        """The candidates this shape supports (the tensor-core engine needs
        d = 64 or 128 and G <= 64; an unsupported variant has workspace size 0)."""
        return [c for c in self.candidates
                if kv_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size, c) > 0]

    def workspace_size(self, B, Hq, Hkv, d, max_pages, page_size=16):
        """Bytes a workspace needs to run every usable candidate (0 when none is)."""
        sizes = [kv_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size, c)
                 for c in self.usable(B, Hq, Hkv, d, max_pages, page_size)]
        return max(sizes) if sizes else 0

    @staticmethod
    def signature(seq_lens_host, page_size=16):
        import math

        pages = [-(-int(L) // page_size) for L in seq_lens_host]
        W = sum(pages)
        mean = W / max(1, len(pages))
        ratio = (max(pages) / mean) if W else 0.0
        return (len(pages), int(math.log2(W)) if W else -1, round(ratio))

    def pages_per_split(self, seq_lens_host, q, k_pool, v_pool, block_table, seq_lens, scale, out,
                        lse, ws, stream=None):
        sig = self.signature(seq_lens_host, k_pool.shape[2])
        if sig not in self.table:
            B, Hq, d = q.shape
            _, Hkv, ps, _ = k_pool.shape
            cands = self.usable(B, Hq, Hkv, d, block_table.shape[1], ps)
            if not cands:
                raise KVError(KV_EINVAL, "DecodePolicy: no candidate supports this shape")
            best, us = kv_decode_tune(q, k_pool, v_pool, block_table, seq_lens, scale, out, lse, ws,
                                      cands, self.reps, stream, flush=self.flush)
            self.table[sig] = (best, dict(zip(cands, us)))
        return self.table[sig][0]


def prepare_decode_hostio(h_q, k_pool, v_pool, h_block_table, h_seq_lens, scale, h_out, h_lse, ws,
                          pages_per_split=0, stream=None):
    """kv_decode_hostio with its arguments marshalled once (see prepare_decode)."""
    B, Hq, d = h_q.shape
    P_, Hkv, ps, _ = k_pool.shape
    fn = lib().kv_decode_hostio
    args = (_p(h_q), _p(k_pool), _p(v_pool), P_, _p(h_block_table), h_block_table.shape[1],
            _p(h_seq_lens), B, ps, Hq, Hkv, d, dtype_code(k_pool), float(scale),
            int(pages_per_split), _p(h_out), _p(h_lse), _p(ws), ws.numel(), _s(stream))
    cargs = [t(a) if a is not None else None for t, a in zip(fn.argtypes, args)]

    def call() -> int:
        return fn(*cargs)

    return call


def kv_profile_next_decode(event_before, event_after):
    """Arm CUDA events (torch.cuda.Event) around the next decode's attention kernel."""
    ev0 = event_before.cuda_event if event_before is not None else None
    ev1 = event_after.cuda_event if event_after is not None else None
    _check(lib().kv_profile_next_decode(ev0, ev1), "kv_profile_next_decode")


def kv_test_consumer_timeout(ns: int):
    """Failure-path test mode: while ns > 0, each decode consumer warp first
    waits ns nanoseconds on a barrier nothing completes, so the kernel ends
    with KV_ETIMEOUT (no GPU fault); 0 turns it off."""
    _check(lib().kv_test_consumer_timeout(int(ns)), "kv_test_consumer_timeout")


def kv_workqueue_workspace_size(B) -> int:
    return lib().kv_workqueue_workspace_size(B)


def kv_build_workqueue(seq_lens, Hkv, page_size, max_pages, pages_per_split, n_workers, tasks,
                       chunk_begin, seq_group_begin, seq_nsplit, meta, ws, stream=None):
    rc = lib().kv_build_workqueue(_p(seq_lens), seq_lens.numel(), Hkv, page_size, max_pages,
                                  pages_per_split, n_workers, _p(tasks), tasks.shape[0],
                                  _p(chunk_begin), chunk_begin.numel(), _p(seq_group_begin),
                                  _p(seq_nsplit), _p(meta), _p(ws), _s(stream))
    _check(rc, "kv_build_workqueue")


# ---------------------------------------------------------------- budgeting
def kv_update_query_summaries(q, Hkv, a_fast, a_slow, first, ema, stream=None):
    B, Hq, d = q.shape
    rc = lib().kv_update_query_summaries(_p(q), B, Hq, Hkv, d, dtype_code(q), float(a_fast),
                                         float(a_slow), int(bool(first)), _p(ema), _s(stream))
    _check(rc, "kv_update_query_summaries")


def kv_mark_active(seq_lens, budget, page_size, mode, active, stream=None):
    rc = lib().kv_mark_active(_p(seq_lens), _p(budget), seq_lens.numel(), page_size, int(mode),
                              _p(active), _s(stream))
    _check(rc, "kv_mark_active")


def kv_page_summaries(k_pool, page_ids, summ, ws, stream=None):
    P_, Hkv, ps, d = k_pool.shape
    rc = lib().kv_page_summaries(_p(k_pool), P_, _p(page_ids), page_ids.numel(), Hkv, ps, d,
                                 dtype_code(k_pool), _p(summ), _p(ws), ws.numel(), _s(stream))
    _check(rc, "kv_page_summaries")


def kv_summarize_last_pages(k_pool, block_table, seq_lens, active, summ, ws, stream=None):
    P_, Hkv, ps, d = k_pool.shape
    B, maxp = block_table.shape
    rc = lib().kv_summarize_last_pages(_p(k_pool), P_, _p(block_table), maxp, _p(seq_lens),
                                       _p(active), B, Hkv, ps, d, dtype_code(k_pool), _p(summ),
                                       _p(ws), ws.numel(), _s(stream))
    _check(rc, "kv_summarize_last_pages")


def kv_score_pages(query_summaries, page_key_summaries, block_table, seq_lens, active, scores, ws,
                   page_size=16, stream=None):
    B, _, Hkv, d = query_summaries.shape
    P_ = page_key_summaries.shape[0]
    maxp = block_table.shape[1]
    rc = lib().kv_score_pages(_p(query_summaries), _p(page_key_summaries), P_, _p(block_table),
                              maxp, _p(seq_lens), _p(active), B, Hkv, d, page_size, _p(scores),
                              _p(ws), ws.numel(), _s(stream))
    _check(rc, "kv_score_pages")


def kv_select_workspace_size(B, max_pages) -> int:
    return lib().kv_select_workspace_size(B, max_pages)


def kv_select_pages(scores, seq_lens, active, budget, n_first, n_last, delta, ws_frac, mode,
                    free_top, keep_mask, grow, drift, ws, page_size=16, stream=None):
    B, maxp, _ = scores.shape
    rc = lib().kv_select_pages(_p(scores), _p(seq_lens), _p(active), _p(budget), B, maxp,
                               page_size, int(n_first), int(n_last), float(delta), float(ws_frac),
                               int(mode), _p(free_top), _p(keep_mask), _p(grow), _p(drift),
                               _p(ws), ws.numel(), _s(stream))
    _check(rc, "kv_select_pages")


def kv_compact_workspace_size(B, max_pages, num_pages=0, token_granular=False) -> int:
    """num_pages: the pool's pages if the compaction will get refcnt, else 0."""
    return lib().kv_compact_workspace_size(B, max_pages, num_pages, int(bool(token_granular)))


def kv_compact(block_table, seq_lens, keep_mask, token_granular, k_pool, v_pool, free_list,
               free_top, ws, stream=None, refcnt=None):
    B, maxp = block_table.shape
    P_, Hkv, ps, d = k_pool.shape
    rc = lib().kv_compact(_p(block_table), maxp, _p(seq_lens), _p(keep_mask),
                          int(bool(token_granular)), _p(k_pool), _p(v_pool), P_, _p(free_list),
                          _p(free_top), _p(refcnt), B, Hkv, d, ps, dtype_code(k_pool), _p(ws),
                          ws.numel(), _s(stream))
    _check(rc, "kv_compact")


def kv_append_workspace_size(B) -> int:
    return lib().kv_append_workspace_size(B)


def kv_append(k_new, v_new, k_pool, v_pool, block_table, seq_lens, free_list, free_top, ws,
              stream=None, refcnt=None):
    B, Hkv, d = k_new.shape
    P_, _, ps, _ = k_pool.shape
    rc = lib().kv_append(_p(k_new), _p(v_new), _p(k_pool), _p(v_pool), P_, _p(block_table),
                         block_table.shape[1], _p(seq_lens), _p(free_list), _p(free_top),
                         _p(refcnt), B, Hkv, d, ps, dtype_code(k_pool), _p(ws), ws.numel(),
                         _s(stream))
    _check(rc, "kv_append")


def kv_budget_step_workspace_size(B, max_pages) -> int:
    return lib().kv_budget_step_workspace_size(B, max_pages)


def kv_budget_step(q, k_new, v_new, k_pool, v_pool, block_table, seq_lens, budget, a_fast, a_slow,
                   update_ema, n_first, n_last, delta, ws_frac, ema, summ, scores, active,
                   keep_mask, grow, drift, free_list, free_top, ws, stream=None):
    """The steady-state step's budgeting part in one launch (see kv.h)."""
    B, Hq, d = q.shape
    P_, Hkv, ps, _ = k_pool.shape
    rc = lib().kv_budget_step(_p(q), _p(k_new), _p(v_new), _p(k_pool), _p(v_pool), P_,
                              _p(block_table), block_table.shape[1], _p(seq_lens), _p(budget), B,
                              Hq, Hkv, d, ps, dtype_code(k_pool), float(a_fast), float(a_slow),
                              int(bool(update_ema)), int(n_first), int(n_last), float(delta),
                              float(ws_frac), _p(ema), _p(summ), _p(scores), _p(active),
                              _p(keep_mask), _p(grow), _p(drift), _p(free_list), _p(free_top),
                              _p(ws), ws.numel(), _s(stream))
    _check(rc, "kv_budget_step")


def kv_free_list_push(first_page, n, free_list, free_top, ws, stream=None):
    """Push pool pages [first_page, first_page + n) onto the free list
    (highest id first, so they pop in ascending order)."""
    rc = lib().kv_free_list_push(int(first_page), int(n), _p(free_list), free_list.numel(),
                                 _p(free_top), _p(ws), _s(stream))
    _check(rc, "kv_free_list_push")

# ---------------------------------------------------------------- elastic pool
class VmmPool:
    """An elastic page pool: a reserved device address range whose backing
    grows and shrinks at the top (kv_vmm_pool_*).  `tensor(shape, dtype)`
    views the range's start as a torch tensor (the caller keeps the pool
    alive and only touches the mapped part)."""

    def __init__(self, max_bytes: int, device: int = 0):
        h, base, gran = C.c_void_p(), C.c_void_p(), C.c_size_t()
        _check(lib().kv_vmm_pool_create(int(device), int(max_bytes), C.byref(h), C.byref(base),
                                        C.byref(gran)), "kv_vmm_pool_create")
        self.handle, self.base, self.granularity = h.value, base.value, gran.value
        self.device = device

    def resize(self, nbytes: int) -> int:
        m = C.c_size_t()
        _check(lib().kv_vmm_pool_resize(self.handle, int(nbytes), C.byref(m)), "kv_vmm_pool_resize")
        return m.value

    @property
    def mapped(self) -> int:
        return lib().kv_vmm_pool_mapped(self.handle)

    def tensor(self, shape, dtype) -> torch.Tensor:
        """A tensor over the start of the range (no copy, no ownership); it
        must lie inside the mapped part, and the pool must outlive it."""
        import math

        esize = torch.empty((), dtype=dtype).element_size()
        n = math.prod(shape)
        if n * esize > self.mapped:
            raise ValueError("view larger than the mapped part of the pool")
        code = {1: "|u1", 2: "<i2", 4: "<i4"}[esize]

        class _View:
            __cuda_array_interface__ = {"shape": (n,), "typestr": code,
                                        "data": (self.base, False), "version": 3}

        raw = torch.as_tensor(_View(), device=f"cuda:{self.device}")
        return raw.view(dtype).view(*shape)

    def close(self):
        if self.handle:
            _check(lib().kv_vmm_pool_destroy(self.handle), "kv_vmm_pool_destroy")
            self.handle = None

