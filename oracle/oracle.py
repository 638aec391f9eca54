"""ctypes front end for the C oracle (``oracle.c``).

TEST INFRASTRUCTURE.  Imported only by the tests, the smoke check and the
benchmark's CPU-baseline leg; the library's product path never loads it.
It builds ``liboracle.so`` next to the source with gcc (fp contraction off,
so the fp32 chain is rounded operation by operation as written) and wraps
each function for numpy arrays.  Nothing here does the method's arithmetic;
it only marshals arguments.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, EBADPAGE, ENOSPACE, EFULL = 0, -1, -2, -3, -6
SELECT_TOPK, SELECT_BOUNDARY = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C, -O2, no fp contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off",
                               "-fno-fast-math", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            _declare(_lib)
    return _lib


P = C.c_void_p
I = C.c_int
I64 = C.c_int64
D = C.c_double
F = C.c_float


def _declare(L):
    L.or_f16_to_f64.argtypes = [C.c_uint16]
    L.or_f16_to_f64.restype = D
    L.or_bf16_to_f64.argtypes = [C.c_uint16]
    L.or_bf16_to_f64.restype = D
    dec = [P, P, P, P, I, I, P, I, I, I, I, I, I, D]
    L.or_decode.argtypes = dec + [P, P, I]
    L.or_decode.restype = I
    L.or_decode_rows.argtypes = dec + [P, I, P, P]
    L.or_decode_rows.restype = I
    L.or_decode_range.argtypes = dec + [I, I, I64, I64, P, P]
    L.or_decode_range.restype = I
    L.or_attend_multi.argtypes = [P, P, P, P, I, I, P, I, I, I, I, I, I, I, D, P, P, I]
    L.or_attend_multi.restype = I
    L.or_merge.argtypes = [P, P, I, I, P, P]
    L.or_merge.restype = None
    L.or_chunk_auto.argtypes = [I64, I64, I64]
    L.or_chunk_auto.restype = I64
    L.or_workqueue.argtypes = [P, I, I, I, I64, P, I64, P, I64, P, P, P]
    L.or_workqueue.restype = I
    L.or_ema_f32.argtypes = [P, I, I, I, I, I, F, F, I, P]
    L.or_ema_f32.restype = None
    L.or_ema_f64.argtypes = [P, I, I, I, I, I, D, D, I, P]
    L.or_ema_f64.restype = None
    L.or_page_summaries_f32.argtypes = [P, I, P, I, I, I, I, I, P]
    L.or_page_summaries_f32.restype = I
    L.or_page_summaries_f64.argtypes = [P, I, P, I, I, I, I, I, P]
    L.or_page_summaries_f64.restype = I
    L.or_score_pages_f32.argtypes = [P, P, I, P, I, P, P, I, I, I, I, P]
    L.or_score_pages_f32.restype = I
    L.or_score_pages_f64.argtypes = [P, P, I, P, I, P, P, I, I, I, I, P]
    L.or_score_pages_f64.restype = I
    L.or_select_pages.argtypes = [P, P, P, P, I, I, I, I, I, F, F, I, I, P, P, P]
    L.or_select_pages.restype = I
    L.or_compact.argtypes = [P, I, P, P, I, P, P, I, P, P, P, I, I, I, I]
    L.or_compact.restype = I
    L.or_append.argtypes = [P, P, P, P, I, P, I, P, P, P, P, I, I, I, I]
    L.or_append.restype = I
    L.or_mark_active.argtypes = [P, P, I, I, I, P]
    L.or_mark_active.restype = I


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    def __init__(self, rc):
        super().__init__(f"oracle returned status {rc}")
        self.rc = rc


def _check(rc):
    if rc != 0:
        raise OracleError(rc)


def f16_to_f64(bits: int) -> float:
    return lib().or_f16_to_f64(bits)


def bf16_to_f64(bits: int) -> float:
    return lib().or_bf16_to_f64(bits)


def _dec_args(x):
    return [_p(x.q), _p(x.k_pool), _p(x.v_pool), _p(x.block_table), x.max_pages, x.num_pages,
            _p(x.seq_lens), x.B, x.page_size, x.Hq, x.Hkv, x.d, x.dtype, float(x.scale)]


def _dec_fix(x):
    x.q = _c(x.q, np.uint16)
    x.k_pool = _c(x.k_pool, np.uint16)
    x.v_pool = _c(x.v_pool, np.uint16)
    x.block_table = _c(x.block_table, np.int32)
    x.seq_lens = _c(x.seq_lens, np.int32)
    return x


def decode(x, nthreads: int = 1):
    """Full decode step -> (out [B, Hq, d] f64, lse [B, Hq] f64)."""
    _dec_fix(x)
    out = np.zeros((x.B, x.Hq, x.d), dtype=np.float64)
    lse = np.zeros((x.B, x.Hq), dtype=np.float64)
    _check(lib().or_decode(*_dec_args(x), _p(out), _p(lse), int(nthreads)))
    return out, lse


def decode_rows(x, rows):
    """Decode only the listed (b, hq) rows -> (out [n, d], lse [n])."""
    _dec_fix(x)
    rows = _c(rows, np.int32).reshape(-1, 2)
    out = np.zeros((len(rows), x.d), dtype=np.float64)
    lse = np.zeros(len(rows), dtype=np.float64)
    _check(lib().or_decode_rows(*_dec_args(x), _p(rows), len(rows), _p(out), _p(lse)))
    return out, lse


def decode_range(x, b, hq, t0, t1):
    _dec_fix(x)
    out = np.zeros(x.d, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    _check(lib().or_decode_range(*_dec_args(x), int(b), int(hq), int(t0), int(t1),
                                 _p(out), _p(lse)))
    return out, float(lse[0])


def attend_multi(x, q_multi, nthreads: int = 1):
    """T query tokens per sequence (the last T tokens, causal) -> (out [B, T, Hq, d] f64,
    lse [B, T, Hq] f64).  q_multi [B, T, Hq, d] 16-bit bits; the rest of x as for decode."""
    _dec_fix(x)
    q_multi = _c(q_multi, np.uint16)
    B, T, Hq, d = q_multi.shape
    out = np.zeros((B, T, Hq, d), dtype=np.float64)
    lse = np.zeros((B, T, Hq), dtype=np.float64)
    _check(lib().or_attend_multi(_p(q_multi), _p(x.k_pool), _p(x.v_pool), _p(x.block_table),
                                 x.max_pages, x.num_pages, _p(x.seq_lens), B, T, x.page_size, Hq,
                                 x.Hkv, d, x.dtype, float(x.scale), _p(out), _p(lse),
                                 int(nthreads)))
    return out, lse


def merge(lse_parts, out_parts):
    lse_parts = _c(lse_parts, np.float64)
    out_parts = _c(out_parts, np.float64)
    n, d = out_parts.shape
    out = np.zeros(d, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib().or_merge(_p(lse_parts), _p(out_parts), n, d, _p(lse), _p(out))
    return out, float(lse[0])


def chunk_auto(W, n_workers, min_chunk):
    return int(lib().or_chunk_auto(int(W), int(n_workers), int(min_chunk)))


def workqueue(seq_lens, Hkv, page_size, chunk):
    """-> dict(tasks [T, 8] int32, chunk_begin [nchunks+1], seq_group_begin [B],
    seq_nsplit [B], T, groups, chunk, nchunks, W)."""
    seq_lens = _c(seq_lens, np.int32)
    B = len(seq_lens)
    W = int(sum(-(-int(L) // page_size) for L in seq_lens))
    max_chunks = (-(-W // chunk) if W else 0) + 2
    max_tasks = Hkv * (B + max_chunks) + 1
    tasks = np.zeros((max_tasks, 8), dtype=np.int32)
    cb = np.zeros(max_chunks, dtype=np.int32)
    sgb = np.zeros(max(B, 1), dtype=np.int32)
    sns = np.zeros(max(B, 1), dtype=np.int32)
    meta = np.zeros(5, dtype=np.int64)
    _check(lib().or_workqueue(_p(seq_lens), B, Hkv, page_size, int(chunk), _p(tasks), max_tasks,
                              _p(cb), max_chunks, _p(sgb), _p(sns), _p(meta)))
    T, ng, ch, nc, W = (int(v) for v in meta)
    return dict(tasks=tasks[:T].copy(), chunk_begin=cb[: nc + 1].copy(),
                seq_group_begin=sgb[:B].copy(), seq_nsplit=sns[:B].copy(),
                T=T, groups=ng, chunk=ch, nchunks=nc, W=W)


def ema_f32(q, B, Hq, Hkv, d, dtype, a_fast, a_slow, first, ema):
    q = _c(q, np.uint16)
    assert ema.dtype == np.float32 and ema.flags.c_contiguous
    lib().or_ema_f32(_p(q), B, Hq, Hkv, d, dtype, float(a_fast), float(a_slow), int(first), _p(ema))
    return ema


def ema_f64(q, B, Hq, Hkv, d, dtype, a_fast, a_slow, first, ema):
    q = _c(q, np.uint16)
    assert ema.dtype == np.float64 and ema.flags.c_contiguous
    lib().or_ema_f64(_p(q), B, Hq, Hkv, d, dtype, float(a_fast), float(a_slow), int(first), _p(ema))
    return ema


def page_summaries_f32(k_pool, page_ids, Hkv, ps, d, dtype, summ):
    k_pool = _c(k_pool, np.uint16)
    page_ids = _c(page_ids, np.int32)
    assert summ.dtype == np.float32 and summ.flags.c_contiguous
    _check(lib().or_page_summaries_f32(_p(k_pool), k_pool.shape[0], _p(page_ids), len(page_ids),
                                       Hkv, ps, d, dtype, _p(summ)))
    return summ


def page_summaries_f64(k_pool, page_ids, Hkv, ps, d, dtype, summ):
    k_pool = _c(k_pool, np.uint16)
    page_ids = _c(page_ids, np.int32)
    assert summ.dtype == np.float64 and summ.flags.c_contiguous
    _check(lib().or_page_summaries_f64(_p(k_pool), k_pool.shape[0], _p(page_ids), len(page_ids),
                                       Hkv, ps, d, dtype, _p(summ)))
    return summ


def score_pages_f32(ema, summ, table, seq_lens, active, Hkv, d, ps, scores):
    table = _c(table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    act = None if active is None else _c(active, np.uint8)
    B, maxp = table.shape
    assert scores.dtype == np.float32 and scores.shape == (B, maxp, 2)
    _check(lib().or_score_pages_f32(_p(_c(ema, np.float32)), _p(_c(summ, np.float32)),
                                    summ.shape[0], _p(table), maxp, _p(seq_lens), _p(act), B,
                                    Hkv, d, ps, _p(scores)))
    return scores


def score_pages_f64(ema, summ, table, seq_lens, active, Hkv, d, ps, scores):
    table = _c(table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    act = None if active is None else _c(active, np.uint8)
    B, maxp = table.shape
    assert scores.dtype == np.float64 and scores.shape == (B, maxp, 2)
    _check(lib().or_score_pages_f64(_p(_c(ema, np.float64)), _p(_c(summ, np.float64)),
                                    summ.shape[0], _p(table), maxp, _p(seq_lens), _p(act), B,
                                    Hkv, d, ps, _p(scores)))
    return scores


def select_pages(scores, seq_lens, active, budget, ps, n_first, n_last, delta, mode, free_count,
                 ws_frac=0.5):
    """-> (keep_mask [B, maxP] u8, grow [B] u8, budget (updated copy), drift [B])."""
    scores = _c(scores, np.float32)
    seq_lens = _c(seq_lens, np.int32)
    B, maxp, _ = scores.shape
    act = None if active is None else _c(active, np.uint8)
    budget = _c(budget, np.int32).copy()
    keep = np.zeros((B, maxp), dtype=np.uint8)
    grow = np.zeros(B, dtype=np.uint8)
    drift = np.zeros(B, dtype=np.int32)
    _check(lib().or_select_pages(_p(scores), _p(seq_lens), _p(act), _p(budget), B, maxp, ps,
                                 int(n_first), int(n_last), float(delta), float(ws_frac),
                                 int(mode), int(free_count), _p(keep), _p(grow), _p(drift)))
    return keep, grow, budget, drift


def compact(table, seq_lens, keep, token_granular, k_pool, v_pool, free_list, free_top,
            Hkv, d, ps, refcnt=None):
    """In-place compaction on copies -> (table, seq_lens, k_pool, v_pool, free_list, free_top, rc);
    with refcnt (shared pages) the updated counts are written back into that array."""
    table = _c(table, np.int32).copy()
    seq_lens = _c(seq_lens, np.int32).copy()
    keep = _c(keep, np.uint8)
    k_pool = _c(k_pool, np.uint16).copy()
    v_pool = _c(v_pool, np.uint16).copy()
    free_list = _c(free_list, np.int32).copy()
    top = np.array([free_top], dtype=np.int32)
    B, maxp = table.shape
    if refcnt is not None:
        assert refcnt.dtype == np.int32 and refcnt.flags.c_contiguous
    rc = lib().or_compact(_p(table), maxp, _p(seq_lens), _p(keep), int(token_granular),
                          _p(k_pool), _p(v_pool), k_pool.shape[0], _p(free_list), _p(top),
                          _p(refcnt), B, Hkv, d, ps)
    return table, seq_lens, k_pool, v_pool, free_list, int(top[0]), rc


def append(k_new, v_new, k_pool, v_pool, table, seq_lens, free_list, free_top, Hkv, d, ps,
           refcnt=None):
    """-> (k_pool, v_pool, table, seq_lens, free_list, free_top, rc), all copies; with refcnt
    (shared pages) the updated counts are written back into that array."""
    k_pool = _c(k_pool, np.uint16).copy()
    v_pool = _c(v_pool, np.uint16).copy()
    table = _c(table, np.int32).copy()
    seq_lens = _c(seq_lens, np.int32).copy()
    free_list = _c(free_list, np.int32).copy()
    top = np.array([free_top], dtype=np.int32)
    B, maxp = table.shape
    if refcnt is not None:
        assert refcnt.dtype == np.int32 and refcnt.flags.c_contiguous
    rc = lib().or_append(_p(_c(k_new, np.uint16)), _p(_c(v_new, np.uint16)), _p(k_pool),
                         _p(v_pool), k_pool.shape[0], _p(table), maxp, _p(seq_lens),
                         _p(free_list), _p(top), _p(refcnt), B, Hkv, d, ps)
    return k_pool, v_pool, table, seq_lens, free_list, int(top[0]), rc


def mark_active(seq_lens, budget, ps, mode):
    seq_lens = _c(seq_lens, np.int32)
    budget = _c(budget, np.int32)
    act = np.zeros(len(seq_lens), dtype=np.uint8)
    _check(lib().or_mark_active(_p(seq_lens), _p(budget), len(seq_lens), ps, int(mode), _p(act)))
    return act


class using:
    """Temporarily route every wrapper above to another build of the oracle
    (used by the tests that plant a mistake in a copy of oracle.c and check
    that the pins catch it)."""

    def __init__(self, so_path: str):
        self.path = so_path

    def __enter__(self):
        global _lib
        with _lock:
            self.saved = _lib
            L = C.CDLL(self.path)
            _declare(L)
            _lib = L
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def build_variant(src_text: str, out_path: str) -> str:
    """Compile a modified copy of oracle.c (for mutation tests)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-w", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-o", out_path, src, "-lm", "-lpthread"])
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def compact_inplace(table, seq_lens, keep, token_granular, k_pool, v_pool, free_list, free_top_arr,
                    Hkv, d, ps, refcnt=None):
    """or_compact on the caller's arrays (all C-contiguous, right dtypes);
    free_top_arr is a 1-element int32 array.  Returns the status."""
    for a, dt in ((table, np.int32), (seq_lens, np.int32), (keep, np.uint8), (k_pool, np.uint16),
                  (v_pool, np.uint16), (free_list, np.int32), (free_top_arr, np.int32)):
        assert a.dtype == dt and a.flags.c_contiguous
    B, maxp = table.shape
    return lib().or_compact(_p(table), maxp, _p(seq_lens), _p(keep), int(token_granular),
                            _p(k_pool), _p(v_pool), k_pool.shape[0], _p(free_list),
                            _p(free_top_arr), _p(refcnt), B, Hkv, d, ps)


def append_inplace(k_new, v_new, k_pool, v_pool, table, seq_lens, free_list, free_top_arr,
                   Hkv, d, ps, refcnt=None):
    """or_append on the caller's arrays.  Returns the status."""
    for a, dt in ((table, np.int32), (seq_lens, np.int32), (k_pool, np.uint16),
                  (v_pool, np.uint16), (free_list, np.int32), (free_top_arr, np.int32)):
        assert a.dtype == dt and a.flags.c_contiguous
    B, maxp = table.shape
    return lib().or_append(_p(_c(k_new, np.uint16)), _p(_c(v_new, np.uint16)), _p(k_pool),
                           _p(v_pool), k_pool.shape[0], _p(table), maxp, _p(seq_lens),
                           _p(free_list), _p(free_top_arr), _p(refcnt), B, Hkv, d, ps)
