"""kv_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a host framework that owns every allocation, or a
plugin interface that forbids allocating on the hot path).  It keeps its
scratch in the library's fixed device array instead of a caller workspace.
Checked through the C ABI against kv_decode on the same inputs and against
the oracle, on two calls in a row, within the decode tolerance the other
tests use; also a batch above 1024 sequences (page offsets kept in the
array) and an empty batch.  Kept in a file that pytest collects last."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_kv_cache_492_b300 import kv
from paged_kv_cache_492_b300 import workloads as W
from tests.gpu_util import DeviceDecode, assert_decode_close, i32, vmax_per_seq

NCPU = len(os.sched_getaffinity(0))

pytestmark = pytest.mark.gpu


def _close(x, out, lse, ref_out, ref_lse):
    vmax = vmax_per_seq(x)
    for b in range(x.B):
        if x.seq_lens[b] == 0:
            assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
            assert np.all(ref_out[b] == 0) and np.all(np.isneginf(ref_lse[b]))
            continue
        assert np.abs(out[b] - ref_out[b]).max() <= 2e-3 * vmax[b], b
        assert np.abs(lse[b] - ref_lse[b]).max() <= 1e-3, b


def _noalloc(dd, pps):
    x = dd.x
    out = torch.full((x.B, x.Hq, x.d), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((x.B, x.Hq), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    L = kv.lib()
    rc = L.kv_decode_noalloc(dd.q.data_ptr(), dd.k.data_ptr(), dd.v.data_ptr(), x.num_pages,
                             dd.table.data_ptr(), x.max_pages, dd.lens.data_ptr(), x.B, 16, x.Hq,
                             x.Hkv, x.d, x.dtype, float(x.scale), pps, out.data_ptr(),
                             lse.data_ptr(), status.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    assert rc == kv.KV_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def test_noalloc_matches_decode_two_calls():
    x = W.small_decode(41, 6, 32, 8, 128, [3000, 0, 17, 900, 2500, 64], dtype=W.BF16)
    dd = DeviceDecode(x)
    # call 1: automatic split (long sequences merge many splits)
    ref_out, ref_lse, rc = dd.run()
    assert rc == 0
    out, lse = _noalloc(dd, 0)
    _close(x, out, lse, ref_out, ref_lse)
    o64, l64 = O.decode(x, nthreads=NCPU)
    assert_decode_close(x, out, lse, o64, l64)
    # call 2, right after: other lengths and another split size, so the
    # scratch left by call 1 must not leak into it
    lens = np.array([1200, 0, 5, 899, 2048, 63], np.int32)  # within each row's pages
    dd.lens.copy_(i32(lens))
    x2 = W.DecodeInputs(**{**x.__dict__, "seq_lens": lens})
    dd.x = x2
    ref_out, ref_lse, rc = dd.run(pages_per_split=3)
    assert rc == 0
    out, lse = _noalloc(dd, 3)
    _close(x2, out, lse, ref_out, ref_lse)
    o64, l64 = O.decode(x2, nthreads=NCPU)
    assert_decode_close(x2, out, lse, o64, l64)


def test_noalloc_large_batch_and_empty():
    """Above 1024 sequences the page offsets come from a separate pass and
    live in the fixed array too; two calls in a row against kv_decode and the
    oracle.  An empty batch only zeroes the status word."""
    rng = np.random.default_rng(43)
    lens = rng.integers(0, 70, size=1100).astype(np.int32)
    lens[::13] = 0
    x = W.small_decode(43, 1100, 8, 2, 128, lens.tolist(), dtype=W.F16)
    dd = DeviceDecode(x)
    for pps in (0, 3):
        ref_out, ref_lse, rc = dd.run(pages_per_split=pps)
        assert rc == 0
        out, lse = _noalloc(dd, pps)
        _close(x, out, lse, ref_out, ref_lse)
        o64, l64 = O.decode(x, nthreads=NCPU)
        assert_decode_close(x, out, lse, o64, l64)
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    rc = kv.lib().kv_decode_noalloc(dd.q.data_ptr(), dd.k.data_ptr(), dd.v.data_ptr(),
                                    x.num_pages, dd.table.data_ptr(), x.max_pages,
                                    dd.lens.data_ptr(), 0, 16, x.Hq, x.Hkv, x.d, x.dtype,
                                    float(x.scale), 0, dd.out.data_ptr(), dd.lse.data_ptr(),
                                    status.data_ptr(), None)
    assert rc == kv.KV_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_noalloc_rejects_oversized_scratch():
    """A batch whose scratch exceeds the fixed array is refused, nothing runs."""
    x = W.small_decode(42, 2, 32, 8, 128, [16, 16])
    dd = DeviceDecode(x)
    out = torch.zeros((x.B, x.Hq, x.d), dtype=torch.float32, device="cuda")
    lse = torch.zeros((x.B, x.Hq), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    big_pages = 1 << 16   # one page per split over 2 x 65536-page rows: far beyond 16 MiB
    table = torch.zeros((x.B, big_pages), dtype=torch.int32, device="cuda")
    rc = kv.lib().kv_decode_noalloc(dd.q.data_ptr(), dd.k.data_ptr(), dd.v.data_ptr(),
                                    x.num_pages, table.data_ptr(), big_pages, dd.lens.data_ptr(),
                                    x.B, 16, x.Hq, x.Hkv, x.d, x.dtype, float(x.scale), 1,
                                    out.data_ptr(), lse.data_ptr(), status.data_ptr(), None)
    assert rc == kv.KV_EWORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 0) and not math.isnan(float(lse.sum()))
