"""GPU parity of multi-token query attention (kv_attend_multi): T new query
tokens per sequence, the last T of its cached tokens, each attending
causally, over the same pool and block table as decode."""
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_kv_cache_492_b300 import kv
from paged_kv_cache_492_b300 import workloads as W
from tests.gpu_util import DeviceDecode, bits_to_dev, vmax_per_seq

pytestmark = pytest.mark.gpu
NCPU = len(os.sched_getaffinity(0))


def _run(x, qm, T, pps=0):
    dd = DeviceDecode(x)
    q = bits_to_dev(qm, x.dtype)
    out = torch.full((x.B, T, x.Hq, x.d), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((x.B, T, x.Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = kv.alloc_workspace(kv.kv_attend_multi_workspace_size(x.B, T, x.Hq, x.Hkv, x.d,
                                                              x.max_pages, 16, pps))
    kv.kv_attend_multi(q, dd.k, dd.v, dd.table, dd.lens, x.scale, out, lse, ws,
                       pages_per_split=pps)
    assert kv.kv_get_status(ws) == 0
    return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _check(x, T, out, lse, ref_out, ref_lse):
    vmax = vmax_per_seq(x)
    for b in range(x.B):
        for i in range(T):
            if int(x.seq_lens[b]) - T + 1 + i <= 0:
                assert np.all(out[b, i] == 0) and np.all(np.isneginf(lse[b, i])), (b, i)
                continue
            assert np.abs(out[b, i] - ref_out[b, i]).max() <= 2e-3 * vmax[b], (b, i)
            assert np.abs(lse[b, i] - ref_lse[b, i]).max() <= 1e-3, (b, i)


# d = 128 runs on the tensor-core kernel (one consumer warp per 16 rows), in
# the fewest passes of at most 64 / G tokens where T * G > 64.
@pytest.mark.parametrize("T,dtype,G,lens,pps", [
    (4, W.F16, 4, [3000, 17, 0, 2, 900], 0),
    (4, W.BF16, 4, [2500, 3, 0, 16, 48, 4100], 0),
    (2, W.BF16, 4, [1, 16, 33, 5000], 3),
    (8, W.F16, 2, [100, 7, 1200], 0),
    (16, W.BF16, 1, [16, 15, 17, 700], 0),
    (1, W.BF16, 8, [640, 12], 0),
    (1, W.F16, 16, [900, 31], 0),
    (3, W.F16, 4, [2000, 5], 0),
    (8, W.F16, 4, [1000, 3, 40], 0),            # 32 rows: two row blocks
    (2, W.F16, 8, [5000], 1),
    (5, W.F16, 4, [1500, 4, 0, 333], 0),        # 20 rows: a partial second block
    (16, W.F16, 4, [2100, 9, 700], 0),          # 64 rows: four row blocks
    (8, W.BF16, 8, [1800, 30], 5),              # 64 rows, bf16, fixed splits
    (12, W.BF16, 2, [64, 2000], 0),             # 24 rows
    (12, W.F16, 4, [900, 11, 2600], 0),         # 48 rows: three row blocks
    (16, W.F16, 8, [1200, 20], 0),              # 128 rows: two passes of 8 tokens
    (20, W.F16, 4, [1500, 7, 0, 300], 0),       # 80 rows: passes of 12 + 8 tokens
    (33, W.BF16, 2, [900, 40, 2, 33], 0),       # 66 rows: 24 + 9 tokens; L < T rows
    (70, W.F16, 1, [500, 69, 71, 64], 0),       # G = 1: 48 + 22 tokens
    (24, W.BF16, 8, [2000, 10, 25], 3),         # 192 rows: three passes, fixed splits
    (40, W.F16, 4, [4000, 1, 39, 41], 1),       # 160 rows, one-page splits
    (1, W.F16, 4, [20000, 40, 0], 1),           # 1250 one-page splits: groups of 36
    (4, W.BF16, 4, [17000, 3], 2),              # 532 splits x 16 rows: groups of 24
])
def test_attend_multi_small(T, dtype, G, lens, pps):
    rng = np.random.default_rng(T * 10 + G)
    Hkv = 8 if G * 8 <= 64 else 2
    x = W.small_decode(90 + T, len(lens), Hkv * G, Hkv, 128, lens, dtype=dtype, pad_pages=1)
    qm = W.normal_bits(rng, (x.B, T, x.Hq, x.d), dtype)
    out, lse = _run(x, qm, T, pps)
    ref_out, ref_lse = O.attend_multi(x, qm, nthreads=NCPU)
    _check(x, T, out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("T,dtype,G,lens", [
    (4, W.F16, 4, [900, 3, 0, 2000]),           # 16 rows: one pass
    (16, W.BF16, 4, [1500, 20, 700]),           # 64 rows: one pass, four row blocks
    (20, W.F16, 4, [1200, 7, 300]),             # 80 rows: passes of 12 + 8 tokens
    (3, W.BF16, 8, [640, 2]),
])
def test_attend_multi_d64(T, dtype, G, lens):
    """d = 64 on the tensor-core kernel (one 64-channel half per head row)."""
    rng = np.random.default_rng(T * 7 + G)
    Hkv = 4
    x = W.small_decode(190 + T, len(lens), Hkv * G, Hkv, 64, lens, dtype=dtype, pad_pages=1)
    qm = W.normal_bits(rng, (x.B, T, x.Hq, x.d), dtype)
    out, lse = _run(x, qm, T)
    ref_out, ref_lse = O.attend_multi(x, qm, nthreads=NCPU)
    _check(x, T, out, lse, ref_out, ref_lse)


def test_attend_multi_bimodal_t4():
    """Four query tokens per sequence on the batch-8 bimodal fp16 workload."""
    x = W.bimodal()
    rng = np.random.default_rng(4)
    qm = W.normal_bits(rng, (x.B, 4, x.Hq, x.d), x.dtype)
    out, lse = _run(x, qm, 4)
    ref_out, ref_lse = O.attend_multi(x, qm, nthreads=NCPU)
    _check(x, 4, out, lse, ref_out, ref_lse)


def test_attend_multi_t1_matches_decode():
    """One query token: the tensor-core engine against the fused decode kernel
    and the oracle."""
    x = W.small_decode(97, 3, 32, 8, 128, [700, 33, 2100])
    out, lse = _run(x, x.q[:, None], 1)
    o, l, rc = DeviceDecode(x).run()
    assert rc == 0
    vmax = vmax_per_seq(x)
    for b in range(x.B):
        assert np.abs(out[b, 0] - o[b]).max() <= 2e-3 * vmax[b]
        assert np.abs(lse[b, 0] - l[b]).max() <= 1e-3
    ref_out, ref_lse = O.attend_multi(x, x.q[:, None], nthreads=NCPU)
    _check(x, 1, out, lse, ref_out, ref_lse)


def _rows_of(x, rows):
    """The batch restricted to `rows` (same pools), for oracle samples."""
    rows = np.asarray(rows)
    return W.DecodeInputs(**{**x.__dict__, "B": len(rows), "q": x.q[rows],
                             "block_table": np.ascontiguousarray(x.block_table[rows]),
                             "seq_lens": np.ascontiguousarray(x.seq_lens[rows])})


def test_attend_multi_large_batch_passes():
    """Above 1024 sequences the page offsets come from a separate pass, which
    takes each pass's shortened lengths: 1100 sequences, T = 20 (80 rows per
    KV head: passes of 12 + 8 tokens), lengths from 0 to 60 (many below T)."""
    rng = np.random.default_rng(61)
    lens = rng.integers(0, 61, size=1100).astype(np.int32)
    x = W.small_decode(61, 1100, 32, 8, 128, lens.tolist(), dtype=W.F16)
    T = 20
    qm = W.normal_bits(rng, (x.B, T, x.Hq, x.d), x.dtype)
    out, lse = _run(x, qm, T)
    ref_out, ref_lse = O.attend_multi(x, qm, nthreads=NCPU)
    _check(x, T, out, lse, ref_out, ref_lse)


def test_attend_multi_bimodal_t32_sampled():
    """32 query tokens per sequence on the batch-8 bimodal fp16 workload (128
    rows per KV head: two passes of 16 tokens), checked against the oracle on
    three of the sequences (a long one, a short one, and the longest)."""
    x = W.bimodal()
    T = 32
    rng = np.random.default_rng(32)
    qm = W.normal_bits(rng, (x.B, T, x.Hq, x.d), x.dtype)
    out, lse = _run(x, qm, T)
    rows = [int(np.argmax(x.seq_lens)), int(np.argmin(x.seq_lens)), 1]
    y = _rows_of(x, rows)
    ref_out, ref_lse = O.attend_multi(y, qm[rows], nthreads=NCPU)
    _check(y, T, out[rows], lse[rows], ref_out, ref_lse)
