"""GPU parity of the tensor-core decode engine (kv_decode with
pages_per_split = KV_DECODE_TENSOR_CORE) against the oracle, and its place
beside the fused decode kernel: one workspace shared by both engines, the
host-buffer entry point, calibration among engines, device-side errors."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_kv_cache_492_b300 import kv
from paged_kv_cache_492_b300 import workloads as W
from tests.gpu_util import DeviceDecode, assert_decode_close, bits_to_dev, i32

pytestmark = pytest.mark.gpu
NCPU = len(os.sched_getaffinity(0))
TC = kv.KV_DECODE_TENSOR_CORE

SMALL = [
    # seed, B, Hq, Hkv, d, lens, dtype
    (41, 1, 4, 1, 128, [256], W.F16),                          # Hkv = 1: one-warp head block
    (42, 3, 8, 2, 128, [1, 15, 16], W.F16),                    # partial / exact pages
    (43, 4, 32, 8, 128, [17, 0, 300, 1000], W.F16),            # empty row
    (44, 4, 32, 8, 128, [17, 0, 300, 1000], W.BF16),
    (45, 2, 8, 8, 128, [33, 70], W.F16),                       # G = 1
    (46, 2, 64, 8, 128, [99, 513], W.BF16),                    # G = 8
    (47, 2, 96, 6, 128, [700, 20], W.F16),                     # G = 16, head block 6
    (48, 3, 48, 12, 128, [640, 48, 2000], W.BF16),             # 12 heads: two blocks of 6
    (49, 5, 16, 16, 128, [0, 0, 64, 0, 31], W.F16),            # two blocks of 8, mostly empty
    (50, 8, 32, 8, 128, [4000, 16, 17, 2048, 0, 1, 777, 3000], W.BF16),
    (51, 1, 32, 8, 128, [20000], W.F16),                       # one sequence over every chunk
    (60, 3, 64, 2, 128, [900, 0, 2500], W.BF16),               # G = 32: two row blocks
    (61, 2, 128, 2, 128, [3000, 77], W.F16),                   # G = 64: four row blocks
    (65, 3, 12, 3, 128, [500, 1700, 16], W.BF16),              # head block 3, 8-stage ring
    (66, 2, 20, 5, 128, [2300, 64], W.F16),                    # head block 5, 4-stage ring
    (67, 2, 56, 7, 128, [1000, 999], W.BF16),                  # head block 7, 3-stage ring
    (68, 2, 48, 1, 128, [1800, 33], W.F16),                    # Hkv = 1, G = 48: three row blocks
    # d = 64: one 64-channel half per head row, twice the ring stages
    (70, 1, 4, 1, 64, [256], W.F16),                           # the tiny workload's shape
    (71, 3, 8, 2, 64, [1, 15, 700], W.F16),
    (72, 4, 32, 8, 64, [17, 0, 300, 5000], W.BF16),
    (73, 2, 64, 4, 64, [2000, 33], W.F16),                     # G = 16
    (74, 2, 128, 2, 64, [1500, 40], W.BF16),                   # G = 64: four row blocks
]


def _ws(x, pps=TC):
    return kv.alloc_workspace(kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages, 16,
                                                          pps))


@pytest.mark.parametrize("case", SMALL, ids=[f"s{c[0]}" for c in SMALL])
def test_engine_small(case):
    seed, B, Hq, Hkv, d, lens, dtype = case
    x = W.small_decode(seed, B, Hq, Hkv, d, lens, dtype=dtype, pad_pages=1)
    out, lse, rc = DeviceDecode(x).run(pages_per_split=TC, ws=_ws(x))
    assert rc == kv.KV_OK
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    assert_decode_close(x, out, lse, ref_out, ref_lse)


FULL = {
    "bimodal": W.bimodal,
    "bimodal_b4": W.bimodal_b4,
    "uniform": W.uniform_lengths,
    "zipf": W.zipf_lengths,
    "bucket128k": lambda: W.bucketed_long(131072),
    "budgeted_b64": lambda: W.budgeted_serving()["decode"],
    "tiny": lambda: W.tiny()["decode"],
}


@pytest.mark.parametrize("name", list(FULL))
def test_engine_full_config(name):
    """Every (sequence, query head) of the full-size workload against the oracle."""
    x = FULL[name]()
    out, lse, rc = DeviceDecode(x).run(pages_per_split=TC, ws=_ws(x))
    assert rc == kv.KV_OK
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    worst = assert_decode_close(x, out, lse, ref_out, ref_lse)
    print(f"{name}: worst |out-oracle|/max|V| = {worst:.2e}")


def test_large_batch_offsets_pass():
    """Above 1024 sequences the page offsets come from a separate pass."""
    rng = np.random.default_rng(52)
    lens = rng.integers(0, 100, size=1300).astype(np.int32)
    lens[::7] = 0
    x = W.small_decode(52, 1300, 16, 4, 128, lens.tolist(), pool_factor=1.2)
    out, lse, rc = DeviceDecode(x).run(pages_per_split=TC, ws=_ws(x))
    assert rc == 0
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    assert_decode_close(x, out, lse, ref_out, ref_lse)


def test_engines_share_a_workspace():
    """The tensor-core engine's scratch lies past the fused kernel's merge
    tickets for every split size: alternating engines on one workspace keeps
    every call clean, each engine repeats itself bit for bit, and the two
    agree within the tolerance."""
    x = W.small_decode(53, 6, 32, 8, 128, [3000, 40, 0, 1500, 17, 900])
    dd = DeviceDecode(x)
    ws = kv.alloc_workspace(max(kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages, 16, 1),
                                kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages, 16, TC)))
    runs = {}
    for pps in (0, TC, 1, TC, 8, 0, TC, 1):
        out, lse, rc = dd.run(pages_per_split=pps, ws=ws)
        assert rc == 0, pps
        if pps in runs:
            assert np.array_equal(out, runs[pps][0]) and np.array_equal(lse, runs[pps][1]), pps
        runs[pps] = (out, lse)
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    for out, lse in runs.values():
        assert_decode_close(x, out, lse, ref_out, ref_lse)


def test_attend_multi_t1_is_the_engine():
    """kv_attend_multi with one query token runs the same tensor-core engine."""
    x = W.small_decode(54, 3, 32, 8, 128, [700, 33, 2100])
    o1, l1, rc = DeviceDecode(x).run(pages_per_split=TC, ws=_ws(x))
    assert rc == 0
    dd = DeviceDecode(x)
    out = torch.empty((x.B, 1, x.Hq, x.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((x.B, 1, x.Hq), dtype=torch.float32, device="cuda")
    ws = kv.alloc_workspace(kv.kv_attend_multi_workspace_size(x.B, 1, x.Hq, x.Hkv, x.d,
                                                              x.max_pages))
    kv.kv_attend_multi(dd.q.view(x.B, 1, x.Hq, x.d), dd.k, dd.v, dd.table, dd.lens, x.scale, out,
                       lse, ws)
    assert kv.kv_get_status(ws) == 0
    assert np.array_equal(out[:, 0].cpu().numpy(), o1.astype(np.float32))
    assert np.array_equal(lse[:, 0].cpu().numpy(), l1.astype(np.float32))


def test_hostio_engine_matches_device_call():
    x = W.small_decode(55, 4, 32, 8, 128, [1200, 0, 35, 5000], dtype=W.BF16)
    o_dev, l_dev, rc = DeviceDecode(x).run(pages_per_split=TC, ws=_ws(x))
    assert rc == 0
    dd = DeviceDecode(x)
    hq = torch.from_numpy(x.q.view(np.int16).copy()).view(dd.q.dtype).pin_memory()
    ht = torch.from_numpy(x.block_table.copy()).pin_memory()
    hl = torch.from_numpy(x.seq_lens.copy()).pin_memory()
    ho = torch.empty((x.B, x.Hq, x.d), dtype=torch.float32).pin_memory()
    hls = torch.empty((x.B, x.Hq), dtype=torch.float32).pin_memory()
    ws = kv.alloc_workspace(kv.kv_decode_hostio_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages,
                                                               16, TC))
    call = kv.prepare_decode_hostio(hq, dd.k, dd.v, ht, hl, x.scale, ho, hls, ws,
                                    pages_per_split=TC)
    assert call() == 0
    torch.cuda.synchronize()
    assert kv.kv_get_status(ws) == 0
    assert np.array_equal(ho.numpy(), o_dev.astype(np.float32))
    assert np.array_equal(hls.numpy(), l_dev.astype(np.float32))


def test_hostio_pageable_buffers():
    """Pinned host buffers go through copy kernels on mapped memory, pageable
    ones through per-buffer copies: both give the device call's result."""
    x = W.small_decode(62, 3, 32, 8, 128, [900, 0, 2500])
    o_dev, l_dev, rc = DeviceDecode(x).run(pages_per_split=TC, ws=_ws(x))
    assert rc == 0
    dd = DeviceDecode(x)
    for pinned in (False, True):
        mk = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
        hq = mk(torch.from_numpy(x.q.view(np.int16).copy()).view(dd.q.dtype))
        ht = mk(torch.from_numpy(x.block_table.copy()))
        hl = mk(torch.from_numpy(x.seq_lens.copy()))
        ho = mk(torch.full((x.B, x.Hq, x.d), float("nan"), dtype=torch.float32))
        hls = mk(torch.full((x.B, x.Hq), float("nan"), dtype=torch.float32))
        ws = kv.alloc_workspace(kv.kv_decode_hostio_workspace_size(x.B, x.Hq, x.Hkv, x.d,
                                                                   x.max_pages, 16, TC))
        call = kv.prepare_decode_hostio(hq, dd.k, dd.v, ht, hl, x.scale, ho, hls, ws,
                                        pages_per_split=TC)
        assert call() == 0
        torch.cuda.synchronize()
        assert kv.kv_get_status(ws) == 0
        assert np.array_equal(ho.numpy(), o_dev.astype(np.float32)), pinned
        assert np.array_equal(hls.numpy(), l_dev.astype(np.float32)), pinned


def test_tune_and_policy_include_the_engine():
    x = W.bimodal_b4()
    dd = DeviceDecode(x)
    cands = [0, 32, TC]
    pol = kv.DecodePolicy(candidates=cands, reps=3)
    ws = kv.alloc_workspace(pol.workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages))
    best, us = kv.kv_decode_tune(dd.q, dd.k, dd.v, dd.table, dd.lens, x.scale, dd.out, dd.lse, ws,
                                 cands, reps=3)
    assert best in cands and len(us) == 3 and all(u > 0 for u in us)
    assert us[cands.index(best)] == min(us)
    # timed with L2 flushed before every call, as the bench times a step
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    best_f, us_f = kv.kv_decode_tune(dd.q, dd.k, dd.v, dd.table, dd.lens, x.scale, dd.out, dd.lse,
                                     ws, cands, reps=3, flush=flush)
    assert best_f in cands and us_f[cands.index(best_f)] == min(us_f)
    out, lse, rc = dd.run(pages_per_split=best, ws=ws)
    assert rc == 0
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    assert_decode_close(x, out, lse, ref_out, ref_lse)
    p1 = pol.pages_per_split(x.seq_lens, dd.q, dd.k, dd.v, dd.table, dd.lens, x.scale, dd.out,
                             dd.lse, ws)
    p2 = pol.pages_per_split(x.seq_lens, dd.q, dd.k, dd.v, dd.table, dd.lens, x.scale, dd.out,
                             dd.lse, ws)
    assert p1 == p2 and p1 in cands and len(pol.table) == 1
    print(f"B4 bimodal engines {dict(zip(cands, [round(u, 1) for u in us]))} us; best {best}")


def test_engine_device_errors():
    x = W.small_decode(56, 2, 16, 4, 128, [40, 40])
    x.block_table = x.block_table.copy()
    x.block_table[1, 2] = x.num_pages + 5
    _, _, rc = DeviceDecode(x).run(pages_per_split=TC, ws=_ws(x))
    assert rc == kv.KV_EBADPAGE
    x.block_table[1, 2] = -1
    _, _, rc = DeviceDecode(x).run(pages_per_split=TC, ws=_ws(x))
    assert rc == kv.KV_EBADPAGE
    x = W.small_decode(57, 2, 16, 4, 128, [40, 40])
    dd = DeviceDecode(x)
    ws = _ws(x)
    dd.lens.copy_(i32([40, -3]))
    out, lse, rc = dd.run(pages_per_split=TC, ws=ws)
    assert rc == kv.KV_EINVAL
    assert np.all(out[1] == 0) and np.all(lse[1] == -math.inf)
    dd.lens.copy_(i32([16 * x.max_pages + 1, 40]))
    out, lse, rc = dd.run(pages_per_split=TC, ws=ws)
    assert rc == kv.KV_EINVAL and np.all(out[0] == 0)


def test_engine_keeps_no_state_between_calls():
    """The tensor-core engine rewrites all of its scratch (page offsets,
    partials) on every call and keeps no counters between calls: a workspace
    full of leftovers gives the same result as a clean one, call after call."""
    x = W.small_decode(62, 3, 32, 8, 128, [20000, 900, 0])
    dd = DeviceDecode(x)
    ws = _ws(x)
    ws[256:].fill_(1)
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    first = None
    for _ in range(3):
        out, lse, rc = dd.run(pages_per_split=TC, ws=ws)
        assert rc == 0
        assert_decode_close(x, out, lse, ref_out, ref_lse)
        if first is None:
            first = (out, lse)
        assert np.array_equal(out, first[0]) and np.array_equal(lse, first[1])


def test_engine_argument_checks():
    # d = 96 and groups above 64 have no tensor-core form
    assert kv.kv_decode_workspace_size(2, 8, 2, 96, 4, 16, TC) == 0
    assert kv.kv_decode_workspace_size(2, 256, 2, 128, 4, 16, TC) == 0
    assert kv.kv_decode_workspace_size(2, 8, 2, 128, 4, 16, -2) == 0
    assert kv.kv_decode_workspace_size(2, 8, 2, 64, 4, 16, TC) > 0
    x = W.small_decode(58, 1, 8, 2, 96, [40])
    dd = DeviceDecode(x)
    ws = kv.alloc_workspace(1 << 20)
    with pytest.raises(kv.KVError) as e:
        dd.run(pages_per_split=TC, ws=ws)
    assert e.value.code == kv.KV_EINVAL
    x = W.small_decode(59, 2, 16, 4, 128, [400, 40])
    dd = DeviceDecode(x)
    small = kv.alloc_workspace(kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages, 16,
                                                           0))
    with pytest.raises(kv.KVError) as e:
        dd.run(pages_per_split=TC, ws=small)
    assert e.value.code == kv.KV_EWORKSPACE
    # the no-allocation entry point has no tensor-core form
    with pytest.raises(kv.KVError) as e:
        kv.kv_decode_noalloc(dd.q, dd.k, dd.v, dd.table, dd.lens, x.scale, dd.out, dd.lse,
                             torch.zeros(1, dtype=torch.int32, device="cuda"), pages_per_split=TC)
    assert e.value.code == kv.KV_EINVAL
