"""GPU parity: kv_decode and the workqueue builder against the oracle."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_kv_cache_492_b300 import kv
from paged_kv_cache_492_b300 import workloads as W
from tests.gpu_util import DeviceDecode, assert_decode_close, i32

pytestmark = pytest.mark.gpu
NCPU = len(os.sched_getaffinity(0))

SMALL = [
    # seed, B, Hq, Hkv, d, lens, dtype, pages_per_split
    (1, 1, 4, 1, 64, [256], W.F16, 0),
    (2, 3, 8, 2, 128, [1, 15, 16], W.F16, 0),
    (3, 4, 32, 8, 128, [17, 0, 300, 1000], W.F16, 0),
    (4, 4, 32, 8, 128, [17, 0, 300, 1000], W.BF16, 3),
    (5, 2, 8, 8, 128, [33, 70], W.F16, 1),       # G = 1
    (6, 2, 16, 8, 64, [200, 5], W.BF16, 2),      # G = 2
    (7, 2, 64, 8, 128, [99, 513], W.F16, 5),     # G = 8
    (8, 5, 8, 1, 64, [0, 0, 64, 0, 31], W.F16, 0),
    (9, 8, 32, 8, 128, [4000, 16, 17, 2048, 0, 1, 777, 3000], W.BF16, 0),
    (10, 1, 32, 8, 128, [20000], W.F16, 0),
]


@pytest.mark.parametrize("case", SMALL, ids=[f"s{c[0]}" for c in SMALL])
def test_decode_small(case):
    seed, B, Hq, Hkv, d, lens, dt, pps = case
    x = W.small_decode(seed, B, Hq, Hkv, d, lens, dtype=dt, pad_pages=2)
    out, lse, rc = DeviceDecode(x).run(pages_per_split=pps)
    assert rc == kv.KV_OK
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    assert_decode_close(x, out, lse, ref_out, ref_lse)


def test_split_sizes_agree():
    """Any split size gives the oracle's result (and the same to fp32 noise)."""
    x = W.small_decode(21, 3, 32, 8, 128, [1500, 40, 900])
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    dd = DeviceDecode(x)
    for pps in (0, 1, 2, 7, 64, 1000):
        out, lse, rc = dd.run(pages_per_split=pps)
        assert rc == 0
        assert_decode_close(x, out, lse, ref_out, ref_lse)


def test_deterministic():
    x = W.small_decode(22, 4, 32, 8, 128, [3000, 100, 0, 50])
    dd = DeviceDecode(x)
    o1, l1, _ = dd.run()
    o2, l2, _ = dd.run()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_workspace_reused_across_calls():
    """One decode workspace serves many calls (its merge tickets return to
    zero after each); lengths, split sizes and batch contents change."""
    x = W.small_decode(27, 6, 32, 8, 128, [2000, 3, 0, 700, 1500, 64])
    dd = DeviceDecode(x)
    ws = kv.alloc_workspace(kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages, 16, 1))
    rng = np.random.default_rng(5)
    for it in range(6):
        lens = x.seq_lens.copy()
        if it % 2:
            lens = np.array([int(rng.integers(0, L + 1)) for L in x.seq_lens], np.int32)
        y = W.DecodeInputs(**{**x.__dict__, "seq_lens": lens})
        dd.lens.copy_(i32(lens))
        out, lse, rc = dd.run(pages_per_split=(0, 1, 3)[it % 3], ws=ws)
        assert rc == 0
        ref_out, ref_lse = O.decode(y, nthreads=NCPU)
        assert_decode_close(y, out, lse, ref_out, ref_lse)


def test_dirty_workspace_reported():
    """A decode workspace whose merge tickets were not zeroed is reported."""
    x = W.small_decode(28, 2, 8, 2, 64, [900, 500])
    dd = DeviceDecode(x)
    ws = kv.alloc_workspace(kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages, 16, 4))
    ws[256:].fill_(1)
    _, _, rc = dd.run(pages_per_split=4, ws=ws)
    assert rc == kv.KV_EWORKSPACE
    kv.kv_workspace_reset(ws)
    out, lse, rc = dd.run(pages_per_split=4, ws=ws)
    assert rc == 0
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    assert_decode_close(x, out, lse, ref_out, ref_lse)


def test_large_batch_offsets_pass():
    """Batches above 1024 sequences take their page offsets from a separate
    pass; ragged short lengths, empty rows and splits across sequences."""
    rng = np.random.default_rng(29)
    lens = rng.integers(0, 100, size=1500).astype(np.int32)
    lens[::11] = 0
    x = W.small_decode(29, 1500, 8, 2, 64, lens.tolist(), pool_factor=1.2)
    dd = DeviceDecode(x)
    for pps in (0, 3):
        out, lse, rc = dd.run(pages_per_split=pps)
        assert rc == 0
        ref_out, ref_lse = O.decode(x, nthreads=NCPU)
        assert_decode_close(x, out, lse, ref_out, ref_lse)


def test_bad_page_reported():
    x = W.small_decode(23, 2, 8, 2, 64, [40, 40])
    x.block_table = x.block_table.copy()
    x.block_table[1, 2] = -1
    _, _, rc = DeviceDecode(x).run()
    assert rc == kv.KV_EBADPAGE
    x.block_table[1, 2] = x.num_pages + 5
    _, _, rc = DeviceDecode(x).run()
    assert rc == kv.KV_EBADPAGE


def test_bad_lengths_reported():
    x = W.small_decode(24, 2, 8, 2, 64, [40, 40])
    dd = DeviceDecode(x)
    dd.lens.copy_(i32([40, -3]))
    out, lse, rc = dd.run()
    assert rc == kv.KV_EINVAL
    assert np.all(out[1] == 0) and np.all(lse[1] == -math.inf)
    dd.lens.copy_(i32([40, 16 * x.max_pages + 1]))
    _, _, rc = dd.run()
    assert rc == kv.KV_EINVAL


def test_host_argument_checks():
    x = W.small_decode(25, 1, 8, 2, 64, [40])
    dd = DeviceDecode(x)
    ws = kv.alloc_workspace(256)
    with pytest.raises(kv.KVError) as e:
        kv.kv_decode(dd.q, dd.k, dd.v, dd.table, dd.lens, x.scale, dd.out, dd.lse, ws)
    assert e.value.code == kv.KV_EWORKSPACE
    rc = kv.lib().kv_decode(dd.q.data_ptr(), dd.k.data_ptr(), dd.v.data_ptr(), x.num_pages,
                            dd.table.data_ptr(), x.max_pages, dd.lens.data_ptr(), 1, 8, 8, 2, 64,
                            0, 0.1, 0, dd.out.data_ptr(), dd.lse.data_ptr(), ws.data_ptr(),
                            ws.numel(), None)
    assert rc == kv.KV_EINVAL          # page size 8 is not supported
    rc = kv.lib().kv_decode(dd.q.data_ptr(), dd.k.data_ptr(), dd.v.data_ptr(), x.num_pages,
                            dd.table.data_ptr(), x.max_pages, dd.lens.data_ptr(), 1, 16, 6, 4, 64,
                            0, 0.1, 0, dd.out.data_ptr(), dd.lse.data_ptr(), ws.data_ptr(),
                            ws.numel(), None)
    assert rc == kv.KV_EINVAL          # Hq % Hkv != 0


def _wq_device(lens, Hkv, pps, n_workers, max_pages):
    B = len(lens)
    W_ = int(sum(-(-int(L) // 16) for L in lens))
    max_chunks = (-(-W_ // pps) if pps else n_workers) + 2
    max_tasks = Hkv * (B + max_chunks)
    tasks = torch.zeros((max_tasks, 8), dtype=torch.int32, device="cuda")
    cb = torch.zeros(max_chunks, dtype=torch.int32, device="cuda")
    sgb = torch.zeros(B, dtype=torch.int32, device="cuda")
    sns = torch.zeros(B, dtype=torch.int32, device="cuda")
    meta = torch.zeros(8, dtype=torch.int32, device="cuda")
    ws = kv.alloc_workspace(kv.kv_workqueue_workspace_size(B))
    kv.kv_build_workqueue(i32(lens), Hkv, 16, max_pages, pps, n_workers, tasks, cb, sgb, sns, meta, ws)
    assert kv.kv_get_status(ws) == 0
    m = meta.cpu().numpy()
    T, G, chunk, nch = int(m[0]), int(m[1]), int(m[2]), int(m[3])
    return dict(tasks=tasks[:T].cpu().numpy(), chunk_begin=cb[: nch + 1].cpu().numpy(),
                seq_group_begin=sgb.cpu().numpy(), seq_nsplit=sns.cpu().numpy(), T=T, groups=G,
                chunk=chunk, nchunks=nch)


WQ = [([256], 1, 0, 148), ([1, 15, 16, 17, 0, 33], 2, 3, 10), ([0, 0, 0], 8, 0, 148),
      ([5000, 0, 12, 10000], 8, 37, 148), ([32768 + 5], 8, 0, 148)]


@pytest.mark.parametrize("lens,Hkv,pps,nw", WQ)
def test_workqueue_bit_exact(lens, Hkv, pps, nw):
    rng = np.random.default_rng(0)
    maxp = max(1, max(-(-L // 16) for L in lens))
    got = _wq_device(lens, Hkv, pps, nw, maxp)
    W_ = int(sum(-(-int(L) // 16) for L in lens))
    chunk = pps if pps else O.chunk_auto(W_, nw, 8)
    ref = O.workqueue(lens, Hkv, 16, chunk)
    assert got["chunk"] == ref["chunk"] and got["nchunks"] == ref["nchunks"]
    for k in ("tasks", "chunk_begin", "seq_group_begin", "seq_nsplit"):
        assert np.array_equal(got[k], ref[k]), k
    # random batches
    for _ in range(5):
        lens2 = [int(v) for v in rng.integers(0, 3000, size=int(rng.integers(1, 40)))]
        got = _wq_device(lens2, 8, 0, 148, max(1, max(-(-L // 16) for L in lens2)))
        W2 = int(sum(-(-int(L) // 16) for L in lens2))
        ref = O.workqueue(lens2, 8, 16, O.chunk_auto(W2, 148, 8))
        for k in ("tasks", "chunk_begin", "seq_group_begin", "seq_nsplit"):
            assert np.array_equal(got[k], ref[k]), k


def test_hostio_matches_device_call():
    x = W.small_decode(26, 4, 32, 8, 128, [3000, 100, 0, 50])
    dd = DeviceDecode(x)
    out, lse, _ = dd.run()
    ws = kv.alloc_workspace(kv.kv_decode_hostio_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages))
    hq = torch.from_numpy(x.q.view(np.int16)).view(torch.float16).pin_memory()
    ht = torch.from_numpy(x.block_table).pin_memory()
    hl = torch.from_numpy(x.seq_lens).pin_memory()
    ho = torch.empty((x.B, x.Hq, x.d), dtype=torch.float32).pin_memory()
    hls = torch.empty((x.B, x.Hq), dtype=torch.float32).pin_memory()
    kv.kv_decode_hostio(hq, dd.k, dd.v, ht, hl, x.scale, ho, hls, ws)
    torch.cuda.synchronize()
    assert kv.kv_get_status(ws) == 0
    assert np.array_equal(ho.numpy(), out.astype(np.float32))
    assert np.array_equal(hls.numpy(), lse.astype(np.float32))


CONFIGS = {
    "tiny": lambda: W.tiny()["decode"],
    "bimodal": W.bimodal,
    "bimodal_b4": W.bimodal_b4,
    "uniform": W.uniform_lengths,
    "zipf": W.zipf_lengths,
    "bucket32k": lambda: W.bucketed_long(32768),
    "bucket64k": lambda: W.bucketed_long(65536),
    "bucket128k": lambda: W.bucketed_long(131072),
}


@pytest.mark.parametrize("name", list(CONFIGS))
def test_decode_full_config(name):
    """Every (sequence, query head) of the full-size workload against the oracle."""
    x = CONFIGS[name]()
    out, lse, rc = DeviceDecode(x).run()
    assert rc == kv.KV_OK
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    worst = assert_decode_close(x, out, lse, ref_out, ref_lse)
    print(f"{name}: worst |out-oracle|/max|V| = {worst:.2e}")


def test_decode_tune_and_policy():
    """The calibrated choice among split sizes: every candidate is timed, the
    winner's output matches the oracle, and the policy reuses a signature's
    choice without timing again."""
    x = W.bimodal_b4()
    dd = DeviceDecode(x)
    cands = [0, 8, 32, 128]
    ws = kv.alloc_workspace(max(kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages, 16, 8),
                                kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages, 16, 0)))
    best, us = kv.kv_decode_tune(dd.q, dd.k, dd.v, dd.table, dd.lens, x.scale, dd.out, dd.lse, ws,
                                 cands, reps=3)
    assert best in cands and len(us) == len(cands) and all(u > 0 for u in us)
    assert us[cands.index(best)] == min(us)
    out, lse, rc = dd.run(pages_per_split=best, ws=ws)
    assert rc == 0
    ref_out, ref_lse = O.decode(x, nthreads=NCPU)
    assert_decode_close(x, out, lse, ref_out, ref_lse)
    pol = kv.DecodePolicy(candidates=cands, reps=2)
    p1 = pol.pages_per_split(x.seq_lens, dd.q, dd.k, dd.v, dd.table, dd.lens, x.scale, dd.out,
                             dd.lse, ws)
    p2 = pol.pages_per_split(x.seq_lens, dd.q, dd.k, dd.v, dd.table, dd.lens, x.scale, dd.out,
                             dd.lse, ws)
    assert p1 == p2 and len(pol.table) == 1 and p1 in cands
    print(f"B4 bimodal split sizes {dict(zip(cands, [round(u, 1) for u in us]))} us; best {best}")
