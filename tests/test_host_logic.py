"""Host-side logic that needs no GPU: the calibrated policy's workload
signature and caching, the header constants the binding mirrors, and the
bench's launch accounting."""
import math
import os
import re

import numpy as np
import pytest

import bench
from paged_kv_cache_492_b300 import kv
from paged_kv_cache_492_b300 import workloads as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "kv.h")


def _header_defines():
    out = {}
    with open(HEADER) as f:
        for line in f:
            m = re.match(r"#define\s+(KV_\w+)\s+\(?(-?\d+)\)?", line)
            if m:
                out[m.group(1)] = int(m.group(2))
    return out


def test_binding_constants_match_header():
    d = _header_defines()
    for name in ("KV_OK", "KV_EINVAL", "KV_EBADPAGE", "KV_ENOSPACE", "KV_EWORKSPACE", "KV_ECUDA",
                 "KV_EFULL", "KV_ETIMEOUT", "KV_F16", "KV_BF16", "KV_DECODE_TENSOR_CORE"):
        assert getattr(kv, name) == d[name], name


def test_policy_signature():
    sig = kv.DecodePolicy.signature
    # 8 sequences of one page each: 8 pages, log2 = 3, long/mean = 1
    assert sig([16] * 8) == (8, 3, 1)
    # empty batch of 3
    assert sig([0, 0, 0]) == (3, -1, 0.0)
    # lengths round up to pages
    assert sig([1, 17, 33]) == (3, int(math.log2(1 + 2 + 3)), round(3 / 2))
    # the bimodal batch: 8 sequences, ~6,500 pages, the long ones ~2x the mean
    x = W.bimodal()
    B, lg, ratio = sig(x.seq_lens)
    pages = sum(-(-int(L) // 16) for L in x.seq_lens)
    assert (B, lg) == (8, int(math.log2(pages))) and ratio == 2
    # batch order does not change the signature
    assert sig(list(reversed(x.seq_lens))) == sig(x.seq_lens)


def test_policy_calibrates_once_per_signature(monkeypatch):
    calls = []

    def fake_tune(q, k_pool, v_pool, table, lens, scale, out, lse, ws, candidates, reps,
                  stream=None, flush=None):
        calls.append(tuple(candidates))
        us = [10.0 + i for i in range(len(candidates))]
        us[-1] = 5.0  # the last candidate wins
        return candidates[-1], us

    monkeypatch.setattr(kv, "kv_decode_tune", fake_tune)
    # every variant supported except the tensor-core engine at d = 64
    monkeypatch.setattr(kv, "kv_decode_workspace_size",
                        lambda B, Hq, Hkv, d, maxp, ps=16, pps=0: 0 if (pps < 0 and d != 128) else 1)
    pol = kv.DecodePolicy()
    assert pol.candidates[-1] == kv.KV_DECODE_TENSOR_CORE and 0 in pol.candidates

    class Shaped:  # only .shape is read
        def __init__(self, *shape):
            self.shape = shape

    q = Shaped(3, 32, 128)
    table = Shaped(3, 2000)

    class Pool:  # [P, Hkv, page_size, d]
        shape = (10, 8, 16, 128)

    lens_a = [3000, 20, 500]
    lens_b = [3000, 20, 501]     # same pages, same signature
    lens_c = [30000, 20, 500]    # different page count
    for lens in (lens_a, lens_b, lens_a):
        assert pol.pages_per_split(lens, q, Pool(), None, table, None, 1.0, None, None,
                                   None) == kv.KV_DECODE_TENSOR_CORE
    assert len(calls) == 1 and len(pol.table) == 1
    pol.pages_per_split(lens_c, q, Pool(), None, table, None, 1.0, None, None, None)
    assert len(calls) == 2 and len(pol.table) == 2
    best, by_cand = pol.table[kv.DecodePolicy.signature(lens_c)]
    assert best == kv.KV_DECODE_TENSOR_CORE and by_cand[kv.KV_DECODE_TENSOR_CORE] == 5.0
    assert calls[0] == tuple(pol.candidates)
    # d = 64: the tensor-core engine is left out of the calibration
    assert pol.usable(3, 32, 8, 64, 2000) == [c for c in pol.candidates if c >= 0]
    assert pol.workspace_size(3, 32, 8, 64, 2000) == 1

    class Pool64:
        shape = (10, 8, 16, 64)

    pol.pages_per_split([7, 7, 7], Shaped(3, 32, 64), Pool64(), None, table, None, 1.0, None,
                        None, None)
    assert calls[-1] == tuple(c for c in pol.candidates if c >= 0)


def test_bench_launch_accounting():
    # fused kernel: one launch; tensor-core engine: attention + merge; a
    # page-offset pass above 1024 sequences
    assert bench.launches_per_step(8) == 1
    assert bench.launches_per_step(8, tensor_core=True) == 2
    assert bench.launches_per_step(1024, tensor_core=True) == 2
    assert bench.launches_per_step(1025) == 2
    assert bench.launches_per_step(1025, tensor_core=True) == 3


def test_bench_kernel_hash_tracks_engine_sources():
    h_fused, h_tc = bench.kernel_hash("fused"), bench.kernel_hash("tensor_core")
    assert re.fullmatch(r"[0-9a-f]{16}", h_fused) and re.fullmatch(r"[0-9a-f]{16}", h_tc)
    assert h_fused != h_tc


@pytest.mark.parametrize("name", ["bimodal", "uniform"])
def test_algorithmic_bytes_definition(name):
    """Algorithmic bytes per step: valid K/V tokens (2 Hkv d e each), q, and
    one 4-byte table entry per page read."""
    x = bench.WORKLOADS[name]()
    e = 2
    kv_bytes = int(np.sum(x.seq_lens)) * 2 * x.Hkv * x.d * e
    q_bytes = x.B * x.Hq * x.d * e
    table = 4 * sum(-(-int(L) // x.page_size) for L in x.seq_lens)
    assert x.kv_bytes() == kv_bytes
    assert x.algorithmic_bytes() == kv_bytes + q_bytes + table
