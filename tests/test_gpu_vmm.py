"""The elastic page pool (Elastic KV Cache, paperlayer.ai, section 3): K and
V pools in reserved address ranges whose backing grows and shrinks at the
top.  Pages below the mapped size never move, so block tables stay valid and
the decode kernel runs unchanged on a pool that grew between two calls."""
import math
import time

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_kv_cache_492_b300 import kv
from paged_kv_cache_492_b300 import workloads as W
from tests.gpu_util import assert_decode_close, i32

pytestmark = pytest.mark.gpu


def _decode(x, k, v, num_pages):
    dev = "cuda"
    q = torch.from_numpy(x.q.view(np.int16)).to(dev).view(torch.float16)
    out = torch.empty((x.B, x.Hq, x.d), dtype=torch.float32, device=dev)
    lse = torch.empty((x.B, x.Hq), dtype=torch.float32, device=dev)
    ws = kv.alloc_workspace(kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages))
    kv.kv_decode(q, k, v, i32(x.block_table), i32(x.seq_lens), x.scale, out, lse, ws,
                 num_pages=num_pages)
    assert kv.kv_get_status(ws) == 0
    return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def test_elastic_pool_grow_decode_shrink():
    Hkv, d, ps = 8, 128, 16
    page_bytes = Hkv * ps * d * 2
    pk = kv.VmmPool(1 << 30)
    pv = kv.VmmPool(1 << 30)
    try:
        gran_pages = pk.granularity // page_bytes
        P0 = 4 * gran_pages
        assert pk.resize(P0 * page_bytes) == P0 * page_bytes
        assert pv.resize(P0 * page_bytes) == P0 * page_bytes
        # a batch whose pages all lie below P0
        x = W.small_decode(81, 4, 32, Hkv, d, [900, 17, 2000, 333], pool_factor=1.0)
        P = x.num_pages
        assert P <= P0
        host_k = np.zeros((2 * P0, Hkv, ps, d), np.uint16)
        host_v = np.zeros((2 * P0, Hkv, ps, d), np.uint16)
        host_k[:P], host_v[:P] = x.k_pool, x.v_pool
        k0 = pk.tensor((P0, Hkv, ps, d), torch.float16)
        v0 = pv.tensor((P0, Hkv, ps, d), torch.float16)
        k0.copy_(torch.from_numpy(host_k[:P0].view(np.int16)).view(torch.float16))
        v0.copy_(torch.from_numpy(host_v[:P0].view(np.int16)).view(torch.float16))
        y = W.DecodeInputs(**{**x.__dict__, "k_pool": host_k[:P0], "v_pool": host_v[:P0]})
        ref_out, ref_lse = O.decode(y, nthreads=8)
        out, lse = _decode(y, k0, v0, P0)
        assert_decode_close(y, out, lse, ref_out, ref_lse)

        # grow: pages below P0 keep their bytes, pages above are new
        t0 = time.perf_counter()
        assert pk.resize(2 * P0 * page_bytes) == 2 * P0 * page_bytes
        assert pv.resize(2 * P0 * page_bytes) == 2 * P0 * page_bytes
        grow_s = time.perf_counter() - t0
        k1 = pk.tensor((2 * P0, Hkv, ps, d), torch.float16)
        v1 = pv.tensor((2 * P0, Hkv, ps, d), torch.float16)
        assert np.array_equal(k1[:P0].view(torch.int16).cpu().numpy().view(np.uint16), host_k[:P0])
        # move sequence 2 onto pages of the new slice
        rng = np.random.default_rng(2)
        n2 = -(-int(x.seq_lens[2]) // ps)
        new_ids = (P0 + rng.permutation(P0)[:n2]).astype(np.int32)
        table = x.block_table.copy()
        host_k[new_ids] = host_k[table[2, :n2]]
        host_v[new_ids] = host_v[table[2, :n2]]
        table[2, :n2] = new_ids
        k1[P0:].copy_(torch.from_numpy(host_k[P0:].view(np.int16)).view(torch.float16))
        v1[P0:].copy_(torch.from_numpy(host_v[P0:].view(np.int16)).view(torch.float16))
        z = W.DecodeInputs(**{**x.__dict__, "k_pool": host_k, "v_pool": host_v,
                              "block_table": table})
        ref_out2, ref_lse2 = O.decode(z, nthreads=8)
        out2, lse2 = _decode(z, k1, v1, 2 * P0)
        assert_decode_close(z, out2, lse2, ref_out2, ref_lse2)
        assert np.array_equal(out2, out) and np.array_equal(lse2, lse)  # same data, same math

        # shrink back once nothing references the upper slice
        t0 = time.perf_counter()
        assert pk.resize(P0 * page_bytes) == P0 * page_bytes
        assert pv.resize(P0 * page_bytes) == P0 * page_bytes
        shrink_s = time.perf_counter() - t0
        out3, lse3 = _decode(y, k0, v0, P0)
        assert np.array_equal(out3, out) and np.array_equal(lse3, lse)
        print(f"elastic pool: +{P0 * page_bytes * 2 >> 20} MiB in {grow_s * 1e3:.2f} ms, "
              f"-{P0 * page_bytes * 2 >> 20} MiB in {shrink_s * 1e3:.2f} ms")
    finally:
        pk.close()
        pv.close()


def test_elastic_pool_resize_latency():
    """Commit and release of 1 GiB slices (the quantity the Elastic-KV page
    measures for its reserve), one physical allocation per growth."""
    pool = kv.VmmPool(4 << 30)
    try:
        g = pool.granularity
        times_up, times_down = [], []
        for _ in range(3):
            t0 = time.perf_counter()
            pool.resize(1 << 30)
            times_up.append(time.perf_counter() - t0)
            t0 = time.perf_counter()
            assert pool.resize(0) == 0
            times_down.append(time.perf_counter() - t0)
        assert pool.mapped == 0 and g > 0
        print(f"elastic pool 1 GiB: map {min(times_up) * 1e3:.2f} ms, "
              f"unmap {min(times_down) * 1e3:.2f} ms (granularity {g >> 10} KiB)")
    finally:
        pool.close()
    small = kv.VmmPool(1 << 20)
    try:
        with pytest.raises(kv.KVError):
            small.resize(8 << 30)   # beyond the reservation: refused, nothing mapped
        assert small.mapped == 0
    finally:
        small.close()


def test_grown_pages_reach_the_free_list():
    """After the pool grows, kv_free_list_push hands the new pages to the free
    list (highest id first), so the next appends pop them in ascending order
    -- a budgeted grow can then draw on the pool's growth.  A push beyond the
    list's capacity is refused and changes nothing."""
    Hkv, d, ps = 2, 128, 16
    page_bytes = Hkv * ps * d * 2
    pk, pv = kv.VmmPool(1 << 28), kv.VmmPool(1 << 28)
    try:
        P0 = pk.granularity // page_bytes
        pk.resize(P0 * page_bytes)
        pv.resize(P0 * page_bytes)
        x = W.small_decode(82, 3, 8, Hkv, d, [32, 20, 48], pool_factor=1.0, pad_pages=1)
        assert x.num_pages <= P0
        cap = 2 * P0
        free_list = torch.full((cap,), -1, dtype=torch.int32, device="cuda")
        free_top = i32([0])                       # every page of the first slice in use
        ws = kv.alloc_workspace(kv.kv_status_workspace_size())
        # grow by one slice and hand its pages to the free list
        pk.resize(2 * P0 * page_bytes)
        pv.resize(2 * P0 * page_bytes)
        kv.kv_free_list_push(P0, P0, free_list, free_top, ws)
        assert kv.kv_get_status(ws) == 0
        assert int(free_top.item()) == P0
        assert np.array_equal(free_list[:P0].cpu().numpy(), np.arange(2 * P0 - 1, P0 - 1, -1))
        # appends to the sequences whose last page is full pop P0, P0 + 1, ...
        k = pk.tensor((2 * P0, Hkv, ps, d), torch.float16)
        v = pv.tensor((2 * P0, Hkv, ps, d), torch.float16)
        k[:x.num_pages].copy_(torch.from_numpy(x.k_pool.view(np.int16)).view(torch.float16))
        v[:x.num_pages].copy_(torch.from_numpy(x.v_pool.view(np.int16)).view(torch.float16))
        table, lens = i32(x.block_table), i32(x.seq_lens)
        rng = np.random.default_rng(3)
        kn = torch.from_numpy(W.normal_bits(rng, (3, Hkv, d), W.F16).view(np.int16)).cuda().view(
            torch.float16)
        vn = torch.from_numpy(W.normal_bits(rng, (3, Hkv, d), W.F16).view(np.int16)).cuda().view(
            torch.float16)
        wa = kv.alloc_workspace(kv.kv_append_workspace_size(3))
        kv.kv_append(kn, vn, k, v, table, lens, free_list, free_top, wa)
        assert kv.kv_get_status(wa) == 0
        t = table.cpu().numpy()
        assert t[0, 2] == P0 and t[2, 3] == P0 + 1      # full pages at L = 32 and 48
        assert np.array_equal(lens.cpu().numpy(), x.seq_lens + 1)
        assert torch.equal(k[P0, :, 0], kn[0]) and torch.equal(v[P0 + 1, :, 0], vn[2])
        # no room for more: refused, nothing changes
        before = free_list.clone()
        kv.kv_free_list_push(0, cap, free_list, free_top, ws)
        assert kv.kv_get_status(ws) == kv.KV_ENOSPACE
        assert torch.equal(free_list, before) and int(free_top.item()) == P0 - 2
    finally:
        pk.close()
        pv.close()
