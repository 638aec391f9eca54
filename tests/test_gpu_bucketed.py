"""GPU parity of the batch-1 long-context bucketed trace: contexts of 32768,
65536 and 131072 fp16 tokens (Hq=32, Hkv=8, d=128, page 16), 64 decode steps
each; every step appends the new token's K/V (a page comes off the free list
at each page boundary) and decodes over all tokens, with the split size
chosen from the length.  Each step is checked against the oracle run on the
same input state: the append bit for bit, the decode within tolerance, on
both decode engines (the fused kernel and the tensor-core engine the bench's
policy picks for these lengths)."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_kv_cache_492_b300 import kv
from paged_kv_cache_492_b300 import workloads as W
from tests.gpu_util import DeviceDecode, assert_decode_close, bits_to_dev, i32

pytestmark = pytest.mark.gpu
NCPU = len(os.sched_getaffinity(0))
# the oracle's per-row decodes run side by side (the C call releases the GIL)
_ROWS = ThreadPoolExecutor(max_workers=max(1, min(8, NCPU)))


def _decode_rows(y, rows):
    parts = [f.result() for f in [_ROWS.submit(O.decode_rows, y, [r]) for r in rows]]
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def _pool_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("engine", [kv.KV_DECODE_TENSOR_CORE, 0], ids=["tensor_core", "fused"])
@pytest.mark.parametrize("L0", [32768, 65536, 131072])
def test_bucketed_trace(L0, engine):
    # the full 64 steps on the engine the bench picks, half on the other
    steps = int(os.environ.get("KV_BUCKET_STEPS", "64" if engine else "32"))
    seed = 3
    x = W.bucketed_long(L0, seed=seed, steps=steps)
    dd = DeviceDecode(x)
    fl, ft = i32(x.free_list), i32([x.free_top])
    ws = kv.alloc_workspace(kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages, 16,
                                                        engine))
    ws_append = kv.alloc_workspace(kv.kv_append_workspace_size(x.B))
    # host state the oracle advances
    hk, hv = x.k_pool.copy(), x.v_pool.copy()
    ht, hl = x.block_table.copy(), x.seq_lens.copy()
    hfl, htop = x.free_list.copy(), np.array([x.free_top], np.int32)
    page_counts = set()
    for t in range(steps):
        q, kn, vn = W.step_tokens(seed, t, x.B, x.Hq, x.Hkv, x.d, x.dtype, trace=L0)
        L = int(hl[0])
        kv.kv_append(bits_to_dev(kn, x.dtype), bits_to_dev(vn, x.dtype), dd.k, dd.v, dd.table,
                     dd.lens, fl, ft, ws_append)
        assert kv.kv_get_status(ws_append) == 0, t
        rc = O.append_inplace(kn, vn, hk, hv, ht, hl, hfl, htop, x.Hkv, x.d, 16)
        assert rc == 0
        dd.q.copy_(bits_to_dev(q, x.dtype))
        dd.out.fill_(float("nan"))
        kv.kv_decode(dd.q, dd.k, dd.v, dd.table, dd.lens, x.scale, dd.out, dd.lse, ws,
                     pages_per_split=engine)
        assert kv.kv_get_status(ws) == 0, t
        # append: table, length, free list, and the written slot bit for bit
        assert np.array_equal(dd.table.cpu().numpy(), ht), t
        assert np.array_equal(dd.lens.cpu().numpy(), hl), t
        assert int(ft.item()) == int(htop[0]), t
        page = int(ht[0, L // 16])
        assert np.array_equal(_pool_bits(dd.k[page, :, L % 16]), hk[page, :, L % 16]), t
        assert np.array_equal(_pool_bits(dd.v[page, :, L % 16]), hv[page, :, L % 16]), t
        # decode over L + 1 tokens: four query heads every step, rotating so
        # two steps cover all eight KV heads, and all of them every 16 steps
        y = W.DecodeInputs(name=x.name, B=1, Hq=x.Hq, Hkv=x.Hkv, d=x.d, page_size=16,
                           dtype=x.dtype, scale=x.scale, q=q, k_pool=hk, v_pool=hv,
                           block_table=ht, seq_lens=hl)
        out = dd.out.cpu().numpy().astype(np.float64)
        lse = dd.lse.cpu().numpy().astype(np.float64)
        if t % 16 == 15 or t == steps - 1:
            ref_out, ref_lse = O.decode(y, nthreads=NCPU)
            assert_decode_close(y, out, lse, ref_out, ref_lse)
        else:
            G = x.Hq // x.Hkv
            kv_heads = range(t % 2, x.Hkv, 2)           # even KV heads, then odd
            rows = [(0, h * G + (t // 2) % G) for h in kv_heads]
            ref_out, ref_lse = _decode_rows(y, rows)
            assert_decode_close(y, out, lse, ref_out, ref_lse, rows=rows)
        page_counts.add(int(-(-(L + 1) // 16)))
    # the whole pools agree at the end (nothing else was written)
    assert np.array_equal(_pool_bits(dd.k), hk) and np.array_equal(_pool_bits(dd.v), hv)
    assert len(page_counts) == -(-steps // 16)  # a new page every 16 appends
