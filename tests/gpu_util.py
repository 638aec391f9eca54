"""Helpers for the GPU parity tests: move generated inputs to the device,
run the library, compare with the oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import oracle as O
from paged_kv_cache_492_b300 import kv
from paged_kv_cache_492_b300 import workloads as W

DEV = "cuda"


def tdtype(code):
    return torch.float16 if code == W.F16 else torch.bfloat16


def bits_to_dev(bits: np.ndarray, code: int) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(tdtype(code))


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)


class DeviceDecode:
    def __init__(self, x: W.DecodeInputs):
        self.x = x
        self.q = bits_to_dev(x.q, x.dtype)
        self.k = bits_to_dev(x.k_pool, x.dtype)
        self.v = bits_to_dev(x.v_pool, x.dtype)
        self.table = i32(x.block_table)
        self.lens = i32(x.seq_lens)
        self.out = torch.empty((x.B, x.Hq, x.d), dtype=torch.float32, device=DEV)
        self.lse = torch.empty((x.B, x.Hq), dtype=torch.float32, device=DEV)

    def run(self, pages_per_split=0, ws=None):
        x = self.x
        if ws is None:
            ws = kv.alloc_workspace(kv.kv_decode_workspace_size(x.B, x.Hq, x.Hkv, x.d, x.max_pages,
                                                                16, pages_per_split))
        self.out.fill_(float("nan"))
        self.lse.fill_(float("nan"))
        kv.kv_decode(self.q, self.k, self.v, self.table, self.lens, x.scale, self.out, self.lse, ws,
                     pages_per_split=pages_per_split)
        rc = kv.kv_get_status(ws)
        return self.out.cpu().numpy().astype(np.float64), self.lse.cpu().numpy().astype(np.float64), rc


def vmax_per_seq(x: W.DecodeInputs) -> np.ndarray:
    """max |V| over each sequence's valid tokens (the tolerance's scale)."""
    out = np.zeros(x.B)
    for b in range(x.B):
        L = int(x.seq_lens[b])
        if L == 0:
            continue
        pages = x.block_table[b, : -(-L // x.page_size)]
        v = x.v_pool[pages]
        if x.dtype == W.F16:
            vf = v.view(np.float16).astype(np.float32)
        else:
            vf = (v.astype(np.uint32) << 16).view(np.float32)
        vf = vf.transpose(0, 2, 1, 3).reshape(-1, x.Hkv, x.d)[:L]
        out[b] = np.abs(vf).max()
    return out


def assert_decode_close(x, out, lse, ref_out, ref_lse, rows=None):
    """max|out - oracle| <= 2e-3 max|V| and |lse - oracle| <= 1e-3; empty
    sequences exactly 0 / -inf."""
    vmax = vmax_per_seq(x)
    worst = 0.0
    bs = range(x.B) if rows is None else sorted({b for b, _ in rows})
    for b in bs:
        hs = range(x.Hq) if rows is None else [h for bb, h in rows if bb == b]
        for hq in hs:
            o = out[b, hq]
            lo = lse[b, hq]
            if rows is None:
                ro, rl = ref_out[b, hq], ref_lse[b, hq]
            else:
                i = rows.index((b, hq))
                ro, rl = ref_out[i], ref_lse[i]
            if x.seq_lens[b] == 0:
                assert np.all(o == 0) and lo == -math.inf, (b, hq)
                continue
            err = np.abs(o - ro).max()
            assert np.isfinite(o).all() and err <= 2e-3 * vmax[b], (b, hq, err, vmax[b])
            assert abs(lo - rl) <= 1e-3, (b, hq, lo, rl)
            worst = max(worst, err / vmax[b])
    return worst
