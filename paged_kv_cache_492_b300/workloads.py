"""Seeded synthetic inputs for paged GQA decode and page budgeting.

This module only *constructs inputs*: random queries and keys/values, sequence
lengths, block tables, pools and free lists.  It contains none of the
method's arithmetic (no attention, scoring, selection or compaction), so both
the CUDA path and the CPU oracle can consume its output without sharing any
of the computation.

Shapes follow the workloads the PersistentKV summary (aissential.tech,
"PersistentKV: Page-Aware Decode Scheduling ...", Summary) benchmarks on:
page size 16, Hq=32, Hkv=8, d=128, batch-8 bimodal / uniform / Zipf-like
length mixes and a batch-1 bucketed long-context trace.  The budgeting
workload follows GrowPage's setting (mlsanity.com GrowPage page, Abstract):
requests that grow one token per decode step under a per-request page budget.

Conventions (the build's own, stated once here):
  * RNG is numpy ``default_rng(seed)`` (PCG64); integer draws U[a, b] are
    inclusive of both ends.
  * Normal samples are drawn in float32 and rounded to the storage dtype
    (round-to-nearest-even, done by numpy for fp16 and torch for bf16).
  * Every 16-bit array is returned as ``np.uint16`` bit patterns together with
    a dtype code (0 = fp16, 1 = bf16), which is what both sides consume.
  * Pool layout is HND: ``[num_pages, Hkv, page_size, d]``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

F16 = 0
BF16 = 1
DTYPE_NAMES = {F16: "f16", BF16: "bf16"}


def to_bits(x_f32: np.ndarray, dtype: int) -> np.ndarray:
    """Round float32 samples to fp16/bf16 and return the raw 16-bit patterns."""
    x_f32 = np.ascontiguousarray(x_f32, dtype=np.float32)
    if dtype == F16:
        return x_f32.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        import torch

        t = torch.from_numpy(x_f32).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(f"unknown dtype code {dtype}")


def normal_bits(rng: np.random.Generator, shape, dtype: int, scale=None) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale is not None:
        x *= scale
    return to_bits(x, dtype)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


@dataclasses.dataclass
class DecodeInputs:
    """One decode step's inputs (host arrays)."""

    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    dtype: int
    scale: float
    q: np.ndarray            # [B, Hq, d] uint16
    k_pool: np.ndarray       # [P, Hkv, ps, d] uint16
    v_pool: np.ndarray       # [P, Hkv, ps, d] uint16
    block_table: np.ndarray  # [B, max_pages] int32, -1 padded
    seq_lens: np.ndarray     # [B] int32
    free_list: Optional[np.ndarray] = None  # [P] int32 stack (bottom first)
    free_top: int = 0

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def kv_bytes(self) -> int:
        """Bytes of valid K and V tokens (the decode's algorithmic KV traffic)."""
        return int(self.seq_lens.astype(np.int64).sum()) * 2 * self.Hkv * self.d * 2

    def algorithmic_bytes(self) -> int:
        """K/V of valid tokens + q + block-table entries read."""
        npages = sum(ceil_div(int(L), self.page_size) for L in self.seq_lens)
        return self.kv_bytes() + self.B * self.Hq * self.d * 2 + 4 * npages


def scatter_pages(rng, seq_lens, page_size, num_pages, max_pages):
    """Place each sequence's pages at random distinct pool positions.

    Returns (block_table, free_list, free_top): the table is -1 padded, and the
    pool pages not handed out form the free-list stack (in a random order).
    """
    B = len(seq_lens)
    nps = [ceil_div(int(L), page_size) for L in seq_lens]
    total = sum(nps)
    assert total <= num_pages, (total, num_pages)
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((B, max_pages), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        table[b, : nps[b]] = perm[pos: pos + nps[b]]
        pos += nps[b]
    free = perm[pos:].copy()
    free_list = np.full(num_pages, -1, dtype=np.int32)
    free_list[: len(free)] = free
    return table, free_list, len(free)


def make_decode(name, seed, B, Hq, Hkv, d, page_size, dtype, seq_lens,
                pool_factor=1.25, k_channel_scale=None, extra_pages=0,
                max_pages=None, rng=None) -> DecodeInputs:
    rng = rng if rng is not None else np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    nps = [ceil_div(int(L), page_size) for L in seq_lens]
    total = sum(nps)
    num_pages = max(1, int(math.ceil(pool_factor * (total + extra_pages))))
    if max_pages is None:
        max_pages = max(1, max(nps) if nps else 1)
    table, free_list, free_top = scatter_pages(rng, seq_lens, page_size, num_pages, max_pages)
    q = normal_bits(rng, (B, Hq, d), dtype)
    scale_kc = None
    if k_channel_scale is not None:
        lo, hi = k_channel_scale
        scale_kc = rng.uniform(lo, hi, size=(Hkv, d)).astype(np.float32)
    k_shape = (num_pages, Hkv, page_size, d)
    kf = rng.standard_normal(size=k_shape, dtype=np.float32)
    if scale_kc is not None:
        kf *= scale_kc[None, :, None, :]
    k_pool = to_bits(kf, dtype)
    del kf
    v_pool = normal_bits(rng, k_shape, dtype)
    return DecodeInputs(name=name, B=B, Hq=Hq, Hkv=Hkv, d=d, page_size=page_size, dtype=dtype,
                        scale=1.0 / math.sqrt(d), q=q, k_pool=k_pool, v_pool=v_pool,
                        block_table=table, seq_lens=seq_lens, free_list=free_list,
                        free_top=free_top)


# --------------------------------------------------------------------------
# The five workloads.
# --------------------------------------------------------------------------

def tiny(seed: int = 0) -> Dict:
    """Tiny paged decode: B=1, Hq=4, Hkv=1, d=64, ps=16, L=256 in a 64-page fp16
    pool (16 pages at a random permutation), plus 32 prior queries for the
    dual-EMA summaries (decays 0.5 / 0.99) and a keep-8-of-16 page selection."""
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, d, ps, P = 1, 4, 1, 64, 16, 64
    perm = rng.permutation(P).astype(np.int32)
    table = perm[:16].reshape(1, 16).copy()
    free_list = np.full(P, -1, dtype=np.int32)
    free_list[: P - 16] = perm[16:]
    q = normal_bits(rng, (B, Hq, d), F16)
    k_pool = normal_bits(rng, (P, Hkv, ps, d), F16)
    v_pool = normal_bits(rng, (P, Hkv, ps, d), F16)
    prior_q = normal_bits(rng, (32, B, Hq, d), F16)
    dec = DecodeInputs(name="tiny_b1_d64", B=B, Hq=Hq, Hkv=Hkv, d=d, page_size=ps, dtype=F16,
                       scale=1.0 / math.sqrt(d), q=q, k_pool=k_pool, v_pool=v_pool,
                       block_table=table, seq_lens=np.array([256], dtype=np.int32),
                       free_list=free_list, free_top=P - 16)
    return dict(decode=dec, prior_q=prior_q, a_fast=0.5, a_slow=0.99, keep=8)


def bimodal(seed: int = 1) -> DecodeInputs:
    """Batch-8 bimodal fp16 decode: 4 lengths from U[512, 2048] and 4 from
    U[16384, 32768], batch order shuffled; pool = ceil(1.25 x total pages);
    K scaled per (KV head, channel) by U[0.5, 2] drawn once."""
    rng = np.random.default_rng(seed)
    short = rng.integers(512, 2048, size=4, endpoint=True)
    long_ = rng.integers(16384, 32768, size=4, endpoint=True)
    lens = np.concatenate([short, long_])
    rng.shuffle(lens)
    return make_decode("bimodal_b8_fp16", seed, 8, 32, 8, 128, 16, F16, lens,
                       k_channel_scale=(0.5, 2.0), rng=rng)


def bimodal_b4(seed: int = 5) -> DecodeInputs:
    """Batch-4 bimodal fp16 decode (the B4 bimodal case of the PersistentKV
    summary, aissential.tech, Summary): 2 lengths from U[512, 2048] and 2
    from U[16384, 32768], shuffled; otherwise as the batch-8 bimodal case."""
    rng = np.random.default_rng(seed)
    short = rng.integers(512, 2048, size=2, endpoint=True)
    long_ = rng.integers(16384, 32768, size=2, endpoint=True)
    lens = np.concatenate([short, long_])
    rng.shuffle(lens)
    return make_decode("bimodal_b4_fp16", seed, 4, 32, 8, 128, 16, F16, lens,
                       k_channel_scale=(0.5, 2.0), rng=rng)


def uniform_lengths(seed: int = 2) -> DecodeInputs:
    """Batch-8 bf16 decode with lengths U[1024, 32768]."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1024, 32768, size=8, endpoint=True)
    return make_decode("uniform_b8_bf16", seed, 8, 32, 8, 128, 16, BF16, lens, rng=rng)


def zipf_lengths(seed: int = 2) -> DecodeInputs:
    """Batch-8 bf16 decode with lengths min(65536, 256 * Zipf(1.2)); table
    width = max pages, shorter rows padded with -1."""
    rng = np.random.default_rng([seed, 1])
    z = rng.zipf(1.2, size=8)
    lens = np.minimum(65536, 256 * z)
    return make_decode("zipf_b8_bf16", seed, 8, 32, 8, 128, 16, BF16, lens, rng=rng)


def bucketed_long(L0: int, seed: int = 3, steps: int = 64) -> DecodeInputs:
    """Batch-1 fp16 long-context decode at context L0; the pool has room for
    the pages the next `steps` appends allocate (they come off the free list)."""
    rng = np.random.default_rng([seed, L0])
    ps = 16
    extra = ceil_div(L0 + steps, ps) - ceil_div(L0, ps)
    max_pages = ceil_div(L0 + steps, ps)
    return make_decode(f"bucket_b1_{L0}_fp16", seed, 1, 32, 8, 128, ps, F16, [L0],
                       extra_pages=extra + 8, max_pages=max_pages, rng=rng)


def step_tokens(seed: int, step: int, B: int, Hq: int, Hkv: int, d: int, dtype: int,
                trace: Optional[int] = None):
    """The new query and the new token's K/V for one decode step (`trace`
    separates independent traces drawn from one seed)."""
    key = [seed, 1000 + step] if trace is None else [seed, trace, 1000 + step]
    rng = np.random.default_rng(key)
    q = normal_bits(rng, (B, Hq, d), dtype)
    k_new = normal_bits(rng, (B, Hkv, d), dtype)
    v_new = normal_bits(rng, (B, Hkv, d), dtype)
    return q, k_new, v_new


def budgeted_serving(seed: int = 4, B: int = 64, steps: int = 128,
                     len_range=(2048, 16384), budget_range=(32, 256)) -> Dict:
    """Batch-64 bf16 budgeted decode: lengths U[2048, 16384] growing one token
    per step, per-sequence page budgets U[32, 256], EMA decays 0.9 / 0.999.
    The pool holds every initial page plus growth room; pages not in a table
    start on the free list."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(len_range[0], len_range[1], size=B, endpoint=True)
    budget = rng.integers(budget_range[0], budget_range[1], size=B, endpoint=True).astype(np.int32)
    ps = 16
    max_pages = max(ceil_div(int(L), ps) for L in lens) + ceil_div(steps, ps) + 2
    dec = make_decode("budget_b64_bf16", seed, B, 32, 8, 128, ps, BF16, lens,
                      pool_factor=1.0, extra_pages=B * (ceil_div(steps, ps) + 2),
                      max_pages=max_pages, rng=rng)
    return dict(decode=dec, budget=budget, a_fast=0.9, a_slow=0.999, steps=steps,
                n_first=2, n_last=2, delta=0.5, seed=seed)


def small_decode(seed: int, B: int, Hq: int, Hkv: int, d: int, seq_lens: List[int],
                 dtype: int = F16, page_size: int = 16, pool_factor: float = 1.5,
                 pad_pages: int = 0) -> DecodeInputs:
    """Small randomized decode case for parity tests (ragged lengths, -1 padding)."""
    rng = np.random.default_rng(seed)
    nps = [ceil_div(int(L), page_size) for L in seq_lens]
    max_pages = max(1, max(nps) + pad_pages)
    return make_decode(f"small_s{seed}", seed, B, Hq, Hkv, d, page_size, dtype, seq_lens,
                       pool_factor=pool_factor, max_pages=max_pages, rng=rng)


def shared_prefix(seed: int, B: int, group: int, prefix_tokens: int, tail_lens: List[int],
                  Hq: int = 8, Hkv: int = 2, d: int = 64, dtype: int = F16,
                  pool_factor: float = 2.0, pad_pages: int = 2) -> Dict:
    """Sequences in groups of `group` share a cached prompt prefix of
    `prefix_tokens` tokens (the prefix caching GrowPage keeps, mlsanity.com
    GrowPage page, Abstract).  The prefix's full pages are one set of pool
    pages referenced by every member's block table.  A member with
    tail_lens[b] == 0 has not diverged yet (a fork): it also shares the
    prefix's partly filled last page, if any, and L_b = prefix_tokens.  A
    member with a tail owns every page after the full prefix pages (the rest
    of the prefix and its tail_lens[b] own tokens).  Returns the decode
    inputs and refcnt [P] int32, the number of block-table references to
    each pool page (0 = free)."""
    rng = np.random.default_rng(seed)
    ps = 16
    nfull = prefix_tokens // ps
    partial = prefix_tokens % ps != 0
    lens = np.array([prefix_tokens + int(t) for t in tail_lens], dtype=np.int32)
    own = [0 if int(t) == 0 else ceil_div(int(lens[b]), ps) - nfull for b, t in enumerate(tail_lens)]
    ngroups = ceil_div(B, group)
    total = ngroups * (nfull + int(partial)) + sum(own)
    P = max(1, int(math.ceil(pool_factor * total)))
    perm = rng.permutation(P).astype(np.int32)
    pos = 0
    shared = []
    for _ in range(ngroups):
        shared.append(perm[pos: pos + nfull + int(partial)].copy())
        pos += nfull + int(partial)
    max_pages = max(ceil_div(int(L), ps) for L in lens) + pad_pages
    table = np.full((B, max_pages), -1, dtype=np.int32)
    for b in range(B):
        g = shared[b // group]
        if tail_lens[b] == 0:
            table[b, : len(g)] = g
        else:
            table[b, :nfull] = g[:nfull]
            table[b, nfull: nfull + own[b]] = perm[pos: pos + own[b]]
            pos += own[b]
    refcnt = np.zeros(P, dtype=np.int32)
    for b in range(B):
        for j in range(ceil_div(int(lens[b]), ps)):
            refcnt[table[b, j]] += 1
    # the free list: every page no table references (in permutation order)
    free = perm[refcnt[perm] == 0].copy()
    free_list = np.full(P, -1, dtype=np.int32)
    free_list[: len(free)] = free
    q = normal_bits(rng, (B, Hq, d), dtype)
    k_pool = normal_bits(rng, (P, Hkv, ps, d), dtype)
    v_pool = normal_bits(rng, (P, Hkv, ps, d), dtype)
    dec = DecodeInputs(name=f"shared_prefix_s{seed}", B=B, Hq=Hq, Hkv=Hkv, d=d, page_size=ps,
                       dtype=dtype, scale=1.0 / math.sqrt(d), q=q, k_pool=k_pool, v_pool=v_pool,
                       block_table=table, seq_lens=lens, free_list=free_list, free_top=len(free))
    return dict(decode=dec, refcnt=refcnt)
