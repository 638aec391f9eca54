"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
a closed form, an independent library routine, a brute-force enumeration or
an invariant of the definition.  They are collected by ``test_oracle_pins.py``
and re-run against deliberately broken copies of the oracle by
``test_oracle_mutants.py`` (a pin set that cannot see a planted mistake is
not a pin).

Definitions pinned:
  * decode -- PersistentKV (aissential.tech) Summary/Method: GQA decode over a
    block table; the attention itself is the standard scaled-dot-product
    softmax, so torch's fp64 ``scaled_dot_product_attention`` with
    ``enable_gqa`` on a dense copy is an independent implementation;
  * split merge -- exact log-sum-exp recombination (implied by the page's
    "sequence-split" tasks);
  * workqueue -- PersistentKV Method: only non-empty (sequence, KV head,
    split) tasks;
  * summaries, scores, selection, compaction -- GrowPage (mlsanity.com,
    Abstract) as instantiated by this build (dual EMA, mean + channel min/max
    page summaries, top-k with lower-index ties, forced first/last pages,
    grow when the fast and slow working sets diverge).
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch
from scipy.special import logsumexp, softmax

from oracle import oracle as O
from paged_kv_cache_492_b300 import workloads as W


def _f64(bits, dtype):
    """Exact value of fp16/bf16 bit patterns via numpy/torch (not the oracle)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == W.F16:
        return bits.view(np.float16).astype(np.float64)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _gather(x, b):
    """Dense [L, Hkv, d] K and V of sequence b, read through the block table."""
    L = int(x.seq_lens[b])
    pages = x.block_table[b, : -(-L // x.page_size)]
    k = x.k_pool[pages].transpose(0, 2, 1, 3).reshape(-1, x.Hkv, x.d)[:L]
    v = x.v_pool[pages].transpose(0, 2, 1, 3).reshape(-1, x.Hkv, x.d)[:L]
    return k, v


def _fp16_case(q, k_tokens, v_tokens, scale=None, Hkv=1):
    """Build a DecodeInputs with B=1 from explicit float arrays (exactly
    representable in fp16): q [Hq, d], k/v [L, Hkv, d]; pages scattered."""
    rng = np.random.default_rng(123)
    q = np.asarray(q, np.float32)
    k_tokens = np.asarray(k_tokens, np.float32)
    v_tokens = np.asarray(v_tokens, np.float32)
    Hq, d = q.shape
    L = k_tokens.shape[0]
    ps = 16
    npg = -(-L // ps)
    P = npg + 3
    kp = np.zeros((P, Hkv, ps, d), np.float32)
    vp = np.zeros((P, Hkv, ps, d), np.float32)
    perm = rng.permutation(P)[:npg].astype(np.int32)
    for t in range(L):
        kp[perm[t // ps], :, t % ps] = k_tokens[t]
        vp[perm[t // ps], :, t % ps] = v_tokens[t]
    x = W.DecodeInputs(name="hand", B=1, Hq=Hq, Hkv=Hkv, d=d, page_size=ps, dtype=W.F16,
                       scale=(1.0 / math.sqrt(d)) if scale is None else scale,
                       q=W.to_bits(q[None], W.F16), k_pool=W.to_bits(kp, W.F16),
                       v_pool=W.to_bits(vp, W.F16), block_table=perm[None].copy(),
                       seq_lens=np.array([L], np.int32))
    for arr, ref in ((x.q[0], q), (x.k_pool, kp), (x.v_pool, vp)):
        assert np.array_equal(_f64(arr, W.F16), ref.astype(np.float64)), "not fp16-exact"
    return x


# --------------------------------------------------------------------------
# 16-bit formats
# --------------------------------------------------------------------------

def pin_f16_decoding():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([O.f16_to_f64(int(b)) for b in bits])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def pin_bf16_decoding():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = _f64(bits, W.BF16)
    got = np.array([O.bf16_to_f64(int(b)) for b in bits])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


# --------------------------------------------------------------------------
# decode
# --------------------------------------------------------------------------

def pin_decode_vs_sdpa():
    """Random ragged GQA case vs torch fp64 SDPA on a dense gathered copy."""
    for dtype, G in ((W.F16, 4), (W.BF16, 2), (W.F16, 1)):
        Hkv = 2
        x = W.small_decode(7 + G, B=3, Hq=Hkv * G, Hkv=Hkv, d=32, seq_lens=[37, 16, 5],
                           dtype=dtype, pad_pages=1)
        out, lse = O.decode(x)
        for b in range(x.B):
            k, v = _gather(x, b)
            qd = torch.from_numpy(_f64(x.q[b], dtype))[None, :, None, :]       # [1,Hq,1,d]
            kd = torch.from_numpy(_f64(k, dtype)).permute(1, 0, 2)[None]       # [1,Hkv,L,d]
            vd = torch.from_numpy(_f64(v, dtype)).permute(1, 0, 2)[None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qd, kd, vd, scale=x.scale, enable_gqa=True)[0, :, 0].numpy()
            assert np.allclose(out[b], ref, rtol=0, atol=1e-12), np.abs(out[b] - ref).max()
            # lse against scipy's logsumexp of the per-head logits
            kr = np.repeat(_f64(k, dtype), G, axis=1)                           # [L,Hq,d]
            s = x.scale * np.einsum("hd,lhd->hl", _f64(x.q[b], dtype), kr)
            assert np.allclose(lse[b], logsumexp(s, axis=1), rtol=0, atol=1e-12)


def pin_decode_single_token():
    """L = 1: out is that token's value and lse its logit."""
    d = 8
    q = np.array([[1, -2, 0.5, 0, 0, 0, 0, 3]], np.float32)
    k = np.array([[[2, 1, 4, 0, 0, 0, 0, -1]]], np.float32)
    v = np.array([[[0.25, -1, 7, 0, 2, 0, 0, 1]]], np.float32)
    x = _fp16_case(q, k, v)
    out, lse = O.decode(x)
    s = (1 * 2 + -2 * 1 + 0.5 * 4 + 3 * -1) / math.sqrt(d)
    assert abs(lse[0, 0] - s) < 1e-15
    assert np.array_equal(out[0, 0], v[0, 0].astype(np.float64))


def pin_decode_equal_keys():
    """All keys equal: uniform weights -> out = mean(V), lse = s + ln L."""
    d, L = 16, 37
    rng = np.random.default_rng(5)
    q = np.round(rng.standard_normal((1, d)) * 4) / 4
    kk = np.round(rng.standard_normal(d) * 4) / 4
    k = np.tile(kk, (L, 1))[:, None, :]
    v = (np.round(rng.standard_normal((L, 1, d)) * 8) / 8)
    x = _fp16_case(q, k, v)
    out, lse = O.decode(x)
    s = float(q[0] @ kk) / math.sqrt(d)
    assert abs(lse[0, 0] - (s + math.log(L))) < 1e-12
    assert np.allclose(out[0, 0], v[:, 0].mean(axis=0), rtol=0, atol=1e-12)


def pin_decode_zero_query():
    """q = 0: every logit is 0 -> lse = ln L, out = mean(V)."""
    x = W.small_decode(11, B=2, Hq=4, Hkv=2, d=32, seq_lens=[50, 3])
    x.q[:] = 0
    out, lse = O.decode(x)
    for b in range(2):
        _, v = _gather(x, b)
        vm = _f64(v, W.F16).mean(axis=0)                      # [Hkv, d]
        assert np.allclose(lse[b], math.log(x.seq_lens[b]), atol=1e-13)
        assert np.allclose(out[b], np.repeat(vm, 2, axis=0), atol=1e-13)


def pin_decode_onehot_values_give_softmax():
    """V rows = unit vectors e_t: out equals the softmax weights themselves;
    keys along e_0 make every logit a known product (scipy's softmax)."""
    d, L = 32, 20
    alphas = np.arange(L, dtype=np.float32) / 4 - 2.0      # exact in fp16
    beta = 1.5
    q = np.zeros((1, d), np.float32)
    q[0, 0] = beta
    k = np.zeros((L, 1, d), np.float32)
    k[:, 0, 0] = alphas
    v = np.zeros((L, 1, d), np.float32)
    for t in range(L):
        v[t, 0, t] = 1.0
    x = _fp16_case(q, k, v)
    out, lse = O.decode(x)
    s = alphas.astype(np.float64) * beta / math.sqrt(d)
    assert np.allclose(out[0, 0, :L], softmax(s), rtol=0, atol=1e-14)
    assert np.all(out[0, 0, L:] == 0)
    assert abs(lse[0, 0] - logsumexp(s)) < 1e-13


def pin_decode_rows_sum_to_one():
    """V = 1 everywhere: the softmax rows sum to one, so out == 1."""
    x = W.small_decode(13, B=2, Hq=8, Hkv=2, d=32, seq_lens=[70, 17])
    x.v_pool[:] = W.to_bits(np.ones(1, np.float32), W.F16)[0]
    out, _ = O.decode(x)
    assert np.allclose(out, 1.0, rtol=0, atol=1e-13)


def pin_decode_placement_invariance():
    """Moving pages inside the pool and rewriting the table changes nothing
    (bit-identical: same logical order, same arithmetic)."""
    x = W.small_decode(17, B=3, Hq=8, Hkv=4, d=32, seq_lens=[45, 64, 1])
    out0, lse0 = O.decode(x)
    rng = np.random.default_rng(0)
    perm = rng.permutation(x.num_pages)              # new position of page p
    y = W.DecodeInputs(**{**x.__dict__})
    y.k_pool = np.empty_like(x.k_pool)
    y.v_pool = np.empty_like(x.v_pool)
    y.k_pool[perm] = x.k_pool
    y.v_pool[perm] = x.v_pool
    y.block_table = np.where(x.block_table >= 0, perm[np.maximum(x.block_table, 0)], -1).astype(np.int32)
    out1, lse1 = O.decode(y)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_decode_token_permutation():
    """Attention is a set function of the (k, v) pairs: permuting the
    logical token order changes only rounding."""
    x = W.small_decode(19, B=1, Hq=4, Hkv=2, d=32, seq_lens=[53])
    out0, lse0 = O.decode(x)
    L, ps = 53, 16
    rng = np.random.default_rng(1)
    perm = rng.permutation(L)
    y = W.DecodeInputs(**{**x.__dict__})
    y.k_pool = x.k_pool.copy()
    y.v_pool = x.v_pool.copy()
    tb = x.block_table[0]
    for t_new, t_old in enumerate(perm):
        y.k_pool[tb[t_new // ps], :, t_new % ps] = x.k_pool[tb[t_old // ps], :, t_old % ps]
        y.v_pool[tb[t_new // ps], :, t_new % ps] = x.v_pool[tb[t_old // ps], :, t_old % ps]
    out1, lse1 = O.decode(y)
    assert np.allclose(out0, out1, rtol=0, atol=1e-12)
    assert np.allclose(lse0, lse1, rtol=0, atol=1e-12)


def pin_split_merge_invariance():
    """Any partition of the tokens into splits, merged by log-sum-exp, gives
    the unsplit result."""
    x = W.small_decode(23, B=1, Hq=4, Hkv=1, d=32, seq_lens=[100])
    out, lse = O.decode(x)
    rng = np.random.default_rng(2)
    for _ in range(5):
        cuts = np.sort(rng.choice(np.arange(1, 100), size=rng.integers(1, 6), replace=False))
        bounds = [0, *cuts.tolist(), 100]
        for hq in range(4):
            parts = [O.decode_range(x, 0, hq, a, b) for a, b in zip(bounds[:-1], bounds[1:])]
            o, l = O.merge(np.array([p[1] for p in parts]), np.stack([p[0] for p in parts]))
            assert np.allclose(o, out[0, hq], rtol=0, atol=1e-12)
            assert abs(l - lse[0, hq]) < 1e-12
    # an empty part (lse = -inf) contributes nothing
    o0, l0 = O.decode_range(x, 0, 0, 0, 0)
    assert l0 == -math.inf and np.all(o0 == 0)
    o, l = O.merge(np.array([l0, lse[0, 0]]), np.stack([o0, out[0, 0]]))
    assert np.allclose(o, out[0, 0], atol=1e-14) and abs(l - lse[0, 0]) < 1e-14


def pin_attend_multi():
    """T query tokens per sequence (the last T, causal): T = 1 is decode;
    query i is decode over the first L - T + 1 + i tokens; and torch fp64
    SDPA with an explicit causal mask on a dense copy agrees."""
    rng = np.random.default_rng(17)
    for dtype, G, T in ((W.F16, 4, 3), (W.BF16, 2, 1), (W.F16, 1, 5)):
        Hkv = 2
        x = W.small_decode(60 + T, B=3, Hq=Hkv * G, Hkv=Hkv, d=32, seq_lens=[37, 3, 16],
                           dtype=dtype, pad_pages=1)
        qm = W.normal_bits(rng, (x.B, T, x.Hq, x.d), dtype)
        out, lse = O.attend_multi(x, qm)
        for i in range(T):
            y = W.DecodeInputs(**{**x.__dict__, "q": np.ascontiguousarray(qm[:, i]),
                                  "seq_lens": np.maximum(0, x.seq_lens - T + 1 + i).astype(np.int32)})
            o1, l1 = O.decode(y)
            assert np.allclose(out[:, i], o1, rtol=0, atol=1e-13)
            assert np.array_equal(np.isneginf(lse[:, i]), np.isneginf(l1))
            fin = np.isfinite(l1)
            assert np.allclose(lse[:, i][fin], l1[fin], rtol=0, atol=1e-13)
        for b in range(x.B):
            L = int(x.seq_lens[b])
            k, v = _gather(x, b)
            qd = torch.from_numpy(_f64(qm[b], dtype)).permute(1, 0, 2)[None]  # [1,Hq,T,d]
            kd = torch.from_numpy(_f64(k, dtype)).permute(1, 0, 2)[None]
            vd = torch.from_numpy(_f64(v, dtype)).permute(1, 0, 2)[None]
            pos = torch.arange(L)[None, :]
            lim = (L - T + 1 + torch.arange(T))[:, None]
            mask = pos < lim                                                 # [T, L]
            ok = mask.any(dim=1)
            if not ok.any():
                continue
            ref = torch.nn.functional.scaled_dot_product_attention(
                qd[:, :, ok], kd, vd, attn_mask=mask[ok], scale=x.scale, enable_gqa=True)
            got = torch.from_numpy(out[b][ok.numpy()]).permute(1, 0, 2)[None]
            assert torch.allclose(got, ref, rtol=0, atol=1e-12)
        if T == 1:
            o0, l0 = O.decode(W.DecodeInputs(**{**x.__dict__, "q": np.ascontiguousarray(qm[:, 0])}))
            assert np.allclose(out[:, 0], o0, rtol=0, atol=0)


def pin_decode_edge_cases():
    x = W.small_decode(29, B=3, Hq=4, Hkv=2, d=32, seq_lens=[0, 16, 17], pad_pages=2)
    out, lse = O.decode(x)
    assert np.all(out[0] == 0) and np.all(lse[0] == -math.inf)
    bad = W.DecodeInputs(**{**x.__dict__})
    bad.block_table = x.block_table.copy()
    bad.block_table[2, 1] = -1                      # -1 inside the valid range
    try:
        O.decode(bad)
        raise AssertionError("bad page not reported")
    except O.OracleError as e:
        assert e.rc == O.EBADPAGE
    bad.block_table[2, 1] = x.num_pages              # out of range
    try:
        O.decode(bad)
        raise AssertionError("bad page not reported")
    except O.OracleError as e:
        assert e.rc == O.EBADPAGE
    # entries past the valid pages are never read, whatever they hold
    ok = W.DecodeInputs(**{**x.__dict__})
    ok.block_table = x.block_table.copy()
    ok.block_table[1, 1:] = 10 ** 6
    out2, lse2 = O.decode(ok)
    assert np.array_equal(out2, out) and np.array_equal(lse2, lse)


# --------------------------------------------------------------------------
# workqueue
# --------------------------------------------------------------------------

def _workqueue_brute(seq_lens, Hkv, ps, chunk):
    """Assign every page of the flattened batch to a chunk one page at a time
    and group runs of equal (sequence, chunk): an independent formulation."""
    tiles = []  # (b, j, chunk)
    g = 0
    for b, L in enumerate(seq_lens):
        for j in range(-(-int(L) // ps)):
            tiles.append((b, j, g // chunk))
            g += 1
    groups = []
    for key, run in itertools.groupby(tiles, key=lambda t: (t[0], t[2])):
        run = list(run)
        groups.append((key[0], key[1], run[0][1], run[-1][1] + 1))
    tasks = []
    for b in range(len(seq_lens)):
        mine = [gr for gr in groups if gr[0] == b]
        for s, (_, c, p0, p1) in enumerate(mine):
            for h in range(Hkv):
                tasks.append((b, h, s, len(mine), p0, p1, c, int(seq_lens[b])))
    nchunks = -(-g // chunk) if g else 0
    chunk_begin = []
    for c in range(nchunks + 1):
        idx = next((i for i, gr in enumerate(groups) if gr[1] >= c), len(groups))
        chunk_begin.append(idx)
    return np.array(tasks, dtype=np.int32).reshape(-1, 8), np.array(chunk_begin, np.int32)


def pin_workqueue_brute_force():
    rng = np.random.default_rng(3)
    cases = [([256], 1, 16, 4), ([0, 0, 0], 8, 16, 5), ([1, 15, 16, 17, 0, 33], 2, 16, 3),
             ([5000, 0, 12, 70000 // 7], 8, 16, 37)]
    for _ in range(20):
        B = int(rng.integers(1, 9))
        lens = [int(v) for v in rng.integers(0, 400, size=B)]
        lens[int(rng.integers(0, B))] = 0
        cases.append((lens, int(rng.integers(1, 5)), 16, int(rng.integers(1, 30))))
    for lens, Hkv, ps, chunk in cases:
        wq = O.workqueue(lens, Hkv, ps, chunk)
        tasks, cb = _workqueue_brute(lens, Hkv, ps, chunk)
        assert np.array_equal(wq["tasks"], tasks), (lens, Hkv, chunk)
        assert np.array_equal(wq["chunk_begin"], cb), (lens, chunk)
        # every task is non-empty and the tasks tile each sequence exactly once
        assert np.all(wq["tasks"][:, 5] > wq["tasks"][:, 4])
        for b, L in enumerate(lens):
            for h in range(Hkv):
                mine = wq["tasks"][(wq["tasks"][:, 0] == b) & (wq["tasks"][:, 1] == h)]
                covered = sorted(j for t in mine for j in range(t[4], t[5]))
                assert covered == list(range(-(-L // ps)))
        assert O.chunk_auto(wq["W"], 148, 8) >= 8


# --------------------------------------------------------------------------
# budgeting chain
# --------------------------------------------------------------------------

def pin_ema_closed_forms():
    B, Hq, Hkv, d = 2, 8, 2, 32
    rng = np.random.default_rng(4)
    qs = [W.normal_bits(rng, (B, Hq, d), W.F16) for _ in range(6)]
    a_f, a_s = 0.9, 0.5
    # constant queries: the averages equal the group mean at every step
    e = np.zeros((B, 2, Hkv, d))
    for t in range(5):
        O.ema_f64(qs[0], B, Hq, Hkv, d, W.F16, a_f, a_s, t == 0, e)
    gm = _f64(qs[0], W.F16).reshape(B, Hkv, Hq // Hkv, d).mean(axis=2)
    assert np.allclose(e[:, 0], gm, atol=1e-14) and np.allclose(e[:, 1], gm, atol=1e-14)
    # unrolled: ema_T = a^(T-1) g_1 + sum_{i=2..T} (1-a) a^(T-i) g_i
    e = np.zeros((B, 2, Hkv, d))
    for t, q in enumerate(qs):
        O.ema_f64(q, B, Hq, Hkv, d, W.F16, a_f, a_s, t == 0, e)
    g = [_f64(q, W.F16).reshape(B, Hkv, Hq // Hkv, d).mean(axis=2) for q in qs]
    T = len(qs)
    for u, a in ((0, a_f), (1, a_s)):
        ref = a ** (T - 1) * g[0] + sum((1 - a) * a ** (T - 1 - i) * g[i] for i in range(1, T))
        assert np.allclose(e[:, u], ref, atol=1e-13)
    # fp32 version stays within a few fp32 ulps of the fp64 one
    e32 = np.zeros((B, 2, Hkv, d), np.float32)
    for t, q in enumerate(qs):
        O.ema_f32(q, B, Hq, Hkv, d, W.F16, a_f, a_s, t == 0, e32)
    assert np.allclose(e32, e, rtol=0, atol=1e-5 * max(1.0, np.abs(e).max()))
    # first step is exactly the group mean in fp32 too (G = 4 -> exact /4)
    f = np.zeros((B, 2, Hkv, d), np.float32)
    O.ema_f32(qs[1], B, Hq, Hkv, d, W.F16, a_f, a_s, True, f)
    g1 = _f64(qs[1], W.F16).reshape(B, Hkv, Hq // Hkv, d)
    ref32 = ((((g1[:, :, 0].astype(np.float32) + g1[:, :, 1].astype(np.float32))
               + g1[:, :, 2].astype(np.float32)) + g1[:, :, 3].astype(np.float32)) / np.float32(4))
    assert np.array_equal(f[:, 0], ref32) and np.array_equal(f[:, 1], ref32)


def pin_page_summaries():
    rng = np.random.default_rng(6)
    P, Hkv, ps, d = 9, 2, 16, 32
    for dtype in (W.F16, W.BF16):
        kp = W.normal_bits(rng, (P, Hkv, ps, d), dtype)
        ids = np.array([3, 0, 8], np.int32)
        s64 = np.zeros((P, Hkv, 3, d))
        s32 = np.zeros((P, Hkv, 3, d), np.float32)
        O.page_summaries_f64(kp, ids, Hkv, ps, d, dtype, s64)
        O.page_summaries_f32(kp, ids, Hkv, ps, d, dtype, s32)
        kv = _f64(kp, dtype)
        for p in ids:
            assert np.allclose(s64[p, :, 0], kv[p].mean(axis=1), atol=1e-15)
            assert np.array_equal(s64[p, :, 1], kv[p].min(axis=1))
            assert np.array_equal(s64[p, :, 2], kv[p].max(axis=1))
            assert np.array_equal(s32[p, :, 1:], s64[p, :, 1:].astype(np.float32))
            bound = ps * 2.0 ** -24 * np.abs(kv[p]).max()
            assert np.abs(s32[p, :, 0] - s64[p, :, 0]).max() <= bound
        untouched = [p for p in range(P) if p not in ids]
        assert np.all(s64[untouched] == 0) and np.all(s32[untouched] == 0)


def _score_setup(rng, B=2, Hkv=2, d=32, ps=16, lens=(40, 64), P=12):
    ema = rng.standard_normal((B, 2, Hkv, d))
    kp = W.normal_bits(rng, (P, Hkv, ps, d), W.F16)
    summ = np.zeros((P, Hkv, 3, d))
    O.page_summaries_f64(kp, np.arange(P, dtype=np.int32), Hkv, ps, d, W.F16, summ)
    maxp = 5
    table = np.full((B, maxp), -1, np.int32)
    perm = rng.permutation(P)
    pos = 0
    for b, L in enumerate(lens):
        n = -(-L // ps)
        table[b, :n] = perm[pos:pos + n]
        pos += n
    return ema, kp, summ, table, np.array(lens, np.int32)


def pin_scores_identical_keys():
    """A page whose tokens all share key k: mean = min = max = k, so the
    score is sum_h 2 <u_h, k_h>."""
    rng = np.random.default_rng(8)
    B, Hkv, d, ps, P = 1, 2, 32, 16, 3
    k = np.round(rng.standard_normal((P, Hkv, d)) * 8) / 8
    kp = np.repeat(k[:, :, None, :], ps, axis=2).astype(np.float32)
    bits = W.to_bits(kp, W.F16)
    summ = np.zeros((P, Hkv, 3, d))
    O.page_summaries_f64(bits, np.arange(P, dtype=np.int32), Hkv, ps, d, W.F16, summ)
    ema = rng.standard_normal((B, 2, Hkv, d))
    table = np.array([[2, 0, 1]], np.int32)
    sc = np.zeros((B, 3, 2))
    O.score_pages_f64(ema, summ, table, np.array([48], np.int32), None, Hkv, d, ps, sc)
    kv = _f64(bits, W.F16)[:, :, 0, :]
    for j, p in enumerate(table[0]):
        for u in range(2):
            ref = 2 * sum(float(ema[0, u, h] @ kv[p, h]) for h in range(Hkv))
            assert abs(sc[0, j, u] - ref) < 1e-12


def pin_scores_corner_bound():
    """sum_c max(u_c min_c, u_c max_c) is the maximum of <u, x> over the box
    [min, max]: compare with all 2^d corners on a small d (mean set to 0),
    and check it bounds every token's logit from above."""
    rng = np.random.default_rng(9)
    d, Hkv, ps = 6, 1, 16
    kp = W.normal_bits(rng, (2, Hkv, ps, d), W.F16)
    summ = np.zeros((2, Hkv, 3, d))
    O.page_summaries_f64(kp, np.array([0, 1], np.int32), Hkv, ps, d, W.F16, summ)
    summ0 = summ.copy()
    summ0[:, :, 0] = 0.0
    ema = rng.standard_normal((1, 2, Hkv, d))
    sc = np.zeros((1, 2, 2))
    O.score_pages_f64(ema, summ0, np.array([[1, 0]], np.int32), np.array([32], np.int32), None,
                      Hkv, d, ps, sc)
    kv = _f64(kp, W.F16)
    for j, p in enumerate((1, 0)):
        for u in range(2):
            uu = ema[0, u, 0]
            best = max(float(uu @ np.array(c)) for c in itertools.product(
                *[(summ[p, 0, 1, i], summ[p, 0, 2, i]) for i in range(d)]))
            assert abs(sc[0, j, u] - best) < 1e-12
            assert sc[0, j, u] >= (kv[p, 0] @ uu).max() - 1e-12
    # the mean term is the mean of the token logits
    sc2 = np.zeros((1, 2, 2))
    summ1 = summ.copy()
    summ1[:, :, 1:] = 0.0
    O.score_pages_f64(ema, summ1, np.array([[1, 0]], np.int32), np.array([32], np.int32), None,
                      Hkv, d, ps, sc2)
    for j, p in enumerate((1, 0)):
        for u in range(2):
            assert abs(sc2[0, j, u] - (kv[p, 0] @ ema[0, u, 0]).mean()) < 1e-12


def pin_scores_f32_vs_f64_and_layout():
    rng = np.random.default_rng(10)
    ema, kp, summ, table, lens = _score_setup(rng)
    B, maxp = table.shape
    Hkv, d, ps = 2, 32, 16
    s64 = np.zeros((B, maxp, 2))
    O.score_pages_f64(ema, summ, table, lens, None, Hkv, d, ps, s64)
    e32 = ema.astype(np.float32)
    summ32 = np.zeros(summ.shape, np.float32)
    O.page_summaries_f32(kp, np.arange(summ.shape[0], dtype=np.int32), Hkv, ps, d, W.F16, summ32)
    s32 = np.zeros((B, maxp, 2), np.float32)
    O.score_pages_f32(e32, summ32, table, lens, None, Hkv, d, ps, s32)
    s64b = np.zeros((B, maxp, 2))
    O.score_pages_f64(e32.astype(np.float64), summ32.astype(np.float64), table, lens, None,
                      Hkv, d, ps, s64b)
    fin = np.isfinite(s64)
    assert np.array_equal(fin, np.isfinite(s32))
    assert np.all(s32[~fin] == -np.inf)
    # fp32 error bound for the stated order: each term carries <= 2 roundings
    # of its own, each lane sums Hkv*d/32 terms, then 5 butterfly adds:
    # |err| <= (Hkv*d/32 + 5 + 2) * 2^-24 * sum |terms| (first order).
    for b in range(B):
        for j in range(-(-int(lens[b]) // ps)):
            p = table[b, j]
            for u in range(2):
                uu = e32[b, u].astype(np.float64)
                sm = summ32[p].astype(np.float64)
                terms = np.abs(uu * sm[:, 0]) + np.maximum(np.abs(uu * sm[:, 1]), np.abs(uu * sm[:, 2]))
                bound = (Hkv * d / 32 + 7) * 2.0 ** -24 * terms.sum()
                assert abs(float(s32[b, j, u]) - s64b[b, j, u]) <= bound, (b, j, u)
    # inactive rows stay untouched
    s = np.full((B, maxp, 2), 7.0, np.float32)
    O.score_pages_f32(e32, summ32, table, lens, np.array([0, 1], np.uint8), Hkv, d, ps, s)
    assert np.all(s[0] == 7.0) and np.array_equal(s[1], s32[1])


def _topk_brute(keys, cands, k):
    """Best k-subset: compare subsets by their keys sorted descending
    (lexicographically), ties by the sorted index list ascending."""
    best, best_key = None, None
    for sub in itertools.combinations(cands, k):
        key = (tuple(sorted((-keys[j] for j in sub))), tuple(sorted(sub)))
        if best_key is None or key < best_key:
            best, best_key = set(sub), key
    return best if best is not None else set()


def pin_topk_brute_force():
    rng = np.random.default_rng(12)
    n, k = 16, 8
    for trial in range(6):
        sf = rng.standard_normal(n).astype(np.float32)
        ss = rng.standard_normal(n).astype(np.float32)
        if trial % 2:  # planted ties
            sf[[1, 5, 9]] = sf[3]
            ss[[1, 5, 9]] = ss[3] - 0.0
            ss[2] = sf[2] = 0.0
        scores = np.stack([sf, ss], -1)[None]
        keep, grow, budget, _ = O.select_pages(scores, np.array([256], np.int32), None,
                                               np.array([k], np.int32), 16, 0, 0, 0.5,
                                               O.SELECT_TOPK, 0)
        R = (sf + ss).astype(np.float32)
        ref = _topk_brute({j: float(R[j]) for j in range(n)}, range(n), k)
        assert set(np.nonzero(keep[0])[0]) == ref
        assert grow[0] == 0 and budget[0] == k


def pin_select_forced_and_boundary_rule():
    """Hand-built rows for the boundary rule.  n = 12 resident pages,
    F = {0, 1, 10, 11}, C = {2..9} (8 pages), k = 7, w = ceil(0.5 * 8) = 4,
    delta = 0.5 -> grow iff D > 2."""
    ps, maxp, n = 16, 14, 12
    lens = np.array([n * ps] * 4 + [5 * ps], np.int32)
    B = len(lens)
    sc = np.full((B, maxp, 2), -np.inf, np.float32)
    j = np.arange(n, dtype=np.float32)
    sc[0, :n, 0] = j          # b0: fast and slow agree -> D = 0 -> compact
    sc[0, :n, 1] = j
    sc[1, :n, 0] = j          # b1: W_f = {6..9}, W_s = {2..5} -> D = 4 -> grow
    sc[1, :n, 1] = -j
    sc[2, :n, 0] = j          # b2: same drift, but the only free page went to b1
    sc[2, :n, 1] = -j
    sc[3, :n, 0] = j          # b3: W_s = {2, 3, 6, 7} -> D = |{8, 9}| = 2 = delta*w
    sc[3, :n, 1] = 0.0
    sc[3, [6, 7], 1] = 10.0
    sc[3, [2, 3], 1] = 9.0
    act = np.array([1, 1, 1, 1, 0], np.uint8)   # b4 inactive
    budget = np.array([n, n, n, n, 3], np.int32)
    keep, grow, bud, drift = O.select_pages(sc, lens, act, budget, ps, 2, 2, 0.5,
                                            O.SELECT_BOUNDARY, 1, ws_frac=0.5)
    assert drift.tolist()[:4] == [0, 4, 4, 2]
    assert grow.tolist() == [0, 1, 0, 0, 0] and bud.tolist() == [n, n + 1, n, n, 3]
    # b0 evicts the lowest R = 2j in C: page 2
    assert keep[0, :n].tolist() == [1, 1, 0, 1, 1, 1, 1, 1, 1, 1, 1, 1]
    assert keep[1, :n].all() and not keep[1, n:].any()
    # b2: R = 0 on all of C -> ties broken by lower index -> page 9 evicted
    assert keep[2, :n].tolist() == [1, 1, 1, 1, 1, 1, 1, 1, 1, 0, 1, 1]
    # b3: D = 2 is not > 2 -> compact; R = {2: 11, 3: 12, 4: 4, 5: 5, 6: 16, 7: 17, 8: 8, 9: 9}
    assert keep[3, :n].tolist() == [1, 1, 1, 1, 0, 1, 1, 1, 1, 1, 1, 1]
    assert keep[4, :5].all() and not keep[4, 5:].any()
    # two free pages: b1 and b2 both grow
    _, grow2, bud2, _ = O.select_pages(sc, lens, act, budget, ps, 2, 2, 0.5,
                                       O.SELECT_BOUNDARY, 2, ws_frac=0.5)
    assert grow2.tolist() == [0, 1, 1, 0, 0] and bud2.tolist() == [n, n + 1, n + 1, n, 3]
    # plenty of free pages: b3 sits exactly at D = delta*w and must not grow
    _, grow4, _, _ = O.select_pages(sc, lens, act, budget, ps, 2, 2, 0.5,
                                    O.SELECT_BOUNDARY, 9, ws_frac=0.5)
    assert grow4.tolist() == [0, 1, 1, 0, 0]
    # smaller working sets: w = ceil(0.25 * 8) = 2 -> b3's W_s = {6, 7}, W_f = {8, 9}: D = 2 > 1
    _, grow3, _, drift3 = O.select_pages(sc, lens, act, budget, ps, 2, 2, 0.5,
                                         O.SELECT_BOUNDARY, 9, ws_frac=0.25)
    assert drift3.tolist()[:4] == [0, 2, 2, 2] and grow3.tolist() == [0, 1, 1, 1, 0]
    # fractional working-set size rounds up: w = ceil(0.3 * 8) = 3
    _, _, _, drift5 = O.select_pages(sc, lens, act, budget, ps, 2, 2, 0.5,
                                     O.SELECT_BOUNDARY, 9, ws_frac=0.3)
    assert drift5.tolist()[:4] == [0, 3, 3, 2]
    # forced pages survive even with the worst scores
    sc2 = sc.copy()
    sc2[0, [0, 1, n - 2, n - 1], :] = -1e30
    keep, *_ = O.select_pages(sc2, lens, act, budget, ps, 2, 2, 0.5, O.SELECT_BOUNDARY, 0)
    assert keep[0, [0, 1, n - 2, n - 1]].all() and keep[0, :n].sum() == n - 1
    # TOPK fit: keep F plus budget-|F| best of C (by R = 2j on b0)
    keep, grow, bud, _ = O.select_pages(sc, lens, np.array([1, 0, 0, 0, 0], np.uint8),
                                        np.array([6, 0, 0, 0, 0], np.int32), ps, 2, 2, 0.5,
                                        O.SELECT_TOPK, 0)
    assert keep[0, :n].tolist() == [1, 1, 0, 0, 0, 0, 0, 0, 1, 1, 1, 1]
    assert keep[1, :n].all() and not grow.any() and bud[0] == 6
    # no candidates (all pages forced): the sequence asks to grow
    small = np.array([3 * ps], np.int32)
    sc3 = np.zeros((1, 4, 2), np.float32)
    _, g, b_, _ = O.select_pages(sc3, small, None, np.array([3], np.int32), ps, 2, 2, 0.5,
                                 O.SELECT_BOUNDARY, 1)
    assert g[0] == 1 and b_[0] == 4


def _compact_naive(table, seq_lens, keep, token_gran, k_pool, v_pool, free_list, top, ps):
    """Token-list re-pack written from the definition with Python lists."""
    table = table.copy()
    seq_lens = seq_lens.copy()
    k_pool = k_pool.copy()
    v_pool = v_pool.copy()
    free = list(free_list[:top])
    plans = []
    fresh_needed = 0
    for b in range(table.shape[0]):
        L = int(seq_lens[b])
        toks = [t for t in range(L) if keep[b, t if token_gran else t // ps]]
        pages = [toks[i:i + ps] for i in range(0, len(toks), ps)]
        plan = []
        for grp in pages:
            j = grp[0] // ps
            if grp == list(range(j * ps, j * ps + len(grp))):
                plan.append(("reuse", j, grp))
            else:
                plan.append(("fresh", None, grp))
                fresh_needed += 1
        plans.append((toks, plan))
    if fresh_needed > len(free):
        return None
    freed = []
    for b, (toks, plan) in enumerate(plans):
        old = table[b].copy()
        row = [-1] * table.shape[1]
        used = set()
        for m, (kind, j, grp) in enumerate(plan):
            if kind == "reuse":
                row[m] = int(old[j])
                used.add(j)
            else:
                page = free.pop()
                row[m] = page
                for s, t in enumerate(grp):
                    k_pool[page, :, s] = k_pool[old[t // ps], :, t % ps]
                    v_pool[page, :, s] = v_pool[old[t // ps], :, t % ps]
        for j in range(-(-int(seq_lens[b]) // ps)):
            if j not in used:
                freed.append(int(old[j]))
        table[b] = row
        seq_lens[b] = len(toks)
    free += freed
    fl = free_list.copy()
    fl[: len(free)] = free
    return table, seq_lens, k_pool, v_pool, fl, len(free)


def pin_compaction():
    rng = np.random.default_rng(14)
    ps, Hkv, d = 16, 2, 8
    for trial in range(8):
        B = 3
        lens = rng.integers(0, 90, size=B).astype(np.int32)
        x = W.small_decode(100 + trial, B=B, Hq=2 * Hkv, Hkv=Hkv, d=d, seq_lens=lens.tolist(),
                           pool_factor=3.0, pad_pages=1)
        token_gran = trial % 2 == 1
        width = x.max_pages * (ps if token_gran else 1)
        keep = (rng.random((B, width)) < 0.6).astype(np.uint8)
        if trial == 2:
            keep[:] = 1
        res = O.compact(x.block_table, x.seq_lens, keep, token_gran, x.k_pool, x.v_pool,
                        x.free_list, x.free_top, Hkv, d, ps)
        ref = _compact_naive(x.block_table, x.seq_lens, keep, token_gran, x.k_pool, x.v_pool,
                             x.free_list, x.free_top, ps)
        assert ref is not None and res[-1] == 0
        t, sl, kp, vp, fl, top, _ = res
        assert np.array_equal(t, ref[0]) and np.array_equal(sl, ref[1])
        assert np.array_equal(kp, ref[2]) and np.array_equal(vp, ref[3])
        assert top == ref[5] and np.array_equal(fl[:top], ref[4][:top])
        # conservation: resident + free = everything that was resident or free
        resident = [int(p) for b in range(B) for p in t[b, : -(-int(sl[b]) // ps)]]
        before = [int(p) for b in range(B) for p in x.block_table[b, : -(-int(x.seq_lens[b]) // ps)]]
        assert sorted(resident + fl[:top].tolist()) == sorted(before + x.free_list[:x.free_top].tolist())
        assert len(set(resident)) == len(resident)
        # kept tokens keep their bytes
        for b in range(B):
            L = int(x.seq_lens[b])
            toks = [tt for tt in range(L) if keep[b, tt if token_gran else tt // ps]]
            for i, tt in enumerate(toks):
                assert np.array_equal(kp[t[b, i // ps], :, i % ps],
                                      x.k_pool[x.block_table[b, tt // ps], :, tt % ps])
    # page-granular masks only rewrite tables: no fresh page, so an empty free
    # list is fine, and the freed pages become the whole free list
    x = W.small_decode(6, B=2, Hq=2, Hkv=1, d=8, seq_lens=[70, 33], pool_factor=1.0)
    keep = np.ones((2, x.max_pages), np.uint8)
    keep[0, [1, 2]] = 0
    keep[1, 0] = 0
    t, sl, kp, vp, fl, top, rc = O.compact(x.block_table, x.seq_lens, keep, False, x.k_pool,
                                           x.v_pool, x.free_list, 0, 1, 8, ps)
    assert rc == 0 and sl.tolist() == [70 - 32, 33 - 16] and top == 3
    assert fl[:3].tolist() == [x.block_table[0, 1], x.block_table[0, 2], x.block_table[1, 0]]
    assert np.array_equal(kp, x.k_pool) and np.array_equal(vp, x.v_pool)
    # exhausted free list: nothing changes
    x = W.small_decode(5, B=1, Hq=2, Hkv=1, d=8, seq_lens=[64], pool_factor=1.0)
    keep = np.zeros((1, x.max_pages * ps), np.uint8)
    keep[0, 1::2] = 1
    res = O.compact(x.block_table, x.seq_lens, keep, True, x.k_pool, x.v_pool, x.free_list, 0,
                    1, 8, ps)
    assert res[-1] == O.ENOSPACE and np.array_equal(res[0], x.block_table)


def _compact_naive_shared(x, keep, token_gran, refcnt, top):
    """Refcounted re-pack written from the definition with Python lists:
    plan as for private pages; fresh pages get one reference; every old page
    not reused loses one reference in (b, j) order and goes back on the free
    list when none is left."""
    ps = x.page_size
    table = x.block_table.copy()
    lens = x.seq_lens.copy()
    kp, vp = x.k_pool.copy(), x.v_pool.copy()
    rc = refcnt.copy()
    free = list(x.free_list[:top])
    out_rows, freed = [], []
    for b in range(x.B):
        L = int(lens[b])
        toks = [t for t in range(L) if keep[b, t if token_gran else t // ps]]
        old = table[b].copy()
        row = [-1] * table.shape[1]
        used = set()
        for m in range(0, len(toks), ps):
            grp = toks[m: m + ps]
            j = grp[0] // ps
            if grp == list(range(j * ps, j * ps + len(grp))):
                row[m // ps] = int(old[j])
                used.add(j)
            else:
                page = free.pop()
                rc[page] = 1
                row[m // ps] = page
                for s_, t in enumerate(grp):
                    kp[page, :, s_] = kp[old[t // ps], :, t % ps]
                    vp[page, :, s_] = vp[old[t // ps], :, t % ps]
        freed += [int(old[j]) for j in range(-(-L // ps)) if j not in used]
        out_rows.append(row)
        lens[b] = len(toks)
    for pg in freed:
        rc[pg] -= 1
        if rc[pg] == 0:
            free.append(pg)
    table[:] = np.array(out_rows, np.int32)
    return table, lens, kp, vp, free, rc


def _refs(table, lens, P, ps=16):
    n = np.zeros(P, np.int64)
    for b in range(table.shape[0]):
        for j in range(-(-int(lens[b]) // ps)):
            n[table[b, j]] += 1
    return n


def pin_shared_pages():
    """Shared (prefix) pages through compaction and append: the oracle against
    a refcounted re-pack written independently, plus the invariants -- a
    page's count equals its block-table references, the free list is exactly
    the unreferenced pages, a page still referenced is never written, and an
    append into a shared partly filled page copies it first."""
    rng = np.random.default_rng(21)
    ps = 16
    for trial in range(8):
        tails = [int(v) for v in rng.integers(0, 60, size=6)]
        tails[trial % 6] = 0
        c = W.shared_prefix(40 + trial, 6, 3, int(rng.integers(17, 60)), tails,
                            pool_factor=3.0)
        x, refcnt = c["decode"], c["refcnt"]
        token_gran = trial % 2 == 1
        width = x.max_pages * (ps if token_gran else 1)
        keep = (rng.random((x.B, width)) < 0.6).astype(np.uint8)
        if trial == 4:
            keep[:] = 0
        rc = refcnt.copy()
        t, sl, kp, vp, fl, top, st = O.compact(x.block_table, x.seq_lens, keep, token_gran,
                                               x.k_pool, x.v_pool, x.free_list, x.free_top,
                                               x.Hkv, x.d, ps, refcnt=rc)
        assert st == 0
        nt, nl, nkp, nvp, nfree, nrc = _compact_naive_shared(x, keep, token_gran, refcnt,
                                                             x.free_top)
        assert np.array_equal(t, nt) and np.array_equal(sl, nl) and np.array_equal(rc, nrc)
        assert np.array_equal(kp, nkp) and np.array_equal(vp, nvp)
        assert top == len(nfree) and fl[:top].tolist() == nfree
        P = x.num_pages
        assert np.array_equal(rc, _refs(t, sl, P))
        assert sorted(fl[:top].tolist()) == sorted(np.nonzero(rc == 0)[0].tolist())
        for pg in np.nonzero(rc > 0)[0]:
            if refcnt[pg] > 0:  # referenced before and after: untouched
                assert np.array_equal(kp[pg], x.k_pool[pg]) and np.array_equal(vp[pg], x.v_pool[pg])
    # append: forks (no own tokens) share the prefix's partly filled page
    c = W.shared_prefix(60, 6, 3, 37, [0, 0, 9, 0, 40, 0], pool_factor=3.0)
    x, refcnt = c["decode"], c["refcnt"]
    kn = W.normal_bits(rng, (x.B, x.Hkv, x.d), W.F16)
    vn = W.normal_bits(rng, (x.B, x.Hkv, x.d), W.F16)
    rc = refcnt.copy()
    kp, vp, t, sl, fl, top, st = O.append(kn, vn, x.k_pool, x.v_pool, x.block_table, x.seq_lens,
                                          x.free_list, x.free_top, x.Hkv, x.d, ps, refcnt=rc)
    assert st == 0 and sl.tolist() == (x.seq_lens + 1).tolist()
    pops, cows, running = 0, 0, refcnt.astype(np.int64).copy()
    for b in range(x.B):
        L = int(x.seq_lens[b])
        j = L // ps
        old = int(x.block_table[b, j]) if L % ps else -1
        if L % ps and running[old] > 1:  # copy-on-write, pops in ascending b
            assert t[b, j] == x.free_list[x.free_top - 1 - pops] != old
            pops += 1
            cows += 1
            running[old] -= 1
            assert np.array_equal(kp[t[b, j], :, : L % ps], x.k_pool[old, :, : L % ps])
            assert np.array_equal(vp[t[b, j], :, : L % ps], x.v_pool[old, :, : L % ps])
        elif L % ps == 0:
            pops += 1
        else:  # sole owner (last sharer after the others copied): in place
            assert t[b, j] == old
        assert np.array_equal(kp[t[b, j], :, L % ps], kn[b])
        assert np.array_equal(vp[t[b, j], :, L % ps], vn[b])
    assert cows == 2 and top == x.free_top - pops  # two fork pairs: the first of each copies
    assert np.array_equal(rc, _refs(t, sl, x.num_pages))
    # every page referenced before the call and still referenced by a
    # sequence that did not write into it is unchanged
    for b in range(x.B):
        for jj in range(-(-int(x.seq_lens[b]) // ps) - 1):
            pg = t[b, jj]
            assert np.array_equal(kp[pg], x.k_pool[pg]) and np.array_equal(vp[pg], x.v_pool[pg])
    # without counts nothing is shared: the page is written in place
    kp2, _, t2, *_ = O.append(kn, vn, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.free_list,
                              x.free_top, x.Hkv, x.d, ps)
    assert t2[0, 2] == x.block_table[0, 2]


def pin_append():
    ps, Hkv, d = 16, 2, 8
    x = W.small_decode(31, B=4, Hq=4, Hkv=Hkv, d=d, seq_lens=[16, 5, 32, 0], pool_factor=2.0,
                       pad_pages=2)
    rng = np.random.default_rng(15)
    kn = W.normal_bits(rng, (4, Hkv, d), W.F16)
    vn = W.normal_bits(rng, (4, Hkv, d), W.F16)
    kp, vp, t, sl, fl, top, rc = O.append(kn, vn, x.k_pool, x.v_pool, x.block_table, x.seq_lens,
                                          x.free_list, x.free_top, Hkv, d, ps)
    assert rc == 0 and sl.tolist() == [17, 6, 33, 1]
    # pops in ascending b for rows at a page boundary (b = 0, 2, 3)
    top0 = x.free_top
    assert t[0, 1] == x.free_list[top0 - 1] and t[2, 2] == x.free_list[top0 - 2]
    assert t[3, 0] == x.free_list[top0 - 3] and top == top0 - 3
    for b, L in enumerate([16, 5, 32, 0]):
        assert np.array_equal(kp[t[b, L // ps], :, L % ps], kn[b])
        assert np.array_equal(vp[t[b, L // ps], :, L % ps], vn[b])
    # rows full / free list empty -> error, no change
    *_, rc = O.append(kn, vn, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.free_list, 2,
                      Hkv, d, ps)
    assert rc == O.ENOSPACE
    full = x.seq_lens.copy()
    full[1] = x.max_pages * ps
    *_, rc = O.append(kn, vn, x.k_pool, x.v_pool, x.block_table, full, x.free_list, x.free_top,
                      Hkv, d, ps)
    assert rc == O.EFULL


def pin_mark_active():
    lens = np.array([0, 16, 32, 33, 48, 160], np.int32)
    bud = np.array([0, 1, 3, 2, 2, 20], np.int32)
    assert O.mark_active(lens, bud, 16, 0).tolist() == [0, 0, 0, 1, 1, 0]
    assert O.mark_active(lens, bud, 16, 1).tolist() == [0, 1, 0, 0, 1, 0]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
