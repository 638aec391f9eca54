"""GPU parity of the budgeting kernels against the oracle: bit-exact for
every integer decision and every fp32 value that feeds one."""
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_kv_cache_492_b300 import budget as BG
from paged_kv_cache_492_b300 import kv
from paged_kv_cache_492_b300 import workloads as W
from tests.budget_oracle import OracleBudget
from tests.decision_check import DecisionAnchor
from tests.gpu_util import DeviceDecode, assert_decode_close, bits_to_dev, i32

pytestmark = pytest.mark.gpu
NCPU = len(os.sched_getaffinity(0))
DEV = "cuda"


def f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("G,d", [(4, 128), (4, 64), (1, 128), (8, 64)])
def test_ema_bit_exact(dtype, G, d):
    rng = np.random.default_rng(1)
    B, Hkv = 5, 2
    Hq = G * Hkv
    ema_ref = np.zeros((B, 2, Hkv, d), np.float32)
    ema = torch.zeros((B, 2, Hkv, d), dtype=torch.float32, device=DEV)
    for t in range(6):
        q = W.normal_bits(rng, (B, Hq, d), dtype)
        O.ema_f32(q, B, Hq, Hkv, d, dtype, 0.9, 0.999, t == 0, ema_ref)
        kv.kv_update_query_summaries(bits_to_dev(q, dtype), Hkv, 0.9, 0.999, t == 0, ema)
    assert np.array_equal(ema.cpu().numpy(), ema_ref)


def test_mark_active_exact():
    rng = np.random.default_rng(2)
    lens = rng.integers(0, 5000, size=300).astype(np.int32)
    lens[::7] = (lens[::7] // 16) * 16
    bud = rng.integers(0, 300, size=300).astype(np.int32)
    act = torch.zeros(300, dtype=torch.uint8, device=DEV)
    for mode in (0, 1):
        kv.kv_mark_active(i32(lens), i32(bud), 16, mode, act)
        assert np.array_equal(act.cpu().numpy(), O.mark_active(lens, bud, 16, mode))


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
def test_page_summaries_bit_exact(dtype):
    rng = np.random.default_rng(3)
    P, Hkv, d = 40, 8, 128
    kp = W.normal_bits(rng, (P, Hkv, 16, d), dtype)
    ids = rng.permutation(P)[:17].astype(np.int32)
    ref = np.zeros((P, Hkv, 3, d), np.float32)
    O.page_summaries_f32(kp, ids, Hkv, 16, d, dtype, ref)
    summ = torch.zeros((P, Hkv, 3, d), dtype=torch.float32, device=DEV)
    ws = kv.alloc_workspace(256)
    kdev = bits_to_dev(kp, dtype)
    kv.kv_page_summaries(kdev, i32(ids), summ, ws)
    assert kv.kv_get_status(ws) == 0
    assert np.array_equal(summ.cpu().numpy(), ref)
    # last full page of active sequences
    table = rng.permutation(P)[:24].reshape(3, 8).astype(np.int32)
    lens = np.array([32, 100, 128], np.int32)
    act = np.array([1, 1, 0], np.uint8)
    summ.zero_()
    kv.kv_summarize_last_pages(kdev, i32(table), i32(lens), u8(act), summ, ws)
    ref2 = np.zeros_like(ref)
    O.page_summaries_f32(kp, np.array([table[0, 1], table[1, 5]], np.int32), Hkv, 16, d, dtype, ref2)
    assert np.array_equal(summ.cpu().numpy(), ref2)
    # a bad id is reported, nothing read out of bounds
    kv.kv_page_summaries(kdev, i32([0, P + 3]), summ, ws)
    assert kv.kv_get_status(ws) == kv.KV_EBADPAGE


@pytest.mark.parametrize("d", [128, 64])
def test_scores_bit_exact(d):
    rng = np.random.default_rng(4)
    B, Hkv, P, maxp = 6, 8, 60, 9
    ema = rng.standard_normal((B, 2, Hkv, d)).astype(np.float32)
    kp = W.normal_bits(rng, (P, Hkv, 16, d), W.BF16)
    summ = np.zeros((P, Hkv, 3, d), np.float32)
    O.page_summaries_f32(kp, np.arange(P, dtype=np.int32), Hkv, 16, d, W.BF16, summ)
    lens = np.array([0, 1, 16, 17, 140, 144], np.int32)
    table = np.full((B, maxp), -1, np.int32)
    perm = rng.permutation(P)
    pos = 0
    for b, L in enumerate(lens):
        n = -(-int(L) // 16)
        table[b, :n] = perm[pos:pos + n]
        pos += n
    act = np.array([1, 1, 1, 0, 1, 1], np.uint8)
    ref = np.full((B, maxp, 2), 7.0, np.float32)
    O.score_pages_f32(ema, summ, table, lens, act, Hkv, d, 16, ref)
    sc = torch.full((B, maxp, 2), 7.0, dtype=torch.float32, device=DEV)
    ws = kv.alloc_workspace(256)
    kv.kv_score_pages(f32(ema), f32(summ), i32(table), i32(lens), u8(act), sc, ws)
    assert kv.kv_get_status(ws) == 0
    got = sc.cpu().numpy()
    assert np.array_equal(got, ref)
    # and the fp32 scores sit within rounding of the fp64 definition
    r64 = np.zeros((B, maxp, 2))
    O.score_pages_f64(ema.astype(np.float64), summ.astype(np.float64), table, lens, act, Hkv, d,
                      16, r64)
    fin = np.isfinite(ref) & (ref != 7.0)
    assert np.allclose(got[fin], r64[fin], rtol=1e-4, atol=1e-3)


def _run_select(scores, lens, act, budget, mode, free_top, n_first=2, n_last=2, delta=0.5,
                ws_frac=0.5):
    B, maxp, _ = scores.shape
    keep = torch.zeros((B, maxp), dtype=torch.uint8, device=DEV)
    grow = torch.zeros(B, dtype=torch.uint8, device=DEV)
    drift = torch.zeros(B, dtype=torch.int32, device=DEV)
    bud = i32(budget)
    ws = kv.alloc_workspace(kv.kv_select_workspace_size(B, maxp))
    kv.kv_select_pages(f32(scores), i32(lens), None if act is None else u8(act), bud, n_first,
                       n_last, delta, ws_frac, mode, i32([free_top]), keep, grow, drift, ws)
    assert kv.kv_get_status(ws) == 0
    return keep.cpu().numpy(), grow.cpu().numpy(), bud.cpu().numpy(), drift.cpu().numpy()


@pytest.mark.parametrize("trial", range(6))
def test_select_bit_exact(trial):
    rng = np.random.default_rng(10 + trial)
    B, maxp = 12, 300
    lens = rng.integers(0, maxp * 16, size=B).astype(np.int32)
    lens[:4] = (lens[:4] // 16) * 16
    sc = rng.standard_normal((B, maxp, 2)).astype(np.float32)
    if trial % 2:
        sc = np.round(sc * 2) / 2          # many exact ties
    if trial == 3:
        sc[:, :, 1] = sc[:, :, 0]          # no drift
    act = (rng.random(B) < 0.7).astype(np.uint8)
    budget = rng.integers(0, 200, size=B).astype(np.int32)
    for mode, free in ((O.SELECT_TOPK, 0), (O.SELECT_BOUNDARY, 2), (O.SELECT_BOUNDARY, 100)):
        for ws_frac, delta in ((0.5, 0.5), (0.25, 0.3)):
            ref = O.select_pages(sc, lens, act, budget, 16, 2, 2, delta, mode, free, ws_frac=ws_frac)
            got = _run_select(sc, lens, act, budget, mode, free, delta=delta, ws_frac=ws_frac)
            for r, g, name in zip(ref, got, ("keep", "grow", "budget", "drift")):
                assert np.array_equal(r, g), (name, mode, free)


@pytest.mark.parametrize("trial", range(3))
def test_select_bit_exact_long_rows(trial):
    """Rows above 1024 pages (the sorted ranking) and short ones (the counted
    one) side by side, with exact ties and signed zeros among the keys."""
    rng = np.random.default_rng(40 + trial)
    B, maxp = 6, 2500
    lens = rng.integers(1000 * 16, maxp * 16, size=B).astype(np.int32)
    lens[0] = 700 * 16
    lens[1:3] = (lens[1:3] // 16) * 16
    sc = rng.standard_normal((B, maxp, 2)).astype(np.float32)
    if trial >= 1:
        sc = np.round(sc * 2) / 2
    if trial == 2:
        zero = rng.random((B, maxp, 2)) < 0.3
        sc[zero] = np.where(rng.random(zero.sum()) < 0.5, np.float32(-0.0), np.float32(0.0))
    act = np.ones(B, dtype=np.uint8)
    budget = rng.integers(100, 2400, size=B).astype(np.int32)
    for mode, free in ((O.SELECT_TOPK, 0), (O.SELECT_BOUNDARY, 1)):
        ref = O.select_pages(sc, lens, act, budget, 16, 2, 2, 0.5, mode, free, ws_frac=0.5)
        got = _run_select(sc, lens, act, budget, mode, free, delta=0.5, ws_frac=0.5)
        for r, g, name in zip(ref, got, ("keep", "grow", "budget", "drift")):
            assert np.array_equal(r, g), (name, mode, free)


def _compact_case(seed, token_granular, free_top=None):
    rng = np.random.default_rng(seed)
    B = 5
    lens = rng.integers(0, 200, size=B).astype(np.int32)
    lens[0] = 0
    x = W.small_decode(seed, B, 8, 2, 64, lens.tolist(), pool_factor=3.0, pad_pages=2)
    width = x.max_pages * (16 if token_granular else 1)
    keep = (rng.random((B, width)) < 0.55).astype(np.uint8)
    top = x.free_top if free_top is None else free_top
    return x, keep, top


@pytest.mark.parametrize("seed,token_granular", [(1, False), (2, False), (3, True), (4, True),
                                                 (5, True)])
def test_compact_bit_exact(seed, token_granular):
    x, keep, top = _compact_case(seed, token_granular)
    ref = O.compact(x.block_table, x.seq_lens, keep, token_granular, x.k_pool, x.v_pool,
                    x.free_list, top, x.Hkv, x.d, 16)
    assert ref[-1] == 0
    dd = DeviceDecode(x)
    fl = i32(x.free_list)
    ft = i32([top])
    ws = kv.alloc_workspace(kv.kv_compact_workspace_size(x.B, x.max_pages, 0, token_granular))
    kv.kv_compact(dd.table, dd.lens, u8(keep), token_granular, dd.k, dd.v, fl, ft, ws)
    assert kv.kv_get_status(ws) == 0
    t, sl, kp, vp, fl_ref, top_ref, _ = ref
    assert np.array_equal(dd.table.cpu().numpy(), t)
    assert np.array_equal(dd.lens.cpu().numpy(), sl)
    assert int(ft.item()) == top_ref
    assert np.array_equal(fl.cpu().numpy()[:top_ref], fl_ref[:top_ref])
    assert np.array_equal(dd.k.view(torch.int16).cpu().numpy().view(np.uint16), kp)
    assert np.array_equal(dd.v.view(torch.int16).cpu().numpy().view(np.uint16), vp)


def test_compact_no_space_changes_nothing():
    x, keep, _ = _compact_case(7, True)
    dd = DeviceDecode(x)
    t0 = dd.table.clone()
    fl = i32(x.free_list)
    ft = i32([0])
    ws = kv.alloc_workspace(kv.kv_compact_workspace_size(x.B, x.max_pages, 0, True))
    ref = O.compact(x.block_table, x.seq_lens, keep, True, x.k_pool, x.v_pool, x.free_list, 0,
                    x.Hkv, x.d, 16)
    kv.kv_compact(dd.table, dd.lens, u8(keep), True, dd.k, dd.v, fl, ft, ws)
    rc = kv.kv_get_status(ws)
    if ref[-1] == O.ENOSPACE:
        assert rc == kv.KV_ENOSPACE and torch.equal(dd.table, t0)
    else:
        assert rc == 0


def test_append_bit_exact_and_errors():
    rng = np.random.default_rng(8)
    x = W.small_decode(9, 6, 8, 2, 128, [16, 5, 32, 0, 47, 48], pool_factor=2.0, pad_pages=2)
    kn = W.normal_bits(rng, (6, 2, 128), W.F16)
    vn = W.normal_bits(rng, (6, 2, 128), W.F16)
    ref = O.append(kn, vn, x.k_pool, x.v_pool, x.block_table, x.seq_lens, x.free_list, x.free_top,
                   2, 128, 16)
    assert ref[-1] == 0
    dd = DeviceDecode(x)
    fl, ft = i32(x.free_list), i32([x.free_top])
    ws = kv.alloc_workspace(kv.kv_append_workspace_size(6))
    kv.kv_append(bits_to_dev(kn, W.F16), bits_to_dev(vn, W.F16), dd.k, dd.v, dd.table, dd.lens, fl,
                 ft, ws)
    assert kv.kv_get_status(ws) == 0
    kp, vp, t, sl, flr, top, _ = ref
    assert np.array_equal(dd.table.cpu().numpy(), t) and np.array_equal(dd.lens.cpu().numpy(), sl)
    assert int(ft.item()) == top
    assert np.array_equal(dd.k.view(torch.int16).cpu().numpy().view(np.uint16), kp)
    assert np.array_equal(dd.v.view(torch.int16).cpu().numpy().view(np.uint16), vp)
    # too few free pages: error, no change
    t0, l0 = dd.table.clone(), dd.lens.clone()
    kv.kv_append(bits_to_dev(kn, W.F16), bits_to_dev(vn, W.F16), dd.k, dd.v, dd.table, dd.lens, fl,
                 i32([0]), ws)
    assert kv.kv_get_status(ws) == kv.KV_ENOSPACE
    assert torch.equal(dd.table, t0) and torch.equal(dd.lens, l0)
    # a full row: error, no change
    full = dd.lens.clone()
    full[0] = 16 * x.max_pages
    kv.kv_append(bits_to_dev(kn, W.F16), bits_to_dev(vn, W.F16), dd.k, dd.v, dd.table, full, fl,
                 ft, ws)
    assert kv.kv_get_status(ws) == kv.KV_EFULL


def test_tiny_selection_pipeline():
    """Tiny workload: EMAs over 32 prior queries, page summaries, scores and
    keep-8-of-16, against the oracle bit for bit; then the fp64 definition
    picks the same 8 pages."""
    c = W.tiny()
    x = c["decode"]
    B, Hq, Hkv, d = x.B, x.Hq, x.Hkv, x.d
    ema = torch.zeros((B, 2, Hkv, d), dtype=torch.float32, device=DEV)
    ref = np.zeros((B, 2, Hkv, d), np.float32)
    ref64 = np.zeros((B, 2, Hkv, d))
    for t in range(32):
        q = c["prior_q"][t]
        kv.kv_update_query_summaries(bits_to_dev(q, W.F16), Hkv, c["a_fast"], c["a_slow"], t == 0, ema)
        O.ema_f32(q, B, Hq, Hkv, d, W.F16, c["a_fast"], c["a_slow"], t == 0, ref)
        O.ema_f64(q, B, Hq, Hkv, d, W.F16, c["a_fast"], c["a_slow"], t == 0, ref64)
    assert np.array_equal(ema.cpu().numpy(), ref)
    dd = DeviceDecode(x)
    summ = torch.zeros((x.num_pages, Hkv, 3, d), dtype=torch.float32, device=DEV)
    ws = kv.alloc_workspace(kv.kv_select_workspace_size(B, 16))
    kv.kv_page_summaries(dd.k, i32(x.block_table[0]), summ, ws)
    sref = np.zeros((x.num_pages, Hkv, 3, d), np.float32)
    O.page_summaries_f32(x.k_pool, x.block_table[0], Hkv, 16, d, W.F16, sref)
    assert np.array_equal(summ.cpu().numpy(), sref)
    sc = torch.zeros((B, 16, 2), dtype=torch.float32, device=DEV)
    kv.kv_score_pages(ema, summ, dd.table, dd.lens, None, sc, ws)
    scr = np.zeros((B, 16, 2), np.float32)
    O.score_pages_f32(ref, sref, x.block_table, x.seq_lens, None, Hkv, d, 16, scr)
    assert np.array_equal(sc.cpu().numpy(), scr)
    keep, grow, bud, _ = _run_select(scr, x.seq_lens, None, [8], O.SELECT_TOPK, 0, 0, 0)
    kref, *_ = O.select_pages(scr, x.seq_lens, None, [8], 16, 0, 0, 0.5, O.SELECT_TOPK, 0)
    assert np.array_equal(keep, kref) and keep.sum() == 8
    # the fp64 definition keeps the same 8 pages, with the margin at the cut
    # above the certified fp32 error bound
    anchor = DecisionAnchor(B, Hq, Hkv, d, x.num_pages, W.F16, c["a_fast"], c["a_slow"])
    for t in range(32):
        anchor.update_ema(c["prior_q"][t], t == 0)
    anchor.summarize(x.k_pool, x.block_table[0])
    st = anchor.check(table=x.block_table, lens=x.seq_lens, active=None, budget=np.array([8]),
                      free_count=0, mode=O.SELECT_TOPK, n_first=0, n_last=0, delta=0.5,
                      ws_frac=0.5, ema32=ref, summ32=sref, scores32=scr, keep=keep, grow=grow,
                      drift=np.zeros(B, np.int32), budget_after=bud, tag="tiny")
    assert st.decisions == 1 and st.near_ties == 0, st.log


@pytest.mark.parametrize("engine", [kv.KV_DECODE_TENSOR_CORE, 0], ids=["tensor_core", "fused"])
def test_budgeted_serving_trajectory(engine):
    """Batch-64 budgeted decode: the fit, then every step's compress-or-grow,
    append and block-table state bit-exact against the oracle's trajectory.
    Every step is also checked differentially: the oracle decodes the GPU's
    input state for the sequences that compacted, grew or took a fresh page
    that step plus 8 others drawn at random (the whole batch every 16 steps),
    on the decode engine given.  With the tensor-core engine (the one the
    bench picks) every budgeting decision is also checked against the fp64
    definition: equal wherever its margin clears the fp32 error bound, and
    near-ties reported."""
    # all 128 steps with the fp64 anchor on the tensor-core engine, 64 on the other
    steps = int(os.environ.get("KV_BUDGET_STEPS",
                               "128" if engine == kv.KV_DECODE_TENSOR_CORE else "64"))
    c = W.budgeted_serving(steps=steps)
    x = c["decode"]
    cfg = BG.BudgetConfig(a_fast=c["a_fast"], a_slow=c["a_slow"], n_first=c["n_first"],
                          n_last=c["n_last"], delta=c["delta"])
    anchor = (DecisionAnchor(x.B, x.Hq, x.Hkv, x.d, x.num_pages, x.dtype, c["a_fast"],
                             c["a_slow"]) if engine == kv.KV_DECODE_TENSOR_CORE else None)
    orc = OracleBudget(x, c["budget"], cfg, anchor=anchor)
    orc.summarize_all()
    dd = DeviceDecode(x)
    dec = BG.BudgetedDecoder(dd.k, dd.v, dd.table, dd.lens, i32(x.free_list), i32([x.free_top]),
                             i32(c["budget"]), x.Hq, cfg, pages_per_split=engine)
    dec.summarize_pages(i32(np.arange(x.num_pages)))
    q0, _, _ = W.step_tokens(c["seed"], 0, x.B, x.Hq, x.Hkv, x.d, x.dtype)
    dec.fit(bits_to_dev(q0, x.dtype))
    orc.fit(q0)

    def check_state(where):
        assert dec.status() == 0, where
        assert np.array_equal(dec.table.cpu().numpy(), orc.table), where
        assert np.array_equal(dec.lens.cpu().numpy(), orc.lens), where
        assert np.array_equal(dec.budget.cpu().numpy(), orc.budget), where
        top = int(dec.free_top.item())
        assert top == int(orc.top[0]), where
        assert np.array_equal(dec.free_list.cpu().numpy()[:top], orc.free_list[:top]), where
        assert np.array_equal(dec.ema.cpu().numpy(), orc.ema), where

    def check_decisions(where):
        if anchor is None:
            return
        pre = orc.pre
        anchor.check(table=pre["table"], lens=pre["lens"], active=pre["active"],
                     budget=pre["budget"], free_count=pre["free_count"], mode=pre["mode"],
                     n_first=cfg.n_first, n_last=cfg.n_last, delta=cfg.delta,
                     ws_frac=cfg.ws_frac, ema32=orc.ema, summ32=orc.summ,
                     scores32=dec.scores.cpu().numpy(), keep=dec.keep.cpu().numpy(),
                     grow=dec.grow.cpu().numpy(), drift=dec.drift.cpu().numpy(),
                     budget_after=dec.budget.cpu().numpy(), tag=where)

    check_state("fit")
    check_decisions("fit")
    rng = np.random.default_rng(1234)
    grows = compacts = checked_rows = 0
    for t in range(steps):
        q, kn, vn = W.step_tokens(c["seed"], t, x.B, x.Hq, x.Hkv, x.d, x.dtype)
        dec.step(bits_to_dev(q, x.dtype), bits_to_dev(kn, x.dtype), bits_to_dev(vn, x.dtype), t)
        orc.step(q, kn, vn, t)
        check_state(f"step {t}")
        act = orc.active.astype(bool)
        assert np.array_equal(dec.active.cpu().numpy(), orc.active)
        assert np.array_equal(dec.grow.cpu().numpy()[act], orc.grow[act])
        assert np.array_equal(dec.drift.cpu().numpy()[act], orc.drift[act])
        check_decisions(f"step {t}")
        grows += int(orc.grow[act].sum())
        compacts += int(act.sum() - orc.grow[act].sum())
        # decode on the GPU's input state, every step
        y = orc.decode_inputs(q)
        out = dec.out.cpu().numpy().astype(np.float64)
        lse = dec.lse.cpu().numpy().astype(np.float64)
        if t % 16 == 15 or t == steps - 1:
            ref_out, ref_lse = O.decode(y, nthreads=NCPU)
            assert_decode_close(y, out, lse, ref_out, ref_lse)
            checked_rows += x.B
        else:
            others = [b for b in range(x.B) if b not in orc.changed]
            seqs = sorted(set(orc.changed) |
                          set(rng.choice(others, size=min(8, len(others)), replace=False).tolist()))
            ys = W.DecodeInputs(**{**y.__dict__, "B": len(seqs), "q": y.q[seqs],
                                   "block_table": y.block_table[seqs], "seq_lens": y.seq_lens[seqs]})
            ref_out, ref_lse = O.decode(ys, nthreads=NCPU)
            assert_decode_close(ys, out[seqs], lse[seqs], ref_out, ref_lse)
            checked_rows += len(seqs)
    print(f"budgeted serving ({'tensor-core' if engine else 'fused'} decode): {steps} steps, "
          f"{grows} grows, {compacts} compactions, {checked_rows} sequence decodes checked")
    if anchor is not None:
        print(f"fp64 anchor: {anchor.stats.summary()}")
        for line in anchor.stats.log:
            print("  " + line)
    assert grows > 0 and compacts > 0


# ---------------------------------------------------------------- shared pages
def _shared_case(seed, tails, prefix=37):
    c = W.shared_prefix(seed, len(tails), 3, prefix, tails, pool_factor=3.0)
    return c["decode"], c["refcnt"]


@pytest.mark.parametrize("seed,token_granular", [(51, False), (52, True), (53, False), (54, True)])
def test_compact_shared_bit_exact(seed, token_granular):
    """Refcounted compaction: counts, free list (a page returns when its last
    reference goes), tables and pools bit for bit against the oracle."""
    rng = np.random.default_rng(seed)
    tails = [int(v) for v in rng.integers(0, 80, size=9)]
    tails[seed % 9] = 0
    x, refcnt = _shared_case(seed, tails, prefix=int(rng.integers(17, 70)))
    width = x.max_pages * (16 if token_granular else 1)
    keep = (rng.random((x.B, width)) < 0.5).astype(np.uint8)
    rc_ref = refcnt.copy()
    t, sl, kp, vp, fl, top, st = O.compact(x.block_table, x.seq_lens, keep, token_granular,
                                           x.k_pool, x.v_pool, x.free_list, x.free_top, x.Hkv,
                                           x.d, 16, refcnt=rc_ref)
    assert st == 0
    dd = DeviceDecode(x)
    fl_d, ft_d, rc_d = i32(x.free_list), i32([x.free_top]), i32(refcnt)
    ws = kv.alloc_workspace(kv.kv_compact_workspace_size(x.B, x.max_pages, x.num_pages,
                                                         token_granular))
    kv.kv_compact(dd.table, dd.lens, u8(keep), token_granular, dd.k, dd.v, fl_d, ft_d, ws,
                  refcnt=rc_d)
    assert kv.kv_get_status(ws) == 0
    assert np.array_equal(dd.table.cpu().numpy(), t)
    assert np.array_equal(dd.lens.cpu().numpy(), sl)
    assert np.array_equal(rc_d.cpu().numpy(), rc_ref)
    assert int(ft_d.item()) == top
    assert np.array_equal(fl_d.cpu().numpy()[:top], fl[:top])
    assert np.array_equal(dd.k.view(torch.int16).cpu().numpy().view(np.uint16), kp)
    assert np.array_equal(dd.v.view(torch.int16).cpu().numpy().view(np.uint16), vp)


def test_append_shared_bit_exact():
    """Copy-on-write append of forks sharing a partly filled prefix page."""
    rng = np.random.default_rng(61)
    x, refcnt = _shared_case(61, [0, 0, 9, 0, 40, 0, 0, 0, 0], prefix=37)
    kn = W.normal_bits(rng, (x.B, x.Hkv, x.d), W.F16)
    vn = W.normal_bits(rng, (x.B, x.Hkv, x.d), W.F16)
    rc_ref = refcnt.copy()
    kp, vp, t, sl, fl, top, st = O.append(kn, vn, x.k_pool, x.v_pool, x.block_table, x.seq_lens,
                                          x.free_list, x.free_top, x.Hkv, x.d, 16, refcnt=rc_ref)
    assert st == 0
    dd = DeviceDecode(x)
    fl_d, ft_d, rc_d = i32(x.free_list), i32([x.free_top]), i32(refcnt)
    ws = kv.alloc_workspace(kv.kv_append_workspace_size(x.B))
    kv.kv_append(bits_to_dev(kn, W.F16), bits_to_dev(vn, W.F16), dd.k, dd.v, dd.table, dd.lens,
                 fl_d, ft_d, ws, refcnt=rc_d)
    assert kv.kv_get_status(ws) == 0
    assert np.array_equal(dd.table.cpu().numpy(), t) and np.array_equal(dd.lens.cpu().numpy(), sl)
    assert np.array_equal(rc_d.cpu().numpy(), rc_ref) and int(ft_d.item()) == top
    assert np.array_equal(dd.k.view(torch.int16).cpu().numpy().view(np.uint16), kp)
    assert np.array_equal(dd.v.view(torch.int16).cpu().numpy().view(np.uint16), vp)
    assert (refcnt > 1).sum() > 0 and not np.array_equal(t, x.block_table)  # forks copied


def test_budgeted_shared_prefix_trajectory():
    """Budgeted decode over sequences that share prompt prefixes: 48 steps of
    compress-or-grow, copy-on-write appends and decode, every table, count,
    free list and EMA bit-exact against the oracle; decode within tolerance."""
    rng = np.random.default_rng(71)
    B, steps = 12, 48
    tails = [int(v) for v in rng.integers(200, 1200, size=B)]
    tails[0] = tails[4] = 0           # forks sharing the partial prefix page
    c = W.shared_prefix(71, B, 4, 700, tails, Hq=32, Hkv=8, d=128, dtype=W.BF16, pool_factor=1.6)
    x, refcnt = c["decode"], c["refcnt"]
    budget = rng.integers(20, 60, size=B).astype(np.int32)
    cfg = BG.BudgetConfig(a_fast=0.9, a_slow=0.999, n_first=2, n_last=2, delta=0.5)
    orc = OracleBudget(x, budget, cfg, refcnt=refcnt)
    orc.summarize_all()
    dd = DeviceDecode(x)
    dec = BG.BudgetedDecoder(dd.k, dd.v, dd.table, dd.lens, i32(x.free_list), i32([x.free_top]),
                             i32(budget), x.Hq, cfg, refcnt=i32(refcnt))
    dec.summarize_pages(i32(np.arange(x.num_pages)))
    q0, _, _ = W.step_tokens(71, 0, x.B, x.Hq, x.Hkv, x.d, x.dtype)
    dec.fit(bits_to_dev(q0, x.dtype))
    orc.fit(q0)

    def check(where):
        assert dec.status() == 0, where
        assert np.array_equal(dec.table.cpu().numpy(), orc.table), where
        assert np.array_equal(dec.lens.cpu().numpy(), orc.lens), where
        assert np.array_equal(dec.refcnt.cpu().numpy(), orc.refcnt), where
        top = int(dec.free_top.item())
        assert top == int(orc.top[0]), where
        assert np.array_equal(dec.free_list.cpu().numpy()[:top], orc.free_list[:top]), where

    check("fit")
    for t in range(steps):
        q, kn, vn = W.step_tokens(71, t, x.B, x.Hq, x.Hkv, x.d, x.dtype)
        dec.step(bits_to_dev(q, x.dtype), bits_to_dev(kn, x.dtype), bits_to_dev(vn, x.dtype), t)
        orc.step(q, kn, vn, t)
        check(f"step {t}")
        if t % 12 == 11:
            y = orc.decode_inputs(q)
            ref_out, ref_lse = O.decode(y, nthreads=NCPU)
            assert_decode_close(y, dec.out.cpu().numpy().astype(np.float64),
                                dec.lse.cpu().numpy().astype(np.float64), ref_out, ref_lse)
    assert (orc.refcnt > 1).any()  # some pages are still shared at the end


def test_budgeted_step_graphed_matches_eager():
    """The steady-state step replayed from CUDA graphs gives the same state
    and outputs, bit for bit, as the same steps issued call by call."""
    steps = 24
    c = W.budgeted_serving(steps=steps + 1)
    x = c["decode"]
    cfg = BG.BudgetConfig(a_fast=c["a_fast"], a_slow=c["a_slow"], n_first=c["n_first"],
                          n_last=c["n_last"], delta=c["delta"])
    decs = []
    for _ in range(2):
        dd = DeviceDecode(x)
        dec = BG.BudgetedDecoder(dd.k, dd.v, dd.table, dd.lens, i32(x.free_list),
                                 i32([x.free_top]), i32(c["budget"]), x.Hq, cfg)
        dec.summarize_pages(i32(np.arange(x.num_pages)))
        q0, _, _ = W.step_tokens(c["seed"], 0, x.B, x.Hq, x.Hkv, x.d, x.dtype)
        dec.fit(bits_to_dev(q0, x.dtype))
        decs.append(dec)
    eager, graphed = decs
    toks = [tuple(bits_to_dev(a, x.dtype) for a in W.step_tokens(c["seed"], t, x.B, x.Hq, x.Hkv,
                                                                   x.d, x.dtype))
            for t in range(steps + 1)]
    for dec in decs:
        dec.step(*toks[0], 0)
    graphed.capture()
    for t in range(1, steps + 1):
        eager.step(*toks[t], t)
        if t % 2:
            graphed.step_graphed(*toks[t])
        else:  # the token packed into the graphs' input buffer in one copy
            graphed.step_graphed_packed(graphed.pack_token(*toks[t]))
        torch.cuda.synchronize()
        for name in ("table", "lens", "free_top", "ema", "keep", "grow", "active", "out", "lse"):
            a, b = getattr(eager, name), getattr(graphed, name)
            assert torch.equal(a, b), (t, name)
        top = int(eager.free_top.item())
        assert torch.equal(eager.free_list[:top], graphed.free_list[:top]), t
        assert torch.equal(eager.k_pool, graphed.k_pool) and torch.equal(eager.v_pool, graphed.v_pool), t
    for dec in decs:
        assert dec.status() == 0


# ------------------------------------------------------------- fused step
_STATE = ("table", "lens", "budget", "free_top", "ema", "summ", "keep", "grow", "drift", "active",
          "k_pool", "v_pool", "out", "lse")


def _pair(x, budget, cfg, pages_per_split=0):
    decs = []
    for fused in (True, False):
        dd = DeviceDecode(x)
        dec = BG.BudgetedDecoder(dd.k, dd.v, dd.table, dd.lens, i32(x.free_list),
                                 i32([x.free_top]), i32(budget), x.Hq, cfg,
                                 pages_per_split=pages_per_split, fused_step=fused)
        dec.summarize_pages(i32(np.arange(x.num_pages)))
        decs.append(dec)
    return decs


def _same(a, b, where, outputs=True):
    for name in _STATE if outputs else _STATE[:-2]:
        assert torch.equal(getattr(a, name), getattr(b, name)), (where, name)
    act = a.active.bool()
    assert torch.equal(a.scores[act], b.scores[act]), (where, "scores")
    top = int(a.free_top.item())
    assert torch.equal(a.free_list[:top], b.free_list[:top]), (where, "free_list")
    assert a.status() == b.status(), where


def test_fused_step_matches_the_calls():
    """kv_budget_step (one launch) against the seven calls it replaces, on the
    batch-64 budgeted workload: the whole state, bit for bit, every step."""
    steps = 24
    c = W.budgeted_serving(steps=steps)
    x = c["decode"]
    cfg = BG.BudgetConfig(a_fast=c["a_fast"], a_slow=c["a_slow"], n_first=c["n_first"],
                          n_last=c["n_last"], delta=c["delta"])
    fused, calls = _pair(x, c["budget"], cfg)
    q0, _, _ = W.step_tokens(c["seed"], 0, x.B, x.Hq, x.Hkv, x.d, x.dtype)
    for dec in (fused, calls):
        dec.fit(bits_to_dev(q0, x.dtype))
    _same(fused, calls, "fit", outputs=False)  # nothing decoded yet
    grows = 0
    for t in range(steps):
        toks = [bits_to_dev(a, x.dtype)
                for a in W.step_tokens(c["seed"], t, x.B, x.Hq, x.Hkv, x.d, x.dtype)]
        for dec in (fused, calls):
            dec.step(*toks, t)
        torch.cuda.synchronize()
        _same(fused, calls, f"step {t}")
        grows += int(fused.grow[fused.active.bool()].sum())
    assert grows > 0


@pytest.mark.parametrize("dtype,d,free_top", [(W.F16, 64, 2), (W.BF16, 128, 0)])
def test_fused_step_grants_run_out(dtype, d, free_top):
    """Every row at a capacity boundary wants to grow (delta < 0); the free
    list grants the first `free_top` rows and the rest are compacted by the
    last block; the appends then take the freed pages.  Same state as the
    separate calls."""
    lens = [16 * 9, 16 * 12, 16 * 7, 16 * 30, 16 * 10, 16 * 8]
    budget = np.array([9, 12, 7, 30, 10, 8], np.int32)
    x = W.small_decode(91, len(lens), 8, 2, d, lens, dtype=dtype, pool_factor=1.3, pad_pages=3)
    assert x.free_top >= free_top
    x.free_top = free_top  # only the bottom `free_top` free pages are offered
    cfg = BG.BudgetConfig(a_fast=0.9, a_slow=0.999, n_first=2, n_last=2, delta=-1.0)
    fused, calls = _pair(x, budget, cfg)
    rng = np.random.default_rng(5)
    for t in range(3):
        q = bits_to_dev(W.normal_bits(rng, (x.B, x.Hq, d), dtype), dtype)
        kn = bits_to_dev(W.normal_bits(rng, (x.B, x.Hkv, d), dtype), dtype)
        vn = bits_to_dev(W.normal_bits(rng, (x.B, x.Hkv, d), dtype), dtype)
        for dec in (fused, calls):
            if t == 0:
                dec.update_summaries(q, True)
            dec.step(q, kn, vn, t)
        torch.cuda.synchronize()
        _same(fused, calls, f"step {t}")
        if t == 0:
            act = fused.active.cpu().numpy().astype(bool)
            assert act.all() and int(fused.grow.sum()) == free_top


@pytest.mark.parametrize("B", [2048, 2100])
def test_fused_step_many_sequences(B):
    """Up to 2048 sequences the fused step lists the rows at a capacity
    boundary in shared memory and numbers its work items densely; above that
    it numbers every (sequence, split) pair.  Both against the separate calls,
    bit for bit, over three steps: short rows, two thirds of them at a page
    boundary, budgets of 1 to 5 pages."""
    rng = np.random.default_rng(B)
    pages = rng.integers(1, 6, size=B)
    lens = pages * 16
    lens[::3] -= rng.integers(1, 15, size=len(lens[::3]))
    budget = rng.integers(1, 6, size=B).astype(np.int32)
    x = W.small_decode(93, B, 8, 2, 64, lens.tolist(), dtype=W.F16, pool_factor=1.5, pad_pages=2)
    cfg = BG.BudgetConfig(a_fast=0.9, a_slow=0.999, n_first=1, n_last=1, delta=0.3)
    fused, calls = _pair(x, budget, cfg)
    for t in range(3):
        q = bits_to_dev(W.normal_bits(rng, (x.B, x.Hq, 64), W.F16), W.F16)
        kn = bits_to_dev(W.normal_bits(rng, (x.B, x.Hkv, 64), W.F16), W.F16)
        vn = bits_to_dev(W.normal_bits(rng, (x.B, x.Hkv, 64), W.F16), W.F16)
        for dec in (fused, calls):
            if t == 0:
                dec.update_summaries(q, True)
            dec.step(q, kn, vn, t)
        torch.cuda.synchronize()
        _same(fused, calls, f"step {t}")
        if t == 0:
            assert int(fused.active.sum()) > B // 10  # many rows at a boundary


def test_fused_step_tied_scores():
    """Rows whose pages hold identical keys score every candidate alike, so
    the selection's order comes from the page index alone (and half tied in
    another row): the fused step's threshold selection against the separate
    calls' ranks, bit for bit, over three steps."""
    lens = [16 * 12, 16 * 9, 16 * 20, 16 * 7 + 5]
    budget = np.array([12, 9, 20, 6], np.int32)
    x = W.small_decode(94, len(lens), 8, 2, 128, lens, dtype=W.BF16, pool_factor=1.5, pad_pages=3)
    for b, share in ((0, 1.0), (2, 0.5)):  # all / half of the row's pages copies of one page
        row = x.block_table[b][: lens[b] // 16]
        for p in row[: int(len(row) * share)]:
            x.k_pool[p] = x.k_pool[row[0]]
    cfg = BG.BudgetConfig(a_fast=0.9, a_slow=0.999, n_first=1, n_last=1, delta=0.3)
    fused, calls = _pair(x, budget, cfg)
    rng = np.random.default_rng(7)
    for t in range(3):
        q = bits_to_dev(W.normal_bits(rng, (x.B, x.Hq, 128), W.BF16), W.BF16)
        kn = bits_to_dev(W.normal_bits(rng, (x.B, x.Hkv, 128), W.BF16), W.BF16)
        vn = bits_to_dev(W.normal_bits(rng, (x.B, x.Hkv, 128), W.BF16), W.BF16)
        for dec in (fused, calls):
            if t == 0:
                dec.update_summaries(q, True)
            dec.step(q, kn, vn, t)
        torch.cuda.synchronize()
        _same(fused, calls, f"step {t}")
        if t == 0:
            assert int(fused.active.sum()) == 3


def test_fused_step_append_failure():
    """A row whose last page is full but which is below its budget needs a
    page the free list does not have: both paths report KV_ENOSPACE and
    leave the same state (the compaction stands, the append changes
    nothing)."""
    lens = [16 * 5, 16 * 6, 40]
    budget = np.array([5, 50, 9], np.int32)  # row 1 is below budget: no compaction, needs a page
    x = W.small_decode(92, len(lens), 8, 2, 128, lens, dtype=W.BF16, pool_factor=1.0, pad_pages=2)
    x.free_top = 0
    cfg = BG.BudgetConfig(delta=0.5)
    fused, calls = _pair(x, budget, cfg)
    rng = np.random.default_rng(6)
    q = bits_to_dev(W.normal_bits(rng, (x.B, x.Hq, 128), W.BF16), W.BF16)
    kn = bits_to_dev(W.normal_bits(rng, (x.B, x.Hkv, 128), W.BF16), W.BF16)
    vn = bits_to_dev(W.normal_bits(rng, (x.B, x.Hkv, 128), W.BF16), W.BF16)
    for dec in (fused, calls):
        dec.update_summaries(q, True)
        dec._budget_part(q, kn, vn, False)
    torch.cuda.synchronize()
    for name in _STATE[:-2]:
        assert torch.equal(getattr(fused, name), getattr(calls, name)), name
    assert fused.status() == kv.KV_ENOSPACE
    assert calls.status() == kv.KV_ENOSPACE


def test_dump_and_replay(tmp_path):
    """A decoder restored from a state dump (.npz) continues exactly as the
    original: same tables, lengths, free list, EMAs, pools and outputs."""
    lens = [16 * 9, 16 * 12 + 3, 16 * 7, 16 * 30, 16 * 10 + 9, 16 * 8]
    budget = np.array([6, 10, 5, 20, 8, 8], np.int32)
    x = W.small_decode(93, len(lens), 16, 4, 128, lens, dtype=W.BF16, pool_factor=1.5, pad_pages=4)
    cfg = BG.BudgetConfig(delta=0.25)
    decs = []
    for _ in range(2):
        dd = DeviceDecode(x)
        dec = BG.BudgetedDecoder(dd.k, dd.v, dd.table, dd.lens, i32(x.free_list),
                                 i32([x.free_top]), i32(budget), x.Hq, cfg)
        dec.summarize_pages(i32(np.arange(x.num_pages)))
        decs.append(dec)
    orig, replay = decs
    rng = np.random.default_rng(8)
    toks = [[bits_to_dev(W.normal_bits(rng, shape, W.BF16), W.BF16)
             for shape in ((x.B, x.Hq, 128), (x.B, x.Hkv, 128), (x.B, x.Hkv, 128))]
            for _ in range(40)]
    orig.fit(toks[0][0])
    for t in range(12):
        orig.step(*toks[t], t)
    path = str(tmp_path / "state.npz")
    orig.dump(path)
    replay.restore(path)
    for t in range(12, 40):
        orig.step(*toks[t], t)
        replay.step(*toks[t], t)
    torch.cuda.synchronize()
    for name in ("table", "lens", "budget", "free_top", "ema", "summ", "keep", "grow", "k_pool",
                 "v_pool", "out", "lse"):
        assert torch.equal(getattr(orig, name), getattr(replay, name)), name
    top = int(orig.free_top.item())
    assert torch.equal(orig.free_list[:top], replay.free_list[:top])
    assert orig.status() == 0 and replay.status() == 0
