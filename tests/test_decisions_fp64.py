"""The budgeted batch-64 workload's decisions against the fp64 definition,
on the CPU (oracle only).

GrowPage (mlsanity.com, Abstract) decides at each capacity boundary whether
to compress inside the allocation or to grow it; this library scores pages
in fp32 with a stated reduction order.  Two checks pin those fp32 decisions
to something other than the fp32 arithmetic itself:

* every top-k cut and working-set cut of the fit and of the first boundary
  steps, taken by the fp32 oracle, equals the fp64 definition's unless its
  fp64 margin is inside the certified fp32 error bound (a near-tie, counted
  and printed; the fp32 choice must then still be a valid one);
* scoring with a plain sequential fp32 sum instead of the stated lane order
  gives the same keep masks, except on rows whose cut is a logged near-tie.
"""
import numpy as np
import pytest

from oracle import oracle as O
from paged_kv_cache_492_b300 import budget as BG
from paged_kv_cache_492_b300 import workloads as W
from tests.budget_oracle import OracleBudget
from tests.decision_check import DecisionAnchor

STEPS = 48


@pytest.fixture(scope="module")
def budgeted():
    return W.budgeted_serving(steps=STEPS)


def _cfg(c):
    return BG.BudgetConfig(a_fast=c["a_fast"], a_slow=c["a_slow"], n_first=c["n_first"],
                           n_last=c["n_last"], delta=c["delta"])


def _check(anchor, orc, cfg, tag):
    pre = orc.pre
    return anchor.check(table=pre["table"], lens=pre["lens"], active=pre["active"],
                        budget=pre["budget"], free_count=pre["free_count"], mode=pre["mode"],
                        n_first=cfg.n_first, n_last=cfg.n_last, delta=cfg.delta,
                        ws_frac=cfg.ws_frac, ema32=orc.ema, summ32=orc.summ,
                        scores32=orc.scores, keep=orc.keep, grow=orc.grow, drift=orc.drift,
                        budget_after=orc.budget, tag=tag)


def test_budgeted_decisions_match_fp64(budgeted):
    c = budgeted
    x = c["decode"]
    cfg = _cfg(c)
    anchor = DecisionAnchor(x.B, x.Hq, x.Hkv, x.d, x.num_pages, x.dtype, c["a_fast"], c["a_slow"])
    orc = OracleBudget(x, c["budget"], cfg, anchor=anchor)
    orc.summarize_all()
    q0, _, _ = W.step_tokens(c["seed"], 0, x.B, x.Hq, x.Hkv, x.d, x.dtype)
    orc.fit(q0)
    _check(anchor, orc, cfg, "fit")
    grows = compacts = 0
    for t in range(STEPS):
        q, kn, vn = W.step_tokens(c["seed"], t, x.B, x.Hq, x.Hkv, x.d, x.dtype)
        orc.step(q, kn, vn, t)
        _check(anchor, orc, cfg, f"step {t}")
        act = orc.active.astype(bool)
        grows += int(orc.grow[act].sum())
        compacts += int(act.sum() - orc.grow[act].sum())
    st = anchor.stats
    print(f"budgeted fp64 anchor (CPU, fit + {STEPS} steps): {st.summary()}; "
          f"{grows} grows, {compacts} compactions")
    for line in st.log:
        print("  " + line)
    assert st.decisions > 64 and grows > 0 and compacts > 0


def _scores_sequential_f32(ema, summ, table, lens, Hkv, d):
    """S_u(j) with the terms rounded as the stated order rounds them (one
    rounding per product, one per max-add) but summed strictly left to right
    over (head, channel) in fp32."""
    B, maxp = table.shape
    out = np.full((B, maxp, 2), -np.inf, np.float32)
    for b in range(B):
        n = -(-int(lens[b]) // 16)
        sm = summ[table[b, :n]]                              # n, Hkv, 3, d (fp32)
        for u in range(2):
            uu = ema[b, u][None]                             # 1, Hkv, d
            t1 = (uu * sm[:, :, 0]).astype(np.float32)
            t2 = np.maximum((uu * sm[:, :, 1]).astype(np.float32),
                            (uu * sm[:, :, 2]).astype(np.float32))
            terms = (t1 + t2).astype(np.float32).reshape(n, Hkv * d)
            out[b, :n, u] = np.add.accumulate(terms, axis=1, dtype=np.float32)[:, -1]
    return out


def test_sum_order_does_not_decide(budgeted):
    """The fit of the budgeted workload scored in the stated lane order and in
    a plain sequential order: the same pages are kept wherever the fp64
    margin clears the bound."""
    c = budgeted
    x = c["decode"]
    cfg = _cfg(c)
    anchor = DecisionAnchor(x.B, x.Hq, x.Hkv, x.d, x.num_pages, x.dtype, c["a_fast"], c["a_slow"])
    orc = OracleBudget(x, c["budget"], cfg, anchor=anchor)
    orc.summarize_all()
    q0, _, _ = W.step_tokens(c["seed"], 0, x.B, x.Hq, x.Hkv, x.d, x.dtype)
    orc.fit(q0)
    _check(anchor, orc, cfg, "fit")
    pre = orc.pre
    seq = _scores_sequential_f32(orc.ema, orc.summ, pre["table"], pre["lens"], x.Hkv, x.d)
    lane = np.zeros_like(seq)
    O.score_pages_f32(orc.ema, orc.summ, pre["table"], pre["lens"], pre["active"], x.Hkv, x.d, 16,
                      lane)
    act = pre["active"].astype(bool)
    assert np.array_equal(np.isfinite(seq[act]), np.isfinite(lane[act]))
    assert not np.array_equal(seq[act], lane[act])  # the orders really round differently
    k_lane = O.select_pages(lane, pre["lens"], pre["active"], pre["budget"], 16, cfg.n_first,
                            cfg.n_last, cfg.delta, O.SELECT_TOPK, pre["free_count"],
                            ws_frac=cfg.ws_frac)[0]
    k_seq = O.select_pages(seq, pre["lens"], pre["active"], pre["budget"], 16, cfg.n_first,
                           cfg.n_last, cfg.delta, O.SELECT_TOPK, pre["free_count"],
                           ws_frac=cfg.ws_frac)[0]
    differ = [b for b in range(x.B) if not np.array_equal(k_lane[b], k_seq[b])]
    near = {b for tag, b in anchor.stats.near_rows}
    print(f"sum-order pin: {int(act.sum())} rows cut, {len(differ)} differ, "
          f"near-tie rows {sorted(near)}")
    assert set(differ) <= near, (differ, sorted(near))
