"""Budgeting decisions checked against the fp64 definition.

The budgeting chain runs in fp32 with a stated summation order (kernels and
the fp32 oracle agree bit for bit).  This module checks that those fp32
decisions are the ones the plain fp64 definition takes: GrowPage's
compress-or-grow at each capacity boundary (mlsanity.com, GrowPage,
Abstract), as this library instantiates it -- dual EMAs of the group-mean
query, page scores against mean and channel-wise min/max keys, top-k
retention with forced first/last pages, drift of the two summaries' working
sets.

For every decision it computes, in fp64 from fp64 EMAs and fp64 page
summaries, the margin at the cut (the k-th against the (k+1)-th key of a
top-k, for the retention key and for each summary's working set) and
compares it with a certified bound on |fp32 score - fp64 score|:

    arithmetic part  (Hkv*d/32 + 7) * 2^-24 * sum|terms|   (the stated fp32
                     order: one rounding per product, one per max-add, a
                     32-way lane split and a 5-step butterfly; pinned on CPU)
    input part       |score64(fp32 EMAs, fp32 summaries) - score64(fp64 ...)|
                     (evaluated exactly, so the drift of the fp32 EMAs over
                     the trace is accounted for)

A decision whose margin clears the bound must equal the fp64 one; one that
does not is a near-tie: it is counted and reported, and the fp32 choice is
only required to be valid (no kept page certainly worse than a dropped one).
Test infrastructure: calls only the oracle and numpy.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import oracle as O

TOPK, BOUNDARY = O.SELECT_TOPK, O.SELECT_BOUNDARY
U24 = 2.0 ** -24


def topk_order(keys, cands):
    """Candidates sorted by key descending, ties to the lower logical index."""
    return sorted(cands, key=lambda j: (-keys[j], j))


class Stats:
    def __init__(self):
        self.decisions = 0
        self.near_ties = 0
        self.min_ratio = math.inf   # smallest margin / bound seen at a clear decision
        self.log = []
        self.near_rows = set()      # (tag, b) of every near-tie
        self.near_flipped = 0       # near-ties where the checked choice differs from fp64's

    def cut(self, margin, bound, where, row=None):
        self.decisions += 1
        if margin > bound:
            if bound > 0:
                self.min_ratio = min(self.min_ratio, margin / bound)
            return True
        self.near_ties += 1
        self.near_rows.add(row)
        self.log.append(f"near-tie at {where}: margin {margin:.3e} <= bound {bound:.3e}")
        return False

    def summary(self):
        return (f"{self.decisions} fp64-checked cuts, {self.near_ties} near-ties "
                f"({self.near_flipped} of them decided otherwise than fp64), "
                f"smallest margin/bound at a clear cut {self.min_ratio:.3g}")


class DecisionAnchor:
    """fp64 twin of the budgeting state (EMAs, page summaries) and the
    per-decision check."""

    def __init__(self, B, Hq, Hkv, d, P, dtype, a_fast, a_slow, ps=16):
        self.B, self.Hq, self.Hkv, self.d, self.P, self.dtype, self.ps = B, Hq, Hkv, d, P, dtype, ps
        self.a_fast, self.a_slow = a_fast, a_slow
        self.ema64 = np.zeros((B, 2, Hkv, d))
        self.summ64 = np.zeros((P, Hkv, 3, d))
        self.stats = Stats()

    def update_ema(self, q, first):
        O.ema_f64(q, self.B, self.Hq, self.Hkv, self.d, self.dtype, self.a_fast, self.a_slow,
                  first, self.ema64)

    def summarize(self, k_pool, page_ids):
        page_ids = np.asarray(page_ids, np.int32)
        if len(page_ids):
            O.page_summaries_f64(k_pool, page_ids, self.Hkv, self.ps, self.d, self.dtype,
                                 self.summ64)

    # -- error bounds ------------------------------------------------------
    def _score_error(self, b, pages, ema32, summ32, s64):
        """Certified bound on |fp32 score - fp64 score| for row b's pages
        (n x 2): the stated order's arithmetic bound plus the exact effect of
        the fp32 inputs (their score evaluated in fp64 against the fp64
        definition's)."""
        sm = summ32[pages].astype(np.float64)            # n, Hkv, 3, d
        err = np.zeros((len(pages), 2))
        for u in range(2):
            uu = ema32[b, u].astype(np.float64)          # Hkv, d
            ta, tb = uu * sm[:, :, 1], uu * sm[:, :, 2]
            s64b = (uu * sm[:, :, 0] + np.maximum(ta, tb)).sum(axis=(1, 2))
            terms = np.abs(uu * sm[:, :, 0]) + np.maximum(np.abs(ta), np.abs(tb))
            arith = (self.Hkv * self.d / 32 + 7) * U24 * terms.sum(axis=(1, 2))
            err[:, u] = (arith + np.abs(s64b - s64[:, u]) + 1e-12 * (np.abs(s64[:, u]) +
                                                                      terms.sum(axis=(1, 2))))
        return err

    # -- one select_pages call -----------------------------------------------
    def check(self, *, table, lens, active, budget, free_count, mode, n_first, n_last, delta,
              ws_frac, ema32, summ32, scores32, keep, grow, drift, budget_after, tag=""):
        """table/lens/active/budget/free_count: the state the selection saw;
        ema32/summ32/scores32: the fp32 chain's inputs and scores;
        keep/grow/drift/budget_after: the decisions being checked."""
        B, maxp = table.shape
        act = np.ones(B, np.uint8) if active is None else np.asarray(active, np.uint8)
        s64 = np.zeros((B, maxp, 2))
        O.score_pages_f64(self.ema64, self.summ64, table, lens, act, self.Hkv, self.d, self.ps,
                          s64)
        st = self.stats
        wants64 = {}
        certain_wants = True
        granted = 0
        for b in range(B):
            if not act[b]:
                continue
            n = -(-int(lens[b]) // self.ps)
            pages = table[b, :n]
            err = self._score_error(b, pages, ema32, summ32, s64[b, :n])
            # the fp32 scores really are within the bound of the fp64 ones
            d32 = np.abs(scores32[b, :n].astype(np.float64) - s64[b, :n])
            assert np.all(d32 <= err), (tag, b, float((d32 - err).max()))
            forced = [j for j in range(n) if j < n_first or j >= n - n_last]
            cands = [j for j in range(n) if not (j < n_first or j >= n - n_last)]
            nf, nc = len(forced), len(cands)
            R64 = s64[b, :n, 0] + s64[b, :n, 1]
            Rerr = err[:, 0] + err[:, 1] + U24 * np.abs(R64) * 1.01

            def check_keep(k, where):
                order = topk_order(R64, cands)
                k = max(0, min(k, nc))
                want = set(forced) | set(order[:k])
                got = set(np.nonzero(keep[b, :n])[0].tolist())
                if 0 < k < nc:
                    a, c = order[k - 1], order[k]
                    clear = st.cut(R64[a] - R64[c], Rerr[a] + Rerr[c], f"{tag} b={b} {where}",
                                   (tag, b))
                else:
                    clear = True
                if clear:
                    assert got == want, (tag, b, where, sorted(got ^ want))
                else:
                    # valid: forced pages kept, k candidates kept, and no kept
                    # candidate certainly worse than a dropped one
                    st.near_flipped += int(got != want)
                    assert set(forced) <= got and len(got) == nf + k, (tag, b, where)
                    kept = [j for j in cands if j in got]
                    dropped = [j for j in cands if j not in got]
                    if kept and dropped:
                        lo_kept = min(R64[j] + Rerr[j] for j in kept)
                        hi_drop = max(R64[j] - Rerr[j] for j in dropped)
                        assert lo_kept >= hi_drop, (tag, b, where)

            if mode == TOPK:
                check_keep(int(budget[b]) - nf, "fit top-k")
                continue
            # boundary: drift of the two working sets, then grow or compact
            if nc == 0:
                wants64[b] = True
            else:
                w = int(math.ceil(np.float32(ws_frac) * np.float32(nc)))
                w = max(1, min(w, nc))
                sets, clear = [], True
                for u in range(2):
                    key = s64[b, :n, u]
                    order = topk_order(key, cands)
                    if w < nc:
                        a, c = order[w - 1], order[w]
                        clear &= st.cut(key[a] - key[c], err[a, u] + err[c, u],
                                        f"{tag} b={b} working set {'fast' if u == 0 else 'slow'}",
                                        (tag, b))
                    sets.append(set(order[:w]))
                D64 = len(sets[0] - sets[1])
                if clear:
                    assert int(drift[b]) == D64, (tag, b, int(drift[b]), D64)
                    wants64[b] = D64 > np.float32(delta) * np.float32(w)
                else:
                    certain_wants = False
                    st.near_flipped += int(int(drift[b]) != D64)
                    wants64[b] = int(drift[b]) > np.float32(delta) * np.float32(w)
            grow64 = wants64[b] and granted < free_count
            granted += int(grow64)
            if certain_wants:
                assert bool(grow[b]) == grow64, (tag, b)
                assert int(budget_after[b]) == int(budget[b]) + int(grow64), (tag, b)
            if not grow[b]:
                check_keep(n - 1 - nf, "compact top-k")
            else:
                assert np.all(keep[b, :n] == 1), (tag, b)
        return st
