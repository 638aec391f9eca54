"""CPU mirror of the budgeted decode step (paged_kv_cache_492_b300.budget),
built only from oracle calls, in the same order."""
from __future__ import annotations

import numpy as np

from oracle import oracle as O
from paged_kv_cache_492_b300 import workloads as W


class OracleBudget:
    """`anchor` (optional, tests/decision_check.DecisionAnchor) is kept in
    step with the fp32 chain: fp64 EMAs from the same queries and fp64
    summaries of the same pages at the same time.  `pre` holds the state each
    selection saw, for checking its decisions."""

    def __init__(self, x: W.DecodeInputs, budget, cfg, refcnt=None, anchor=None):
        self.x = x
        self.cfg = cfg
        self.anchor = anchor
        self.pre = None
        self.k = np.ascontiguousarray(x.k_pool).copy()
        self.v = np.ascontiguousarray(x.v_pool).copy()
        self.table = np.ascontiguousarray(x.block_table, dtype=np.int32).copy()
        self.lens = np.ascontiguousarray(x.seq_lens, dtype=np.int32).copy()
        self.free_list = np.ascontiguousarray(x.free_list, dtype=np.int32).copy()
        self.top = np.array([x.free_top], dtype=np.int32)
        self.budget = np.asarray(budget, dtype=np.int32).copy()
        self.refcnt = None if refcnt is None else np.asarray(refcnt, dtype=np.int32).copy()
        B, maxp = self.table.shape
        P = self.k.shape[0]
        self.ema = np.zeros((B, 2, x.Hkv, x.d), np.float32)
        self.summ = np.zeros((P, x.Hkv, 3, x.d), np.float32)
        self.scores = np.zeros((B, maxp, 2), np.float32)
        self.keep = self.grow = self.drift = self.active = None

    def summarize_all(self):
        ids = np.arange(self.k.shape[0], dtype=np.int32)
        O.page_summaries_f32(self.k, ids, self.x.Hkv, 16, self.x.d, self.x.dtype, self.summ)
        if self.anchor is not None:
            self.anchor.summarize(self.k, ids)

    def _select(self, mode):
        self.pre = dict(table=self.table.copy(), lens=self.lens.copy(),
                        active=self.active.copy(), budget=self.budget.copy(),
                        free_count=int(self.top[0]), mode=mode)
        keep, grow, bud, drift = O.select_pages(self.scores, self.lens, self.active, self.budget,
                                                16, self.cfg.n_first, self.cfg.n_last,
                                                self.cfg.delta, mode, int(self.top[0]),
                                                ws_frac=self.cfg.ws_frac)
        self.keep, self.grow, self.drift = keep, grow, drift
        self.budget = bud
        rc = O.compact_inplace(self.table, self.lens, np.ascontiguousarray(keep), False, self.k,
                               self.v, self.free_list, self.top, self.x.Hkv, self.x.d, 16,
                               refcnt=self.refcnt)
        assert rc == 0, rc

    def fit(self, q0):
        x = self.x
        O.ema_f32(q0, x.B, x.Hq, x.Hkv, x.d, x.dtype, self.cfg.a_fast, self.cfg.a_slow, True,
                  self.ema)
        if self.anchor is not None:
            self.anchor.update_ema(q0, True)
        self.active = O.mark_active(self.lens, self.budget, 16, 0)
        O.score_pages_f32(self.ema, self.summ, self.table, self.lens, self.active, x.Hkv, x.d, 16,
                          self.scores)
        self._select(O.SELECT_TOPK)

    def step(self, q, k_new, v_new, t):
        x = self.x
        if t > 0:
            O.ema_f32(q, x.B, x.Hq, x.Hkv, x.d, x.dtype, self.cfg.a_fast, self.cfg.a_slow, False,
                      self.ema)
            if self.anchor is not None:
                self.anchor.update_ema(q, False)
        self.active = O.mark_active(self.lens, self.budget, 16, 1)
        last = [int(self.table[b, self.lens[b] // 16 - 1]) for b in range(x.B)
                if self.active[b] and self.lens[b] >= 16]
        if last:
            O.page_summaries_f32(self.k, np.array(last, np.int32), x.Hkv, 16, x.d, x.dtype,
                                 self.summ)
            if self.anchor is not None:
                self.anchor.summarize(self.k, np.array(last, np.int32))
        O.score_pages_f32(self.ema, self.summ, self.table, self.lens, self.active, x.Hkv, x.d, 16,
                          self.scores)
        self._select(O.SELECT_BOUNDARY)
        # sequences whose pages changed this step: compacted, grown, or about
        # to take a fresh page in the append
        self.changed = sorted(set(np.nonzero(self.active)[0].tolist()) |
                              set(np.nonzero(self.lens % 16 == 0)[0].tolist()))
        rc = O.append_inplace(k_new, v_new, self.k, self.v, self.table, self.lens,
                              self.free_list, self.top, x.Hkv, x.d, 16, refcnt=self.refcnt)
        assert rc == 0, rc

    def decode_inputs(self, q):
        x = self.x
        return W.DecodeInputs(name="budget_state", B=x.B, Hq=x.Hq, Hkv=x.Hkv, d=x.d,
                              page_size=16, dtype=x.dtype, scale=x.scale, q=q, k_pool=self.k,
                              v_pool=self.v, block_table=self.table, seq_lens=self.lens)
