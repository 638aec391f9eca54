"""GrowPage-style budgeted decode step, as a sequence of C-ABI calls.

GrowPage (mlsanity.com, "GrowPage: On-Demand KV Budgeting ...", Abstract):
query summaries at two time scales; at every capacity boundary either compress
the KV states inside the current allocation or take one more physical page
when the recent attention working set has moved beyond the long-term one.
This module only orders the library's kernels on one stream; it does no
arithmetic itself.

Per-step order (this library's reading):
  1. query EMAs with q_t (step 0: initialised from q_0 by `fit`);
  2. capacity boundary = last page full and the sequence holds its budget:
     summarise the page that just filled, score the resident pages, select
     (grow by one page, or keep the forced pages plus the best n-1-|F|),
     compact the block table (page granular: no K/V moves);
  3. append the token's K/V (pops a page when the last one is full);
  4. decode over the resident tokens.
`fit` is the start: every sequence above its budget is cut to it with the
same top-k rule before the first step.
"""
from __future__ import annotations

import dataclasses

import torch

from . import kv


@dataclasses.dataclass
class BudgetConfig:
    a_fast: float = 0.9
    a_slow: float = 0.999
    n_first: int = 2
    n_last: int = 2
    delta: float = 0.5
    ws_frac: float = 0.5


class BudgetedDecoder:
    """Device state of a batch decoding under per-sequence page budgets.

    k_pool, v_pool [P, Hkv, 16, d] (f16/bf16), block_table [B, maxP] int32,
    seq_lens [B] int32, free_list [P] int32 + free_top [1] int32 (stack),
    budget [B] int32, refcnt [P] int32 (block-table references per pool page,
    for batches whose sequences share prefix pages; None = no sharing).  All
    tensors live on one device and are updated in place by the kernels.
    pages_per_split picks the decode engine as kv_decode's argument does
    (0: the fused kernel with the automatic split; KV_DECODE_TENSOR_CORE:
    the tensor-core engine).  fused_step: issue the steady-state step's
    budgeting part as the single kv_budget_step launch (batches without
    shared pages) instead of its seven calls; the results are the same."""

    def __init__(self, k_pool, v_pool, block_table, seq_lens, free_list, free_top, budget,
                 Hq: int, cfg: BudgetConfig, stream=None, refcnt=None, pages_per_split: int = 0,
                 fused_step: bool = True):
        self.k_pool, self.v_pool = k_pool, v_pool
        self.table, self.lens = block_table, seq_lens
        self.free_list, self.free_top = free_list, free_top
        self.budget = budget
        self.refcnt = refcnt
        self.cfg = cfg
        self.stream = stream
        dev = k_pool.device
        P, Hkv, ps, d = k_pool.shape
        B, maxp = block_table.shape
        self.B, self.Hq, self.Hkv, self.d, self.ps, self.maxp, self.P = B, Hq, Hkv, d, ps, maxp, P
        self.ema = torch.zeros((B, 2, Hkv, d), dtype=torch.float32, device=dev)
        self.summ = torch.zeros((P, Hkv, 3, d), dtype=torch.float32, device=dev)
        self.scores = torch.zeros((B, maxp, 2), dtype=torch.float32, device=dev)
        self.active = torch.zeros(B, dtype=torch.uint8, device=dev)
        self.keep = torch.zeros((B, maxp), dtype=torch.uint8, device=dev)
        self.grow = torch.zeros(B, dtype=torch.uint8, device=dev)
        self.drift = torch.zeros(B, dtype=torch.int32, device=dev)
        self.out = torch.empty((B, Hq, d), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        self.fused_step = bool(fused_step) and refcnt is None
        ws = max(kv.kv_select_workspace_size(B, maxp),
                 kv.kv_compact_workspace_size(B, maxp, P if refcnt is not None else 0),
                 kv.kv_append_workspace_size(B))
        self.ws = kv.alloc_workspace(ws, dev)
        # kv_budget_step keeps per-sequence tickets in its workspace between
        # calls: it gets one of its own
        self.step_ws = (kv.alloc_workspace(kv.kv_budget_step_workspace_size(B, maxp), dev)
                        if self.fused_step else None)
        # kv_decode keeps merge tickets in its workspace between calls; sized
        # for both engines so calibrate() can switch between them
        self.pages_per_split = pages_per_split
        self.decode_ws = kv.alloc_workspace(
            max(kv.kv_decode_workspace_size(B, Hq, Hkv, d, maxp, ps, c)
                for c in (0, pages_per_split, kv.KV_DECODE_TENSOR_CORE)), dev)
        self.scale = 1.0 / (d ** 0.5)

    # -- pieces ---------------------------------------------------------
    def summarize_pages(self, page_ids):
        kv.kv_page_summaries(self.k_pool, page_ids, self.summ, self.ws, stream=self.stream)

    def update_summaries(self, q, first):
        kv.kv_update_query_summaries(q, self.Hkv, self.cfg.a_fast, self.cfg.a_slow, first,
                                     self.ema, stream=self.stream)

    def fit(self, q0):
        """Start of decoding: EMAs from q0, then cut every sequence that holds
        more pages than its budget down to it (forced first/last pages kept)."""
        c = self.cfg
        self.update_summaries(q0, True)
        kv.kv_mark_active(self.lens, self.budget, self.ps, 0, self.active, stream=self.stream)
        kv.kv_score_pages(self.ema, self.summ, self.table, self.lens, self.active, self.scores,
                          self.ws, stream=self.stream)
        kv.kv_select_pages(self.scores, self.lens, self.active, self.budget, c.n_first, c.n_last,
                           c.delta, c.ws_frac, kv.KV_SELECT_TOPK, self.free_top, self.keep,
                           self.grow, self.drift, self.ws, stream=self.stream)
        kv.kv_compact(self.table, self.lens, self.keep, False, self.k_pool, self.v_pool,
                      self.free_list, self.free_top, self.ws, stream=self.stream,
                      refcnt=self.refcnt)

    def boundary(self):
        """Compress-or-grow for the sequences at a capacity boundary."""
        c = self.cfg
        kv.kv_mark_active(self.lens, self.budget, self.ps, 1, self.active, stream=self.stream)
        kv.kv_summarize_last_pages(self.k_pool, self.table, self.lens, self.active, self.summ,
                                   self.ws, stream=self.stream)
        kv.kv_score_pages(self.ema, self.summ, self.table, self.lens, self.active, self.scores,
                          self.ws, stream=self.stream)
        kv.kv_select_pages(self.scores, self.lens, self.active, self.budget, c.n_first, c.n_last,
                           c.delta, c.ws_frac, kv.KV_SELECT_BOUNDARY, self.free_top, self.keep,
                           self.grow, self.drift, self.ws, stream=self.stream)
        kv.kv_compact(self.table, self.lens, self.keep, False, self.k_pool, self.v_pool,
                      self.free_list, self.free_top, self.ws, stream=self.stream,
                      refcnt=self.refcnt)

    def step(self, q, k_new, v_new, t: int):
        """One decode step for token t (q [B, Hq, d], k_new/v_new [B, Hkv, d])."""
        self._budget_part(q, k_new, v_new, t > 0)
        self._decode_part(q)

    def _budget_part(self, q, k_new, v_new, update_ema: bool):
        if self.fused_step:
            c = self.cfg
            kv.kv_budget_step(q, k_new, v_new, self.k_pool, self.v_pool, self.table, self.lens,
                              self.budget, c.a_fast, c.a_slow, update_ema, c.n_first, c.n_last,
                              c.delta, c.ws_frac, self.ema, self.summ, self.scores, self.active,
                              self.keep, self.grow, self.drift, self.free_list, self.free_top,
                              self.step_ws, stream=self.stream)
            return
        if update_ema:
            self.update_summaries(q, False)
        self.boundary()
        kv.kv_append(k_new, v_new, self.k_pool, self.v_pool, self.table, self.lens,
                     self.free_list, self.free_top, self.ws, stream=self.stream,
                     refcnt=self.refcnt)

    def _decode_part(self, q):
        kv.kv_decode(q, self.k_pool, self.v_pool, self.table, self.lens, self.scale, self.out,
                     self.lse, self.decode_ws, pages_per_split=self.pages_per_split,
                     stream=self.stream)

    def status(self) -> int:
        """First device-side error recorded by the budgeting calls or the
        decode since the last check (0 = none); synchronises the stream."""
        for ws in (self.ws, self.step_ws, self.decode_ws):
            if ws is not None:
                rc = kv.kv_get_status(ws, stream=self.stream)
                if rc:
                    return rc
        return 0

    # -- state dump for replaying a step ---------------------------------
    STATE = ("table", "lens", "free_list", "free_top", "budget", "ema", "summ", "scores", "active",
             "keep", "grow", "drift")

    def dump(self, path, pools: bool = True):
        """Write the batch's state to an .npz file (host copies): block
        tables, lengths, free list, budgets, query EMAs, page summaries, the
        last step's scores and decisions, reference counts and, with `pools`,
        the K/V pools -- what a failed step needs to be replayed."""
        import json

        import numpy as np

        arrays = {name: getattr(self, name).cpu().numpy() for name in self.STATE}
        if self.refcnt is not None:
            arrays["refcnt"] = self.refcnt.cpu().numpy()
        if pools:
            arrays["k_pool"] = self.k_pool.view(torch.int16).cpu().numpy()
            arrays["v_pool"] = self.v_pool.view(torch.int16).cpu().numpy()
        arrays["config"] = np.array(json.dumps(dataclasses.asdict(self.cfg)))
        np.savez(path, **arrays)

    def restore(self, path):
        """Load a dump written by dump() into this decoder (same shapes and
        configuration); the pools are restored when the dump holds them."""
        import json

        import numpy as np

        with np.load(path) as z:
            if json.loads(str(z["config"])) != dataclasses.asdict(self.cfg):
                raise ValueError("dump was written with another budget configuration")
            for name in self.STATE:
                t = getattr(self, name)
                a = z[name]
                if tuple(a.shape) != tuple(t.shape):
                    raise ValueError(f"dump has {name} of shape {a.shape}, decoder {tuple(t.shape)}")
                t.copy_(torch.from_numpy(a))
            if "refcnt" in z.files and self.refcnt is not None:
                self.refcnt.copy_(torch.from_numpy(z["refcnt"]))
            if "k_pool" in z.files:
                self.k_pool.view(torch.int16).copy_(torch.from_numpy(z["k_pool"]))
                self.v_pool.view(torch.int16).copy_(torch.from_numpy(z["v_pool"]))

    def calibrate(self, q, candidates=(0, kv.KV_DECODE_TENSOR_CORE), reps=5, flush=None):
        """Pick the decode engine for this batch by timing each candidate on
        the current state (kv_decode_tune; `flush`, a device buffer larger
        than L2, is overwritten before every timed call).  Call before
        capture().  Returns (chosen pages_per_split, {candidate: us})."""
        B, Hq, d = self.B, self.Hq, self.d
        cands = [c for c in candidates
                 if kv.kv_decode_workspace_size(B, Hq, self.Hkv, d, self.maxp, self.ps, c) > 0]
        best, us = kv.kv_decode_tune(q, self.k_pool, self.v_pool, self.table, self.lens,
                                     self.scale, self.out, self.lse, self.decode_ws, cands, reps,
                                     self.stream, flush=flush)
        self.pages_per_split = best
        return best, dict(zip(cands, us))

    # -- the step as CUDA graphs ----------------------------------------
    def capture(self):
        """Record the steady-state step (t > 0) as CUDA graphs over static
        input buffers: the whole step as one graph, and its budgeting part
        (EMA, boundary compress-or-grow, append) and decode as two more (to
        time them apart), so a step costs one graph launch instead of a
        sequence of host calls.  Every kernel reads its state from device
        memory, so replays follow the batch as it evolves.  Capture issues no
        work; call after at least one eager step (the library sets up its
        kernels on first use)."""
        import torch

        B, Hq, Hkv, d = self.B, self.Hq, self.Hkv, self.d
        dt = self.k_pool.dtype
        dev = self.k_pool.device
        # q, k and v of the step's token: views of one buffer, so a token packed
        # the same way (pack_token) arrives in one copy
        nq, nk = B * Hq * d, B * Hkv * d
        self.tok_in = torch.zeros(nq + 2 * nk, dtype=dt, device=dev)
        self.q_in = self.tok_in[:nq].view(B, Hq, d)
        self.k_in = self.tok_in[nq:nq + nk].view(B, Hkv, d)
        self.v_in = self.tok_in[nq + nk:].view(B, Hkv, d)
        saved = self.stream
        side = torch.cuda.Stream(device=dev)
        self.g_budget, self.g_decode = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        self.g_step = torch.cuda.CUDAGraph()
        try:
            self.stream = None  # the capturing stream is the current one
            with torch.cuda.graph(self.g_budget, stream=side):
                self._budget_part(self.q_in, self.k_in, self.v_in, True)
            with torch.cuda.graph(self.g_decode, stream=side):
                self._decode_part(self.q_in)
            with torch.cuda.graph(self.g_step, stream=side):
                self._budget_part(self.q_in, self.k_in, self.v_in, True)
                self._decode_part(self.q_in)
        finally:
            self.stream = saved

    def step_graphed(self, q, k_new, v_new, between=None):
        """One steady-state step (t > 0) by graph replay on the current
        stream: copies the token's q/k/v into the static buffers and replays
        the step's graph; with `between`, replays the budgeting graph, calls
        `between()` (e.g. to record an event) and then the decode graph.
        Same kernels, order and results as step()."""
        self.q_in.copy_(q)
        self.k_in.copy_(k_new)
        self.v_in.copy_(v_new)
        self._replay(between)

    @staticmethod
    def pack_token(q, k_new, v_new):
        """The step's q, k and v in the layout of the graphs' input buffer."""
        import torch

        return torch.cat([q.reshape(-1), k_new.reshape(-1), v_new.reshape(-1)])

    def step_graphed_packed(self, tok, between=None):
        """step_graphed with the token already packed (pack_token): one copy
        into the static buffers instead of three."""
        self.tok_in.copy_(tok)
        self._replay(between)

    def _replay(self, between):
        if between is None:
            self.g_step.replay()
            return
        self.g_budget.replay()
        between()
        self.g_decode.replay()
