"""The multi-token passes' decomposition, checked on the oracle alone (no
GPU): T query tokens served as passes over token chunks [t0, t0 + n), where a
pass sees every sequence's length shortened by T - t0 - n, give exactly the
rows of the one-pass problem.  Query t attends to [0, L - T + 1 + t) either
way: in the pass, L' - n + 1 + (t - t0) with L' = L - (T - t0 - n) is the same
limit, and a length that would go below zero leaves every query of the pass
with nothing to attend to, as in the full problem (out = 0, lse = -inf).  So
the oracle's per-row arithmetic is identical and the rows agree bit for bit."""
import numpy as np
import pytest

import bench
from oracle import oracle as O
from paged_kv_cache_492_b300 import workloads as W


def _passes(T, G):
    plan, t0 = [], 0
    for n in bench.multi_pass_plan(T, G):
        plan.append((t0, n))
        t0 += n
    return plan


@pytest.mark.parametrize("T,G,lens,most,plan", [
    (20, 4, [0, 3, 19, 20, 21, 100], 16, [12, 8]),    # 3 + 2 row blocks; L < T rows
    (17, 4, [1, 16, 17, 18, 90], 16, [12, 5]),
    (33, 2, [1, 32, 33, 34, 250], 32, [24, 9]),
    (9, 8, [5, 8, 9, 64], 8, [6, 3]),
    (40, 4, [39, 40, 41, 300], 16, [16, 12, 12]),
    (7, 12, [3, 6, 7, 50], 5, [5, 2]),                # G does not divide 16: full passes
])
def test_passes_reproduce_the_one_pass_rows(T, G, lens, most, plan):
    Hkv = 2
    x = W.small_decode(400 + T, len(lens), Hkv * G, Hkv, 64, lens, dtype=W.F16)
    rng = np.random.default_rng(T)
    qm = W.normal_bits(rng, (x.B, T, x.Hq, x.d), x.dtype)
    full_o, full_l = O.attend_multi(x, qm)
    passes = _passes(T, G)
    assert [n for _, n in passes] == plan
    assert len(passes) == -(-T // most) and all(n <= most for _, n in passes)
    for t0, n in passes:
        shift = T - t0 - n
        y = W.DecodeInputs(**{**x.__dict__,
                              "seq_lens": np.maximum(x.seq_lens - shift, 0).astype(np.int32)})
        o, l = O.attend_multi(y, np.ascontiguousarray(qm[:, t0:t0 + n]))
        assert np.array_equal(o, full_o[:, t0:t0 + n]), (t0, n)
        assert np.array_equal(l, full_l[:, t0:t0 + n]), (t0, n)
