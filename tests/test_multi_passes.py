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

from oracle import oracle as O
from paged_kv_cache_492_b300 import workloads as W


def _passes(T, most):
    passes = -(-T // most)
    per = -(-T // passes)
    return [(t0, min(per, T - t0)) for t0 in range(0, T, per)]


@pytest.mark.parametrize("T,G,lens,most", [
    (20, 4, [0, 3, 19, 20, 21, 100], 16),    # passes of 10 + 10 tokens; L < T rows
    (33, 2, [1, 32, 33, 34, 250], 32),       # 17 + 16
    (9, 8, [5, 8, 9, 64], 8),                # 5 + 4
    (40, 4, [39, 40, 41, 300], 16),          # 14 + 14 + 12
])
def test_passes_reproduce_the_one_pass_rows(T, G, lens, most):
    Hkv = 2
    x = W.small_decode(400 + T, len(lens), Hkv * G, Hkv, 64, lens, dtype=W.F16)
    rng = np.random.default_rng(T)
    qm = W.normal_bits(rng, (x.B, T, x.Hq, x.d), x.dtype)
    full_o, full_l = O.attend_multi(x, qm)
    plan = _passes(T, most)
    assert len(plan) == -(-T // most) and sum(n for _, n in plan) == T
    assert all(n <= most for _, n in plan)
    for t0, n in plan:
        shift = T - t0 - n
        y = W.DecodeInputs(**{**x.__dict__,
                              "seq_lens": np.maximum(x.seq_lens - shift, 0).astype(np.int32)})
        o, l = O.attend_multi(y, np.ascontiguousarray(qm[:, t0:t0 + n]))
        assert np.array_equal(o, full_o[:, t0:t0 + n]), (t0, n)
        assert np.array_equal(l, full_l[:, t0:t0 + n]), (t0, n)
