"""The oracle against the hand-derived fixtures in tests/golden/ (CPU only)."""
import math
import os

import numpy as np

from oracle import oracle as O
from paged_kv_cache_492_b300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = (s.strip() for s in line.split("=", 1))
        vals.setdefault(k, []).append([float(t) for t in v.split()])
    return vals


def _one(v, k):
    return v[k][0]


def test_decode_two_pages():
    g = _read("decode_two_pages.txt")
    ps, P, d = 16, 6, 2
    kp = np.full((P, 1, ps, d), 7.0, np.float32)
    vp = np.full((P, 1, ps, d), 7.0, np.float32)
    table = [int(t) for t in _one(g, "table")]
    L = int(_one(g, "seq_len")[0])
    for t in range(L):
        page = table[t // ps]
        if t < 16:
            kp[page, 0, t % ps], vp[page, 0, t % ps] = [0, 0], [1, 0]
        else:
            kp[page, 0, t % ps], vp[page, 0, t % ps] = [1, 0], [0, 1]
    q = np.array([_one(g, "q0"), _one(g, "q1")], np.float32)[None]
    x = W.DecodeInputs(name="golden", B=1, Hq=2, Hkv=1, d=d, page_size=ps, dtype=W.F16,
                       scale=_one(g, "scale")[0], q=W.to_bits(q, W.F16),
                       k_pool=W.to_bits(kp, W.F16), v_pool=W.to_bits(vp, W.F16),
                       block_table=np.array([table], np.int32), seq_lens=np.array([L], np.int32))
    out, lse = O.decode(x)
    for h in range(2):
        assert np.allclose(out[0, h], _one(g, f"out{h}"), rtol=0, atol=1e-12), h
        assert abs(lse[0, h] - _one(g, f"lse{h}")[0]) < 1e-12, h
    assert math.isclose(_one(g, "lse0")[0], math.log(32), abs_tol=1e-15)


def test_attend_multi_causal():
    g = _read("attend_multi_causal.txt")
    ps, P, d, T = 16, 6, 2, 3
    kp = np.full((P, 1, ps, d), 7.0, np.float32)
    vp = np.full((P, 1, ps, d), 7.0, np.float32)
    lens = [int(t) for t in _one(g, "seq_lens")]
    tables = [[int(t) for t in _one(g, f"table{b}")] for b in range(2)]

    def put(b, t, k, v):
        page = tables[b][t // ps]
        kp[page, 0, t % ps], vp[page, 0, t % ps] = k, v

    for t in range(16):
        put(0, t, [0, 0], [1, 0])
    put(0, 16, [1, 0], [0, 1])
    put(0, 17, [1, 0], [0, 2])
    put(1, 0, [0, 0], [1, 0])
    put(1, 1, [1, 0], [0, 1])
    x = W.DecodeInputs(name="golden_multi", B=2, Hq=1, Hkv=1, d=d, page_size=ps, dtype=W.F16,
                       scale=_one(g, "scale")[0],
                       q=W.to_bits(np.zeros((2, 1, d), np.float32), W.F16),
                       k_pool=W.to_bits(kp, W.F16), v_pool=W.to_bits(vp, W.F16),
                       block_table=np.array(tables, np.int32), seq_lens=np.array(lens, np.int32))
    qm = W.to_bits(np.tile(np.array([1, 0], np.float32), (2, T, 1, 1)), W.F16)
    out, lse = O.attend_multi(x, qm)
    for b in range(2):
        for i in range(T):
            assert np.allclose(out[b, i, 0], g[f"out{b}"][i], rtol=0, atol=1e-12), (b, i)
            want = g[f"lse{b}"][0][i]
            if math.isinf(want):
                assert math.isinf(lse[b, i, 0]) and lse[b, i, 0] < 0, (b, i)
            else:
                assert abs(lse[b, i, 0] - want) < 1e-12, (b, i)
    assert math.isclose(g["lse0"][0][1], math.log(24), abs_tol=1e-15)


def test_workqueue_small():
    g = _read("workqueue_small.txt")
    lens = [int(t) for t in _one(g, "seq_lens")]
    r = O.workqueue(lens, int(_one(g, "Hkv")[0]), 16, int(_one(g, "chunk")[0]))
    assert r["tasks"].tolist() == [[int(t) for t in row] for row in g["task"]]
    assert r["chunk_begin"].tolist() == [int(t) for t in _one(g, "chunk_begin")]
    assert r["seq_group_begin"].tolist() == [int(t) for t in _one(g, "seq_group_begin")]
    assert r["seq_nsplit"].tolist() == [int(t) for t in _one(g, "seq_nsplit")]


def _pool(P=16, d=8):
    rng = np.random.default_rng(0)
    return (rng.integers(0, 1 << 14, size=(P, 1, 16, d)).astype(np.uint16),
            rng.integers(0, 1 << 14, size=(P, 1, 16, d)).astype(np.uint16))


def test_compact_token_mask():
    g = _read("compact_small.txt")
    k, v = _pool()
    table = np.full((1, 4), -1, np.int32)
    old = [int(t) for t in _one(g, "tok_table")]
    table[0, : len(old)] = old
    L = int(_one(g, "tok_len")[0])
    keep = np.zeros((1, 4 * 16), np.uint8)
    keep[0, :L] = 1
    for t in _one(g, "tok_drop"):
        keep[0, int(t)] = 0
    fr = [int(t) for t in _one(g, "tok_free")]
    free = np.full(16, -1, np.int32)
    free[: len(fr)] = fr
    t, sl, kp, vp, fl, top, rc = O.compact(table, np.array([L], np.int32), keep, True, k, v,
                                           free, len(fr), 1, 8, 16)
    assert rc == 0
    new = [int(x) for x in _one(g, "tok_new_table")]
    assert t[0, : len(new)].tolist() == new and (t[0, len(new):] == -1).all()
    assert sl.tolist() == [int(_one(g, "tok_new_len")[0])]
    assert fl[:top].tolist() == [int(x) for x in _one(g, "tok_new_free")]
    sp, ss, dp, ds = (int(x) for x in _one(g, "tok_moved"))
    assert np.array_equal(kp[dp, 0, ds], k[sp, 0, ss]) and np.array_equal(vp[dp, 0, ds], v[sp, 0, ss])


def test_compact_page_mask():
    g = _read("compact_small.txt")
    k, v = _pool()
    table = np.full((1, 4), -1, np.int32)
    old = [int(t) for t in _one(g, "pg_table")]
    table[0, : len(old)] = old
    keep = np.zeros((1, 4), np.uint8)
    keep[0, : len(old)] = [int(x) for x in _one(g, "pg_keep")]
    fr = [int(t) for t in _one(g, "pg_free")]
    free = np.full(16, -1, np.int32)
    free[: len(fr)] = fr
    t, sl, kp, vp, fl, top, rc = O.compact(table, np.array([int(_one(g, "pg_len")[0])], np.int32),
                                           keep, False, k, v, free, len(fr), 1, 8, 16)
    assert rc == 0
    new = [int(x) for x in _one(g, "pg_new_table")]
    assert t[0, : len(new)].tolist() == new
    assert sl.tolist() == [int(_one(g, "pg_new_len")[0])]
    assert fl[:top].tolist() == [int(x) for x in _one(g, "pg_new_free")]
    assert np.array_equal(kp, k) and np.array_equal(vp, v)
