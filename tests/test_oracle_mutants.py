"""Plant a mistake in a copy of the oracle (on the CPU) and check that at
least one pin fails.  Each mutant is a plausible slip: a wrong index, a
dropped factor, a flipped sign or comparison, a reversed order."""
import os

import pytest

from oracle import oracle as O
from tests import oracle_pins

# (name, text in oracle.c, replacement, occurrence index to replace)
MUTANTS = [
    ("gqa_map", "int h = hq / G;", "int h = hq % a->Hkv;", 0),
    ("scale_dropped", "s[t - t0] = a->scale * dot;", "s[t - t0] = dot;", 0),
    ("lse_sign", "*lse = m + log(sum);", "*lse = m - log(sum);", 0),
    ("slot_index", "+ t % a->ps) * d;", "+ (t + 1) % a->ps) * d;", 0),
    ("value_page", "const uint16_t *vt = a->v_pool + (((size_t)page * a->Hkv + h)",
     "const uint16_t *vt = a->v_pool + (((size_t)(page ^ 1) * a->Hkv + h)", 0),
    ("merge_weight", "double w = exp(lse_parts[s] - *lse);", "double w = exp(lse_parts[s] - m);", 0),
    ("wq_first_chunk", "int64_t c_first = O / chunk", "int64_t c_first = (O + 1) / chunk", 0),
    ("wq_page_end", "r[5] = (int32_t)(hi - O);", "r[5] = (int32_t)(hi - O - 1);", 0),
    ("multi_causal", "int64_t lim = (int64_t)a.seq_lens[b] - T + 1 + i;",
     "int64_t lim = (int64_t)a.seq_lens[b] - T + i;", 0),
    ("multi_q_row", "a.q = pool->q + (size_t)i * Hq * d;", "a.q = pool->q + (size_t)(T - 1 - i) * Hq * d;", 0),
    ("f16_bias", "v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);", 0),
    ("bf16_subnormal", "v = ldexp((double)m, -133);", "v = ldexp((double)m, -134);", 0),
    ("ema_decay_swap", "*e = first ? gm : a[u] * *e + (1.0 - a[u]) * gm;",
     "*e = first ? gm : (1.0 - a[u]) * *e + a[u] * gm;", 0),
    ("ema32_one_minus", "float om = 1.0f - a[u];", "float om = a[u];", 0),
    ("summary_mean", "s[c] = acc / ps;", "s[c] = acc / (ps - 1);", 0),
    ("summary_min", "if (x < mn) mn = x;", "if (x > mn) mn = x;", 1),
    ("score_bound_min", "acc += uu * s[c] + (ta > tb ? ta : tb);", "acc += uu * s[c] + (ta < tb ? ta : tb);", 0),
    ("score32_butterfly", "nxt[l] = acc[l] + acc[l ^ sft];", "nxt[l] = acc[l] + acc[l ^ (sft >> 1)];", 0),
    ("topk_tiebreak", "return a->j < b->j ? -1 : (a->j > b->j ? 1 : 0);",
     "return a->j > b->j ? -1 : (a->j < b->j ? 1 : 0);", 0),
    ("forced_last", "(j >= n - n_last)", "(j > n - n_last)", 0),
    ("grow_compare", "wants = (float)D > thr;", "wants = (float)D >= thr;", 0),
    ("grow_grant_order", "if (wants && granted < free_count) {", "if (wants && granted <= free_count) {", 0),
    ("ws_size", "int w = (int)ceilf(ws_frac * (float)nc);", "int w = (int)(ws_frac * (float)nc);", 0),
    ("drift_direction", "D += wf[cands[i]] && !ws[cands[i]];", "D += wf[cands[i]] && ws[cands[i]];", 0),
    ("compact_reuse_count", "int reuse = (t0 % ps) == 0;", "int reuse = 0;", 0),
    ("compact_reuse_apply", "int reuse = (t0 % ps) == 0;", "int reuse = 0;", 1),
    ("compact_reuse_slots", "reuse = kept[b][m * ps + s] == t0 + s;", "reuse = kept[b][m * ps + s] >= t0 + s;", 1),
    ("compact_push_order", "free_list[top++] = freed[i];", "free_list[top++] = freed[nfreed - 1 - i];", 0),
    ("append_pop", "      *slot = free_list[--top];", "      *slot = free_list[top-- - 2];", 0),
    ("cow_copy_len", "sizeof(uint16_t) * (size_t)(L % ps) * d);", "sizeof(uint16_t) * (size_t)(L % ps - 1) * d);", 0),
    ("cow_old_ref", "refcnt[old] -= 1;", "refcnt[old] -= 0;", 0),
    ("shared_free", "if (refcnt[freed[i]] != 0) continue;", "if (refcnt[freed[i]] < 0) continue;", 0),
    ("mark_boundary", "L / ps >= budget[b]", "L / ps > budget[b]", 0),
]


def _replace_nth(text, old, new, n):
    idx = -1
    for _ in range(n + 1):
        idx = text.find(old, idx + 1)
        assert idx >= 0, f"mutant anchor not found: {old!r}"
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, nth, tmp_path):
    src = _replace_nth(O.source(), old, new, nth)
    so = O.build_variant(src, os.path.join(str(tmp_path), f"liboracle_{name}.so"))
    caught = None
    with O.using(so):
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except (AssertionError, O.OracleError, IndexError, ValueError) as e:
                caught = (pin.__name__, type(e).__name__)
                break
    assert caught is not None, f"no pin detects mutant {name}"
