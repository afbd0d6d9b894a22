"""The oracle's pins against planted mistakes.

Each case below plants one plausible mistake in a copy of an oracle function
(a dropped or doubled term, a wrong sign, a transposed operand, an
off-by-one, a wrong tie rule, a skipped bookkeeping step) and runs a battery
of the pin tests against it; at least one pin must fail.  The unmodified
oracle passes the same batteries.  Mistakes are planted only in the oracle,
on the CPU, for the duration of one test (pytest's monkeypatch).
"""
import heapq as _heapq
import inspect
import textwrap

import numpy as np
import pytest

from oracle import attention as A
from oracle import fp8 as F8
from oracle import pakv as P
from oracle import schedule as SCH
from tests import test_oracle_attention as TA
from tests import test_oracle_fp8 as TF
from tests import test_oracle_pakv as TP
from tests import test_oracle_schedule as TS


# ---------------------------------------------------------------- batteries
def _attention_battery():
    return [
        TA.test_hand_computed_two_token_example,
        lambda: TA.test_softmax_attention_matches_brute_force(17, 3, 5),
        TA.test_constant_v_returns_v,
        TA.test_zero_query_gives_mean_of_v,
        TA.test_single_token_context_returns_its_value,
        TA.test_dominant_key_returns_its_value,
        TA.test_scores_use_the_scale,
        TA.test_partial_triple_against_brute_force,
        lambda: TA.test_merge_identity_any_split(3),
        TA.test_merge_needs_the_rescale,
        TA.test_two_phase_single_prefix_equals_definition,
        TA.test_decode_attention_over_trie_matches_brute_force,
        lambda: TA.test_grouped_query_attention_equals_repeated_kv(2),
        lambda: TA.test_multi_token_queries_with_one_token_are_decode_attention(True),
        TA.test_causal_queries_over_a_whole_sequence_are_causal_self_attention,
        TA.test_multi_token_queries_match_the_two_phase_form,
    ]


def _fp8_battery():
    cases = [lambda c=c, v=v: TF.test_landmark_codes(c, v) for c, v in
             [(0x38, 1.0), (0x7E, 448.0), (0x01, 2.0 ** -9), (0x77, 240.0), (0x08, 2.0 ** -6)]]
    cases += [lambda y=y, c=c: TF.test_rounding_ties_subnormals_saturation(y, c) for y, c in
              [(1.0625, 0x38), (1.1875, 0x3A), (3 * 2.0 ** -10, 0x02), (464.0, 0x7E), (-0.0, 0x80)]]
    return cases + [TF.test_nan_codes_and_count_of_finite_values, TF.test_encode_is_nearest_by_brute_force,
                    TF.test_quantize_uses_fp32_reciprocal_scale]


def _trie_battery():
    return [
        TP.test_storage_model_lp_plus_n_ls,
        lambda: TP.test_sharing_matches_brute_force(1, 2),
        lambda: TP.test_remove_everything_frees_every_slot(2),
        TP.test_lowest_free_slot_first_and_reuse,
        TP.test_partial_tail_is_never_shared,
        TP.test_golden_ops_slots_and_stats,
        lambda: TP.test_appends_keep_counts_and_context(1),
    ]


def _schedule_battery():
    return [
        TS.test_golden_schedule_tables,
        lambda: TS.test_random_tree_tables_and_two_phase_equal_definition(4, 2),
        TS.test_batch_permutation_invariance,
    ]


def _failures(battery):
    failed = 0
    for case in battery:
        try:
            case()
        except Exception:                      # a pin tripped (assertion or an error it provoked)
            failed += 1
    return failed


@pytest.mark.parametrize("battery", [_attention_battery, _fp8_battery, _trie_battery, _schedule_battery])
def test_unmodified_oracle_passes_every_pin(battery):
    assert _failures(battery()) == 0


# ------------------------------------------------------- attention mutants
def _softmax_variant(scale_mul=1.0, values_from_keys=False, head_map=None, norm_axis=1, drop_last=False):
    def f(q, k, v, scale):
        q = np.asarray(q, dtype=np.float64)
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        if k.shape[0] == 0:
            raise P.OracleError("invalid", "empty context")
        if drop_last and k.shape[0] > 1:
            k, v = k[:-1], v[:-1]
        g = (head_map or A.kv_head_of)(q.shape[0], k.shape[1])
        k, v = k[:, g], v[:, g]
        x = scale * scale_mul * np.einsum("hd,nhd->hn", q, k)
        w = np.exp(x - x.max(axis=1, keepdims=True))
        w /= w.sum(axis=norm_axis, keepdims=True)
        return np.einsum("hn,nhd->hd", w, k if values_from_keys else v)
    return f


def _partial_unshifted_sum(q, k, v, scale):
    o, m, s = _REAL["partial"](q, k, v, scale)
    return o, m, s * np.exp(m)                    # s without the max shift, o with it


def _merge_variant(sign=1.0, weight_sums=True):
    def f(parts):
        parts = list(parts)
        mstar = np.stack([p[1] for p in parts]).max(axis=0)
        num, den = np.zeros_like(parts[0][0]), np.zeros_like(parts[0][2])
        for o, m, s in parts:
            w = np.where(np.isneginf(m), 0.0, np.exp(sign * (m - mstar)))
            num += w[:, None] * o
            den += (w * s) if weight_sums else s
        return num / den[:, None]
    return f


def _causal_off_by_one(trie, seq_ids, layer, q, scale, causal=False):
    q = np.asarray(q, dtype=np.float64)
    out = np.empty(q.shape, dtype=np.float64)
    for i, s in enumerate(seq_ids):
        k, v = trie.materialize(int(s), layer)
        n, q_len = k.shape[0], q.shape[1]
        for j in range(q_len):
            lim = max(1, n - q_len + j) if causal else n         # one token short
            out[i, j] = A.softmax_attention(q[i, j], k[:lim], v[:lim], scale)
    return out


_REAL = {"partial": A.partial}

ATTENTION_MUTANTS = {
    "scale dropped": ("softmax_attention", _softmax_variant(scale_mul=0.0)),
    "scale applied twice": ("softmax_attention", _softmax_variant(scale_mul=0.5)),
    "keys used as values": ("softmax_attention", _softmax_variant(values_from_keys=True)),
    "query head -> kv head by modulo": ("softmax_attention",
                                        _softmax_variant(head_map=lambda hq, hk: np.arange(hq) % hk)),
    "normalised over heads": ("softmax_attention", _softmax_variant(norm_axis=0)),
    "last context token dropped": ("softmax_attention", _softmax_variant(drop_last=True)),
    "partial sum without the max shift": ("partial", _partial_unshifted_sum),
    "merge rescale with the wrong sign": ("merge", _merge_variant(sign=-1.0)),
    "merge sums not rescaled": ("merge", _merge_variant(weight_sums=False)),
    "causal limit one short": ("decode_attention_multi", _causal_off_by_one),
}


@pytest.mark.parametrize("name", list(ATTENTION_MUTANTS))
def test_attention_pins_catch(name, monkeypatch):
    attr, fn = ATTENTION_MUTANTS[name]
    monkeypatch.setattr(A, attr, fn)
    assert _failures(_attention_battery()) > 0, name


# ------------------------------------------------------------ fp8 mutants
def _values(bias=7, subnormals=True):
    vals = np.empty(256)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e, m = (code >> 3) & 0xF, code & 0x7
        if e == 15 and m == 7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = s * 2.0 ** (1 - bias) * (m / 8.0) if subnormals else s * 0.0
        else:
            vals[code] = s * 2.0 ** (e - bias) * (1.0 + m / 8.0)
    return vals


def _encode_ties_away(y):
    y = np.asarray(y, dtype=np.float32).astype(np.float64)
    a = np.minimum(np.abs(y), F8.MAX_FINITE)
    pos = F8.CODE_VALUES[:0x7F]
    hi = np.minimum(np.searchsorted(pos, a, side="left"), len(pos) - 1)
    lo = np.maximum(hi - 1, 0)
    pick_hi = (pos[hi] - a) <= (a - pos[lo])                  # ties go up, not to even
    mag = np.where(pick_hi, hi, lo)
    return (mag | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def _encode_no_saturation(y):
    codes = _REAL_ENCODE(y)
    y = np.asarray(y, dtype=np.float32)
    return np.where(np.abs(y) > F8.MAX_FINITE, np.where(np.signbit(y), 0xFF, 0x7F), codes).astype(np.uint8)


def _quantize_times_scale(x, scale):
    return F8.encode(np.asarray(x, dtype=np.float16).astype(np.float32) * np.float32(scale))


_REAL_ENCODE = F8.encode

FP8_MUTANTS = {
    "exponent bias 8": {"CODE_VALUES": _values(bias=8)},
    "subnormals flushed": {"CODE_VALUES": _values(subnormals=False)},
    "ties away from zero": {"encode": _encode_ties_away},
    "no saturation (NaN code)": {"encode": _encode_no_saturation},
    "scale multiplied, not divided": {"quantize": _quantize_times_scale},
}


@pytest.mark.parametrize("name", list(FP8_MUTANTS))
def test_fp8_pins_catch(name, monkeypatch):
    for attr, val in FP8_MUTANTS[name].items():
        monkeypatch.setattr(F8, attr, val)
        if attr == "CODE_VALUES":                    # the encoder's sorted table follows it
            monkeypatch.setattr(F8, "_POS_VALUES", val[:0x7F])
    assert _failures(_fp8_battery()) > 0, name


# ---------------------------------------------------- trie and schedule mutants
class _MaxHeap:
    """heapq stand-in that hands out the highest free slot first."""
    heapify = staticmethod(lambda h: h.sort())
    heappush = staticmethod(lambda h, x: (h.append(x), h.sort()))
    heappop = staticmethod(lambda h: h.pop())


def _mutated_method(cls, name, *subs):
    """The class's own method with textual substitutions applied, compiled in
    its module's namespace: a mutant that differs from the oracle exactly
    where the substitution says."""
    src = textwrap.dedent(inspect.getsource(getattr(cls, name)))
    for old, new in subs:
        assert old in src, old
        src = src.replace(old, new)
    ns = {}
    exec(compile(src, f"<mutant {name}>", "exec"), vars(inspect.getmodule(cls)), ns)
    return ns[name]


# the partial last piece is walked and registered like a full chunk
_insert_shares_tails = _mutated_method(
    P.OracleTrie, "insert",
    ("for key in pieces[:n_full]:", "for key in pieces:"),
    ("if len(key) == c and not self.no_sharing:", "if not self.no_sharing:"))


def _insert_no_match_refcount(self, seq_id, tokens, k=None, v=None):
    n = _REAL_INSERT(self, seq_id, tokens, k, v)
    for node in self.paths[seq_id][:n // self.chunk]:
        node.refcount -= 1                              # matched chunks not counted
    return n


def _remove_keeps_slots(self, seq_id):
    held = list(self.free)
    _REAL_REMOVE(self, seq_id)
    self.free[:] = held                                  # freed slots never return
    _heapq.heapify(self.free)


_REAL_INSERT, _REAL_REMOVE = P.OracleTrie.insert, P.OracleTrie.remove


def _schedule_drop_last_sharer(trie, seq_ids):
    t = _REAL_SCHEDULE(trie, seq_ids)
    runs = t["cf_runs"].copy()
    if len(runs):
        runs[0, 3] -= 1                                  # one sharer left out of a run
        t["cf_runs"] = runs
    return t


def _schedule_sf_reversed(trie, seq_ids):
    t = _REAL_SCHEDULE(trie, seq_ids)
    sf = t["sf_chunks"].copy()
    offs = t["sf_offsets"]
    for p in range(len(offs) - 1):
        sf[offs[p]:offs[p + 1]] = sf[offs[p]:offs[p + 1]][::-1]   # path order lost
    t["sf_chunks"] = sf
    return t


_REAL_SCHEDULE = SCH.build_schedule

TRIE_MUTANTS = {
    "highest free slot first": lambda mp: mp.setattr(P, "heapq", _MaxHeap),
    "partial tail chunks shared": lambda mp: mp.setattr(P.OracleTrie, "insert", _insert_shares_tails),
    "matched chunks not refcounted": lambda mp: mp.setattr(P.OracleTrie, "insert", _insert_no_match_refcount),
    "removed chunks keep their slots": lambda mp: mp.setattr(P.OracleTrie, "remove", _remove_keeps_slots),
}

SCHEDULE_MUTANTS = {
    "a sharer left out of a chunk-first run": _schedule_drop_last_sharer,
    "private chunks out of path order": _schedule_sf_reversed,
}


@pytest.mark.parametrize("name", list(TRIE_MUTANTS))
def test_trie_pins_catch(name, monkeypatch):
    TRIE_MUTANTS[name](monkeypatch)
    assert _failures(_trie_battery()) > 0, name


@pytest.mark.parametrize("name", list(SCHEDULE_MUTANTS))
def test_schedule_pins_catch(name, monkeypatch):
    monkeypatch.setattr(TS, "build_schedule", SCHEDULE_MUTANTS[name])
    assert _failures(_schedule_battery()) > 0, name
