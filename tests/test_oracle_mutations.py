"""Planted mistakes in the CPU oracle must be caught by its pins.

Each case replaces one step of the oracle with a plausible wrong version: a dropped term, a
flipped sign, a shifted mask, a reversed tie-break, a transposed index, a wrong grouping of the
query heads. It then runs the pins of test_oracle_pins.py and requires at least one to fail.
The pins are checked against the pages and the mathematics, so they do not only agree with the
oracle as written: they would catch these mistakes. The mistakes are planted in the oracle on
the CPU; the CUDA path is not involved.
"""
import numpy as np
import pytest

import test_oracle_pins as P
from oracle import zipage_oracle as O

PINS = (
    [(P.test_two_block_hand_example_attention, {}), (P.test_two_block_hand_example_redundancy, {})]
    + [(P.test_two_block_hand_example_scores_and_selection, {"case": c}) for c in range(5)]
    + [(P.test_two_block_hand_example_global_update, {"case": c}) for c in range(5)]
    + [(P.test_attention_mass_is_one, {"causal": c}) for c in (True, False)]
    + [(P.test_identical_keys_causal_closed_form, {}), (P.test_window_row_position_and_mask, {}),
       (P.test_gqa_grouping_is_contiguous, {}), (P.test_redundancy_special_cases, {})]
    + [(P.test_lightning_equals_all_pairs_same_block, {"L": L, "b": b}) for L, b in [(64, 16), (40, 16), (17, 4)]]
    + [(P.test_selection_equals_rank_counting, {"seed": s}) for s in range(3)]
    + [(P.test_selection_tie_keeps_earlier, {}), (P.test_global_score_dominates_known_keep_set, {})]
    + [(P.test_pass_invariants, {"prefix": p}) for p in (0, 3)]
    + [(P.test_slot_location_hand_example, {}), (P.test_pass_invariants_after_prefill, {})]
)


def _failing_pins():
    failed = []
    for fn, kw in PINS:
        try:
            fn(**kw)
        except Exception:  # a failed assertion, or a crash the mistake causes
            failed.append(f"{fn.__name__}{kw or ''}")
    return failed


def _block_sizes(L, b):
    """Tokens held by the block of each position (the last block may be partial)."""
    t = np.arange(L)
    return np.minimum(b, L - (t // b) * b)


def _ignore_causality(orig):
    return lambda q, k, scale, causal=True: orig(q, k, scale, False)


def _no_group_average(orig):
    # averages over the window rows only: the sum over the G_q heads is not divided by G_q
    return lambda q, k, scale, causal=True: orig(q, k, scale, causal) * q.shape[1]


def _redundancy_with_self(orig):
    def f(k, b):
        R, m = orig(k, b), _block_sizes(len(k), b)
        return np.where(m > 1, (R * (m - 1) + 1.0) / m, 1.0)
    return f


def _redundancy_over_m(orig):
    def f(k, b):
        R, m = orig(k, b), _block_sizes(len(k), b)
        return R * (m - 1) / m
    return f


def _redundancy_sign(orig):
    return lambda attn, G, R, alpha, beta, window, protect: orig(attn, G, -np.asarray(R), alpha, beta, window, protect)


def _global_score_dropped(orig):
    return lambda attn, G, R, alpha, beta, window, protect: orig(attn, 0 * np.asarray(G), R, alpha, beta, window,
                                                                 protect)


def _window_one_short(orig):
    return lambda attn, G, R, alpha, beta, window, protect: orig(attn, G, R, alpha, beta, window - 1, protect)


def _tie_keeps_later(orig):
    def f(S, k):
        S = np.asarray(S)
        return np.sort(len(S) - 1 - orig(S[::-1].copy(), k))
    return f


def _keeps_lowest(orig):
    return lambda S, k: orig(-np.asarray(S, dtype=np.float64), k)


def _decay_on_attention(orig):
    return lambda G, attn, src, decay, L: orig(G, decay * np.asarray(attn, np.float64), src, decay, L)


def _tail_not_cleared(orig):
    def f(G, attn, src, decay, L):
        out = orig(G, attn, src, decay, L)
        out[len(src):L] = np.asarray(G, np.float64)[len(src):L]
        return out
    return f


def _update_indexed_by_position(orig):
    # survivor scores left at their source positions t instead of compacted to slots j
    def f(G, attn, src, decay, L):
        out = np.zeros(L)
        src = np.asarray(src)
        out[src] = decay * np.asarray(G, np.float64)[src] + np.asarray(attn, np.float64)[src]
        return out
    return f


def _update_attention_of_slot(orig):
    # slot j takes the attention of position j instead of its source token's
    def f(G, attn, src, decay, L):
        out = orig(G, attn, src, decay, L)
        k = len(src)
        out[:k] += np.asarray(attn, np.float64)[:k] - np.asarray(attn, np.float64)[np.asarray(src)]
        return out
    return f


def _update_decay_complement(orig):
    # (1 - decay) in place of decay
    return lambda G, attn, src, decay, L: orig(G, attn, src, 1.0 - decay, L)


def _shared_blocks_in_place(orig):
    def f(table, n_max, refcount, free_ids):
        return np.array(table[:n_max - 1], dtype=np.int32).copy(), []
    return f


def _slot_transposed(orig):
    # block index and row inside the block swapped (t // b <-> t % b)
    return lambda table, slot, b: (int(table[slot % b]), slot // b)


def _interleaved_groups(orig):
    # query head g*H_kv + h serves kv head h (interleaved) instead of h*G_q + g (contiguous)
    def f(pool, block_tables, dst_tables, seq_len, qslot, obs_q, global_scores, p, **kw):
        hkv, hq = pool.shape[3], p["num_q_heads"]
        g = hq // hkv
        perm = [gi * hkv + h for h in range(hkv) for gi in range(g)]
        return orig(pool, block_tables, dst_tables, seq_len, qslot, obs_q[..., perm, :], global_scores, p, **kw)
    return f


MUTANTS = {
    "causal mask ignored": ("window_attention", _ignore_causality),
    "no average over the query group": ("window_attention", _no_group_average),
    "redundancy counts the key itself": ("lightning_redundancy", _redundancy_with_self),
    "redundancy divided by m, not m - 1": ("lightning_redundancy", _redundancy_over_m),
    "redundancy added instead of subtracted": ("combine_scores", _redundancy_sign),
    "global score dropped": ("combine_scores", _global_score_dropped),
    "protected window one token short": ("combine_scores", _window_one_short),
    "tie keeps the later token": ("select_keep", _tie_keeps_later),
    "lowest scores kept": ("select_keep", _keeps_lowest),
    "decay applied to the attention too": ("global_update", _decay_on_attention),
    "global-score tail not cleared": ("global_update", _tail_not_cleared),
    "global score left at the source position": ("global_update", _update_indexed_by_position),
    "global score takes the attention of the slot": ("global_update", _update_attention_of_slot),
    "global score decayed by 1 - decay": ("global_update", _update_decay_complement),
    "shared prefix blocks compacted in place": ("plan_dst_table", _shared_blocks_in_place),
    "block and row of a slot transposed": ("slot_location", _slot_transposed),
    "query heads grouped interleaved": ("compress_pass", _interleaved_groups),
}


def test_unmodified_oracle_passes_every_pin():
    assert _failing_pins() == []


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_fails_a_pin(monkeypatch, name):
    attr, make = MUTANTS[name]
    monkeypatch.setattr(O, attr, make(getattr(O, attr)))
    assert _failing_pins(), f"no pin catches the planted mistake: {name}"


GLOBAL_UPDATE_MUTANTS = ["decay applied to the attention too", "global score left at the source position",
                         "global score takes the attention of the slot", "global score decayed by 1 - decay"]


@pytest.mark.parametrize("name", GLOBAL_UPDATE_MUTANTS)
def test_global_update_mistake_fails_the_hand_worked_values(monkeypatch, name):
    # The update rule is pinned by the hand-worked values of the golden file; the pass-level
    # invariants check only that the pass applies the (pinned) rule to its kept set.
    attr, make = MUTANTS[name]
    monkeypatch.setattr(O, attr, make(getattr(O, attr)))
    failed = []
    for c in range(5):
        try:
            P.test_two_block_hand_example_global_update(case=c)
        except AssertionError:
            failed.append(c)
    assert failed, f"the hand-worked global-score values miss the planted mistake: {name}"
