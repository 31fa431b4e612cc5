"""Plant plausible mistakes in the CPU oracle and show the pins catch each one.

Every mutation replaces one oracle function (on the CPU, for the duration of
one test) with a subtly wrong variant; at least one pin must then fail. This
is what makes the pins evidence rather than a restatement of the oracle.
"""
import math

import pytest
import torch

from oracle import sva_oracle as O
from tests import oracle_pins as P

_orig_anc = O.ancestors
_orig_sw = O._softmax_weighted_sum
_orig_scores = O.block_scores
_orig_select = O.select_blocks
_orig_budget = O.budget_blocks
_orig_reps = O.block_representatives
_orig_sparse = O.sparse_attend
_orig_kept = O.smooth_kept_tokens
_orig_depths = O.draft_depths


def _anc_transposed(parents, t):        # sees later drafts instead of earlier ones
    return list(range(t, len(parents)))


def _anc_without_self(parents, t):      # forgets the draft's own key
    return [u for u in _orig_anc(parents, t) if u != t] or [t]


def _sw_no_norm(scores, values):        # drops the softmax denominator
    m = scores.max()
    return torch.exp(scores - m) @ values


def _sw_unscaled(scores, values):       # softmax without the 1/sqrt(d) scale
    return _orig_sw(scores * 4.0, values)


def _scores_last_draft(q, reps, G):     # scores with the last draft's query
    return _orig_scores(q.flip(1), reps, G)


def _scores_head_mod(q, reps, G):       # maps query head qh to KV head qh % Hkv
    B, T, Hq, d = q.shape
    Hkv = Hq // G
    perm = [(qh % Hkv) * G + (qh // Hkv) for qh in range(Hq)]
    inv = [perm.index(i) for i in range(Hq)]
    return _orig_scores(q[:, :, inv], reps, G)


def _select_high_tie(scores_row, k):    # ties to the higher index
    vals = [float(x) for x in scores_row]
    order = sorted(range(len(vals)), key=lambda j: (-vals[j], -j))
    return sorted(order[:k])


def _select_lowest(scores_row, k):      # keeps the lowest scores
    return _orig_select([-float(x) for x in scores_row], k)


def _budget_no_floor(ctx, nb, mode, fixed=0, short=0, floor=0, fm=0.0, lc=0, fl=0.0):
    return _orig_budget(ctx, nb, mode, fixed, short, 0, fm, lc, fl)


def _budget_floor_division(ctx, nb, mode, fixed=0, short=0, floor=0, fm=0.0, lc=0, fl=0.0):
    if mode == O.BUDGET_FIXED or ctx <= short:
        return _orig_budget(ctx, nb, mode, fixed, short, floor, fm, lc, fl)
    frac = fm if ctx <= lc else fl
    return min(nb, max(floor, int(frac * nb)))


def _kept_mid_dropped(ctx, short, fm, lc, fl):  # forgets the middle piece
    return _orig_kept(ctx, short, 0.0, lc, fl)


def _kept_rates_swapped(ctx, short, fm, lc, fl):  # long rate on the middle piece
    return _orig_kept(ctx, short, fl, lc, fm)


def _reps_off_by_one(k_pool, block_table, n_blocks, blk):
    return _orig_reps(k_pool, block_table, n_blocks, blk) * blk / (blk + 1)


def _sparse_heads_mod(q, k_pool, v_pool, bt, sel, dk, dv, parents, **kw):
    B, T, Hq, d = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    perm = [(qh % Hkv) * G + (qh // Hkv) for qh in range(Hq)]
    inv = [perm.index(i) for i in range(Hq)]
    return _orig_sparse(q[:, :, inv], k_pool, v_pool, bt, sel, dk, dv, parents, **kw)[:, :, perm]


def _sparse_tail_dropped(q, k_pool, v_pool, bt, sel, dk, dv, parents, tail_block=0, tail_len=0):
    return _orig_sparse(q, k_pool, v_pool, bt, sel, dk, dv, parents)  # forgets the partial block


def _depths_as_index(parents):          # position distance = index distance, not depth
    return list(range(len(parents)))


MUTATIONS = {
    "mask_transposed": ("ancestors", _anc_transposed),
    "mask_without_self": ("ancestors", _anc_without_self),
    "softmax_unnormalised": ("_softmax_weighted_sum", _sw_no_norm),
    "softmax_unscaled": ("_softmax_weighted_sum", _sw_unscaled),
    "score_last_draft": ("block_scores", _scores_last_draft),
    "score_head_mapping": ("block_scores", _scores_head_mod),
    "select_ties_high": ("select_blocks", _select_high_tie),
    "select_lowest": ("select_blocks", _select_lowest),
    "budget_no_floor": ("budget_blocks", _budget_no_floor),
    "budget_floor_division": ("budget_blocks", _budget_floor_division),
    "smooth_mid_dropped": ("smooth_kept_tokens", _kept_mid_dropped),
    "smooth_rates_swapped": ("smooth_kept_tokens", _kept_rates_swapped),
    "reps_wrong_divisor": ("block_representatives", _reps_off_by_one),
    "attend_head_mapping": ("sparse_attend", _sparse_heads_mod),
    "attend_tail_dropped": ("sparse_attend", _sparse_tail_dropped),
    "overlap_index_distance": ("draft_depths", _depths_as_index),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_some_pin_catches(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(O)
        except AssertionError:
            caught.append(pin.__name__)
        except Exception:               # a crash in the mutated oracle also counts
            caught.append(pin.__name__ + "(error)")
    assert caught, f"no pin catches mutation {name}"
