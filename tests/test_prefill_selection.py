"""The prefill workload's Top-K is shaped by its inputs, not by position or rounding.

The 16384-token causal prefill draws its indexer keys and queries as N(0, 1) plus a
rank-8 structured component of per-element std 0.5.  These CPU checks run the
oracle on sampled query rows of that exact workload (the indexer inputs do not
depend on the number of attention heads, which is cut to 1 here to keep the draw
small) and show that:

* the selection is not a recency window: the share of the last K positions among
  the chosen ones stays at the chance rate K / n;
* the structured component decides a large part of the selection: the same seed
  with the structure's amplitude set to 0 (the draw order is unchanged, so the
  N(0, 1) part is bit-identical) keeps under 80 % of the chosen positions, yet
  clearly more than chance, so both parts of the input matter;
* the K-th score is decided by value: the scores straddling the boundary differ
  and at most a couple of positions tie there.
"""
import numpy as np
import pytest

import dsa_workloads as W
from oracle import dsa_oracle as O

ROWS = [4095, 6000, 8191, 12287, 14000, 16383]


@pytest.fixture(scope="module")
def selections():
    out = {}
    for amp in (0.5, 0.0):
        wl = W.make(W.spec("prefill_16k", H=1, low_rank_amp=amp), seed=0)
        assert wl.K == 2048 and wl.max_ctx == 16384
        scores = O.indexer_scores(wl, ROWS)
        out[amp] = (scores, O.topk(scores, wl.q_pos[ROWS], wl.K))
        del wl
    return out


def test_selection_is_not_a_recency_window(selections):
    _, sel = selections[0.5]
    K = sel.shape[1]
    for i, t in enumerate(ROWS):
        n = t + 1
        recent = np.count_nonzero(sel[i] >= n - K) / K
        assert abs(recent - K / n) < 0.05, (t, recent, K / n)


def test_structured_component_moves_the_selection(selections):
    _, with_s = selections[0.5]
    _, without = selections[0.0]
    K = with_s.shape[1]
    shared = []
    for i, t in enumerate(ROWS):
        same = np.intersect1d(with_s[i], without[i]).size / K
        chance = K / (t + 1)
        assert chance + 0.1 < same < 0.8, (t, same, chance)
        shared.append(same)
    assert np.mean(shared) < 0.65


def test_boundary_is_decided_by_value(selections):
    scores, sel = selections[0.5]
    K = sel.shape[1]
    for i, t in enumerate(ROWS):
        row = scores[i, :t + 1]
        desc = np.sort(row)[::-1]
        assert desc[K - 1] > desc[K], t
        assert np.count_nonzero(row == desc[K - 1]) <= 2
        # the chosen positions are exactly those scoring at least the K-th value
        assert np.array_equal(np.sort(sel[i]), np.flatnonzero(row >= desc[K - 1]))
