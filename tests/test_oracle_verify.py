"""Pins of the oracle's greedy verification (CPU only).

"Attention Drift", section 2 (preliminaries): the target scores the drafted
tokens in one forward pass and keeps the longest prefix it accepts.  With greedy
drafts the target's distribution is read at temperature 0, so a draft is
accepted when it equals the target's greedy token of the row before it.

The checks below are written from that rule and from the definition of a
greedy pick, not from the oracle's own loops: exhaustive enumeration on tiny
vocabularies, the single-row case (plain next-token decoding), recovery of the
values the input generator plants, and the hand-off to the next step's batch
metadata ("P-EAGLE: parallel speculative decoding in vLLM", Parallel drafting:
the NTP row carries the new token).
"""

import itertools
import math

import numpy as np
import pytest

from oracle import pe_oracle as O
from speculative_drafting_gb300 import workloads as W


def _greedy_by_definition(x):
    """Index i with x[i] >= every x[j] and x[j] < x[i] for every j < i; a NaN is
    above every number and the first NaN wins."""
    nan = [i for i, v in enumerate(x) if math.isnan(v)]
    if nan:
        return nan[0]
    for i, v in enumerate(x):
        if all(v >= w for w in x) and all(w < v for w in x[:i]):
            return i
    raise AssertionError("no greatest element")


def test_greedy_pick_enumerated():
    values = [-1.0, -0.0, 0.0, 2.0, float("nan")]
    rows = [list(c) for c in itertools.product(values, repeat=4)]
    got = O.target_argmax(np.array(rows))
    for row, g in zip(rows, got):
        assert g == _greedy_by_definition(row), row


def test_greedy_pick_signed_zero_tie():
    # -0.0 and +0.0 are the same number: the lower index wins either way round
    assert O.target_argmax(np.array([[-1.0, -0.0, 0.0]]))[0] == 1
    assert O.target_argmax(np.array([[-1.0, 0.0, -0.0]]))[0] == 1


def _one_hot_logits(targets, V):
    lg = np.zeros((len(targets), V))
    lg[np.arange(len(targets)), targets] = 1.0
    return lg


@pytest.mark.parametrize("V", [2, 3])
def test_acceptance_enumerated(V):
    """Every token sequence and every target sequence of 1..4 rows over a tiny
    vocabulary, laid out as one ragged batch."""
    cases = []
    for n in range(1, 5):
        for toks in itertools.product(range(V), repeat=n):
            for tgts in itertools.product(range(V), repeat=n):
                cases.append((toks, tgts))
    n_rows = [len(t) for t, _ in cases]
    qsl = np.concatenate([[0], np.cumsum(n_rows)]).astype(np.int32)
    tok = np.array([x for t, _ in cases for x in t], np.int32)
    tgt = np.array([x for _, t in cases for x in t], np.int32)
    target, accepted, bonus = O.verify_greedy(qsl, tok, _one_hot_logits(tgt, V))
    assert np.array_equal(target, tgt)
    for r, (toks, tgts) in enumerate(cases):
        n, a = len(toks), int(accepted[r])
        assert 0 <= a <= n - 1
        # every accepted draft equals the target's pick of the row before it
        assert all(toks[j] == tgts[j - 1] for j in range(1, a + 1))
        # the prefix is the longest one: the next draft, if any, disagrees
        if a + 1 < n:
            assert toks[a + 1] != tgts[a]
        # the bonus token is the target's pick right after the accepted prefix
        assert bonus[r] == tgts[a]


def test_single_row_is_plain_decoding():
    """A request with no drafts reduces to ordinary greedy next-token decoding."""
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((6, 50))
    qsl = np.arange(7, dtype=np.int32)
    tok = rng.integers(0, 50, 6).astype(np.int32)
    target, accepted, bonus = O.verify_greedy(qsl, tok, lg)
    assert np.all(accepted == 0)
    assert np.array_equal(bonus, [_greedy_by_definition(list(r)) for r in lg])


def test_all_drafts_accepted_and_first_rejected():
    V = 20
    tgt = np.array([4, 9, 9, 1, 0], np.int32)
    lg = _one_hot_logits(tgt, V)
    qsl = np.array([0, 5], np.int32)
    # drafts copy the target's picks: all four accepted, bonus = pick of the last row
    tok = np.array([7, 4, 9, 9, 1], np.int32)
    _, a, b = O.verify_greedy(qsl, tok, lg)
    assert a[0] == 4 and b[0] == 0
    # the first draft differs: nothing accepted, bonus = pick of row 0
    tok = np.array([7, 5, 9, 9, 1], np.int32)
    _, a, b = O.verify_greedy(qsl, tok, lg)
    assert a[0] == 0 and b[0] == 4


def test_empty_request():
    lg = _one_hot_logits(np.array([2, 3], np.int32), 5)
    target, a, b = O.verify_greedy(np.array([0, 0, 2, 2], np.int32), np.array([1, 2], np.int32), lg)
    assert list(a) == [0, 1, 0] and list(b) == [-1, 3, -1]


@pytest.mark.parametrize("name", ["verify_small", "verify_small_bf16"])
def test_planted_batch_recovered(name):
    """The generator plants each row's greatest logit and each request's accepted
    count; the oracle must find exactly those."""
    wl = W.get_verify(name)
    b = W.make_verify_batch(wl)
    lg = O.decode(b["logits"], wl.dtype)
    target, accepted, bonus = O.verify_greedy(b["qsl"], b["tok"], lg)
    assert np.array_equal(target, b["planted_target"])
    assert np.array_equal(accepted, b["planted_accepted"])
    q0 = b["qsl"][:-1]
    assert np.array_equal(bonus, b["planted_target"][q0 + accepted])


def test_hand_off_to_next_step_metadata():
    """The accepted counts and bonus tokens are valid inputs of the next draft
    step: its NTP row carries the bonus token and the rejected rows are the
    drafts past the accepted prefix."""
    wl = W.get_verify("verify_small")
    b = W.make_verify_batch(wl)
    target, accepted, bonus = O.verify_greedy(b["qsl"], b["tok"], O.decode(b["logits"], "f32"))
    qsl = b["qsl"]
    n = np.diff(qsl)
    K, bs = 4, 4
    ctx = np.array([10, 0, 5, 33, 7])
    prev_pos = np.concatenate([c + np.arange(k) for c, k in zip(ctx, n)]).astype(np.int64)
    nblk = [(c + k + K - 1 + bs - 1) // bs for c, k in zip(ctx, n)]
    table = np.full((len(n), max(nblk)), -1, np.int32)
    o = 0
    for r in range(len(n)):
        table[r, :nblk[r]] = np.arange(o, o + nblk[r])
        o += nblk[r]
    m = O.prepare_metadata(qsl, b["tok"], prev_pos, accepted, bonus, table, K, 0, bs)
    oq = m["out_qsl"]
    for r in range(len(n)):
        assert m["tok"][oq[r] + accepted[r]] == bonus[r]
        assert m["is_rejected"][oq[r]:oq[r] + n[r]].sum() == n[r] - 1 - accepted[r]
