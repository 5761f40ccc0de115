"""Pins of the COD index / mask oracle against what the page and arithmetic fix.

"[RFC]: Add random anchor for p-eagle first position": COD sampling (every
loss position starts a chain; each depth keeps a share of the previous one),
max_anchors (a uniform random subset of the loss positions at depth 0) and the
asymmetric mask (queries = the COD tokens, keys = the original sequence plus
the deeper COD tokens).
"""

import math
import os

import numpy as np
import pytest

from oracle import pe_cod as C
from speculative_drafting_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _draws(rng, L, D):
    return (rng.random(L, dtype=np.float32), rng.random((max(D - 1, 0), L), dtype=np.float32))


def test_full_retain_no_cap_is_every_position_in_range():
    # retain 1: u < 1 always holds, so depth k holds every loss position a with a + k < L
    rng = np.random.default_rng(1)
    L, D = 41, 6
    lm = (rng.random(L) < 0.6).astype(np.uint8)
    ua, uk = _draws(rng, L, D)
    lv = C.cod_sample_indices(lm, D, 1.0, 0, ua, uk)
    cand = [i for i in range(L) if lm[i]]
    for k in range(D):
        assert lv[k].tolist() == [a for a in cand if a + k < L]


def test_zero_retain_keeps_depth_zero_only():
    rng = np.random.default_rng(2)
    L, D = 30, 5
    lm = np.ones(L, np.uint8)
    ua, uk = _draws(rng, L, D)
    lv = C.cod_sample_indices(lm, D, 0.0, 0, ua, uk)
    assert lv[0].tolist() == list(range(L))
    assert all(len(x) == 0 for x in lv[1:])


def test_cap_at_or_above_candidates_keeps_all_and_one_below_drops_largest_draw():
    rng = np.random.default_rng(3)
    L, D = 50, 3
    lm = (rng.random(L) < 0.5).astype(np.uint8)
    ua, uk = _draws(rng, L, D)
    cand = np.nonzero(lm)[0]
    n = len(cand)
    for cap in (0, n, n + 5):
        assert C.cod_sample_indices(lm, D, 0.5, cap, ua, uk)[0].tolist() == cand.tolist()
    dropped = cand[np.argmax(ua[cand])]
    got = C.cod_sample_indices(lm, D, 0.5, n - 1, ua, uk)[0].tolist()
    assert got == [a for a in cand.tolist() if a != dropped]


def test_selected_anchors_precede_the_rest_in_draw_order():
    # the chosen A have smaller (u, position) keys than every candidate left out
    for seed in range(30):
        rng = np.random.default_rng(100 + seed)
        L = int(rng.integers(1, 200))
        lm = (rng.random(L) < 0.7).astype(np.uint8)
        ua = rng.random(L, dtype=np.float32)
        # repeated draws, so the position order decides some ties
        ua = np.round(ua * 16).astype(np.float32) / 16
        A = int(rng.integers(1, 40))
        got = set(C.cod_sample_indices(lm, 1, 0.5, A, ua, [])[0].tolist())
        cand = [i for i in range(L) if lm[i]]
        assert len(got) == min(A, len(cand))
        out = [i for i in cand if i not in got]
        if got and out:
            assert max((ua[i], i) for i in got) < min((ua[i], i) for i in out)


def test_anchor_subset_is_uniform():
    # every candidate is chosen with probability A / n
    n, A, trials = 10, 3, 6000
    lm = np.ones(n, np.uint8)
    rng = np.random.default_rng(4)
    hits = np.zeros(n)
    for _ in range(trials):
        hits[C.cod_sample_indices(lm, 1, 0.5, A, rng.random(n, dtype=np.float32), [])[0]] += 1
    p = A / n
    sd = math.sqrt(trials * p * (1 - p))
    assert np.all(np.abs(hits - trials * p) < 5 * sd)


def test_depth_major_lists_match_a_chain_by_chain_walk():
    # the same chains walked one anchor at a time, depth by depth
    for seed in range(20):
        rng = np.random.default_rng(200 + seed)
        L, D = int(rng.integers(0, 90)), int(rng.integers(1, 7))
        lm = (rng.random(L) < 0.6).astype(np.uint8)
        ua, uk = _draws(rng, L, D)
        rho = float(rng.choice([0.0, 0.3, 0.7, 1.0]))
        A = int(rng.integers(0, 12))
        lv = C.cod_sample_indices(lm, D, rho, A, ua, uk)
        want = [[] for _ in range(D)]
        for a in lv[0].tolist():
            depth = 0
            want[0].append(a)
            while depth + 1 < D and a + depth + 1 < L and uk[depth][a] < np.float32(rho):
                depth += 1
                want[depth].append(a)
        assert [x.tolist() for x in lv] == want


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = float(v)
    return vals


def test_mask_size_factors_of_the_page():
    """With retain 0.7 and 4 speculative tokens (depths 0..4) the page sizes the
    queries at anchors x 2.73 and the deeper keys at anchors x 1.73, from
    sum_{n=0..4} 0.7^n.  Far from the sequence end the expected number of depth-k
    tokens is A * rho^k, so Q / A tends to that sum and (KV - L) / A to the sum
    less one."""
    g = _golden("cod_rfc_mask_factors.txt")
    rho, D = g["retain"], int(g["n_depth"])
    s = sum(rho ** n for n in range(D))
    # the printed factors agree with the sum to the two digits the page keeps
    assert abs(s - g["query_factor"]) < 0.05 and abs((s - 1) - g["key_factor"]) < 0.05
    rng = np.random.default_rng(5)
    L, A = 400_000, 200_000
    lm = np.ones(L, np.uint8)
    ua, uk = _draws(rng, L, D)
    lv = C.cod_sample_indices(lm, D, rho, A, ua, uk)
    Q, KV = C.cod_sizes(lv, L)
    assert len(lv[0]) == A
    assert abs(Q / A - s) < 0.012
    assert abs((KV - L) / A - (s - 1)) < 0.012
    for k in range(1, D):   # each depth keeps rho of the one before it
        n0, n1 = len(lv[k - 1]), len(lv[k])
        assert abs(n1 - rho * n0) < 5 * math.sqrt(n0 * rho * (1 - rho))


def _levels(seed, L, D, rho, A):
    rng = np.random.default_rng(seed)
    lm = (rng.random(L) < 0.6).astype(np.uint8)
    ua, uk = _draws(rng, L, D)
    return C.cod_sample_indices(lm, D, rho, A, ua, uk)


@pytest.mark.parametrize("seed", range(6))
def test_mask_row_and_column_sums(seed):
    L, D = 70, 5
    lv = _levels(300 + seed, L, D, 0.7, 16)
    m = C.cod_mask(lv, L)
    Q, KV = C.cod_sizes(lv, L)
    assert m.shape == (Q, KV)
    qa, qk = C.cod_rows(lv)
    # a query at anchor a, depth k sees positions 0..a and its own depths 1..k
    np.testing.assert_array_equal(m.sum(1), qa + 1 + qk)
    # original column j: every query whose anchor is at or after j
    np.testing.assert_array_equal(m[:, :L].sum(0), [(qa >= j).sum() for j in range(L)])
    # chain column (a', k'): the queries of chain a' at depth k' or deeper
    ca, ck = C.cod_rows(lv[1:])
    depth_of = {a: max(k for k in range(D) if a in set(lv[k].tolist())) for a in lv[0].tolist()}
    np.testing.assert_array_equal(m[:, L:].sum(0), [depth_of[a] - k for a, k in zip(ca, ck)])


@pytest.mark.parametrize("seed", range(6))
def test_mask_is_the_draft_steps_visibility(seed):
    """Each chain is a request at inference: context positions 0..a, then draft
    positions a+1..a+k.  A row sees a key iff the key belongs to its request and
    stands at or before the row's position (the draft step's causal rule)."""
    L, D = 60, 6
    lv = _levels(400 + seed, L, D, 0.6, 12)
    m = C.cod_mask(lv, L)
    qa, qk = C.cod_rows(lv)
    keys = [("ctx", j, j) for j in range(L)]
    ca, ck = C.cod_rows(lv[1:])
    keys += [("draft", a, a + k + 1) for a, k in zip(ca, ck)]
    for q in range(len(qa)):
        req, pos = qa[q], qa[q] + qk[q]
        for c, (kind, owner, kpos) in enumerate(keys):
            mine = (owner <= req) if kind == "ctx" else (owner == req)
            assert m[q, c] == (mine and kpos <= pos), (q, c)


def test_edges_empty_and_one_token():
    for L in (0, 1):
        lm = np.ones(L, np.uint8)
        lv = C.cod_sample_indices(lm, 4, 0.9, 3, np.zeros(L, np.float32), np.zeros((3, L), np.float32))
        assert [len(x) for x in lv] == [L, 0, 0, 0]
        assert C.cod_sizes(lv, L) == (L, L)
        assert C.cod_mask(lv, L).sum() == L


def test_workload_batches_are_seeded_and_shaped():
    for name in W.COD_WORKLOADS:
        wl = W.get_cod(name)
        b = W.make_cod_batch(wl)
        b2 = W.make_cod_batch(wl)
        assert b["loss_mask"].shape == (wl.batch, wl.s_max)
        assert b["u_keep"].shape == (wl.batch, wl.n_depth - 1, wl.s_max)
        assert np.array_equal(b["loss_mask"], b2["loss_mask"]) and np.array_equal(b["u_keep"], b2["u_keep"])
        for r, L in enumerate(b["seq_len"]):
            assert not b["loss_mask"][r, L:].any()
        assert (b["u_anchor"] >= 0).all() and (b["u_anchor"] < 1).all()


def test_one_depth_mask_is_causal_over_the_anchors():
    # D = 1: no deeper tokens, so the keys are the sequence and row a sees 0..a
    lm = np.array([0, 1, 1, 0, 1], np.uint8)
    lv = C.cod_sample_indices(lm, 1, 0.5, 0, np.zeros(5, np.float32), [])
    m = C.cod_mask(lv, 5)
    assert m.shape == (3, 5)
    np.testing.assert_array_equal(m, [[1, 1, 0, 0, 0], [1, 1, 1, 0, 0], [1, 1, 1, 1, 1]])


def test_capacity_bound_holds_for_every_mask():
    # the library's sizing helper: q_cap and ld hold any mask of the batch
    from speculative_drafting_gb300 import runner

    for name in W.COD_WORKLOADS:
        for over in ({}, {"retain": 1.0}, {"max_anchors": 0, "retain": 1.0}):
            wl = W.get_cod(name, **over)
            if wl.s_max > 4096 and over:
                continue
            b = W.make_cod_batch(wl)
            q_cap, ld = runner.cod_capacity(b["S_max"], b["n_depth"], b["max_anchors"])
            assert ld % 16 == 0
            for lv, L in zip(C.cod_batch(b["seq_len"], b["loss_mask"], b["n_depth"], b["retain"],
                                         b["max_anchors"], b["u_anchor"], b["u_keep"]), b["seq_len"]):
                Q, KV = C.cod_sizes(lv, int(L))
                assert Q <= q_cap and (KV + 15) // 16 * 16 <= ld


# ---- planted mistakes: each one, put into the oracle, fails a pin above

_orig_mask = C.cod_mask


def _mask_context_before_anchor(levels, L):
    m = _orig_mask(levels, L)
    qa, _ = C.cod_rows(levels)
    m[np.arange(len(qa)), qa] = False           # the row no longer sees its own anchor
    return m


def _mask_chain_strictly_earlier(levels, L):
    qa, qk = C.cod_rows(levels)
    ca, ck = C.cod_rows(levels[1:])
    m = _orig_mask(levels, L)
    for q in range(len(qa)):
        m[q, L:] = (ca == qa[q]) & (ck + 1 < qk[q])  # drops the row's own token
    return m


_orig_sample = C.cod_sample_indices


def _sample_bound_off_by_one(loss_mask, n_depth, retain, max_anchors, u_anchor, u_keep):
    lv = _orig_sample(loss_mask, n_depth, 1.0, 0, u_anchor, u_keep)
    return lv if retain != 1.0 or max_anchors else [
        np.array([a for a in np.nonzero(np.asarray(loss_mask))[0] if a + k <= len(loss_mask)])
        for k in range(n_depth)]


def _sample_ties_to_higher_position(loss_mask, n_depth, retain, max_anchors, u_anchor, u_keep):
    L = len(loss_mask)
    cand = np.nonzero(np.asarray(loss_mask) != 0)[0]
    if max_anchors > 0 and len(cand) > max_anchors:
        order = np.lexsort((-cand, np.asarray(u_anchor, np.float32)[cand]))
        cand = np.sort(cand[order[:max_anchors]])
    return [cand.astype(np.int64)] + _orig_sample(np.isin(np.arange(L), cand), n_depth, retain, 0,
                                                  u_anchor, u_keep)[1:]


@pytest.mark.parametrize("mutant,pin", [
    (_mask_context_before_anchor, lambda: test_mask_row_and_column_sums(0)),
    (_mask_chain_strictly_earlier, lambda: test_mask_row_and_column_sums(0)),
    (_mask_context_before_anchor, lambda: test_mask_is_the_draft_steps_visibility(0)),
    (_mask_chain_strictly_earlier, lambda: test_mask_is_the_draft_steps_visibility(0)),
])
def test_pins_catch_planted_mask_mistakes(monkeypatch, mutant, pin):
    monkeypatch.setattr(C, "cod_mask", mutant)
    with pytest.raises(AssertionError):
        pin()


@pytest.mark.parametrize("mutant,pin", [
    (_sample_bound_off_by_one, test_full_retain_no_cap_is_every_position_in_range),
    (_sample_ties_to_higher_position, test_selected_anchors_precede_the_rest_in_draw_order),
])
def test_pins_catch_planted_sampling_mistakes(monkeypatch, mutant, pin):
    monkeypatch.setattr(C, "cod_sample_indices", mutant)
    with pytest.raises(AssertionError):
        pin()
