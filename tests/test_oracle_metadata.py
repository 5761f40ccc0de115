"""Brute-force pins of the oracle's batch metadata (CPU only).

Every accepted-count vector of small batches is enumerated and the oracle's
output is checked against predicates written from the pages' rules, not from
the oracle's own construction: the input pairing shifted by one and the NTP
row ("P-EAGLE: parallel speculative decoding in vLLM", Parallel drafting), the
MASK slots and the rejected / masked masks (Fused Triton kernel), and rejected
tokens mapped to PADDING_SLOT_ID = -1 (KV cache and CUDA graphs).
"""

import itertools

import numpy as np
import pytest

from oracle import pe_oracle as O

BS = 4
MASK = 0


def _batch(n_prev, ctx, accepted, K, rng):
    B = len(n_prev)
    qsl = np.concatenate([[0], np.cumsum(n_prev)]).astype(np.int32)
    T_in = int(qsl[-1])
    prev_tok = rng.integers(1, 1000, size=T_in).astype(np.int32)
    bonus = rng.integers(1, 1000, size=B).astype(np.int32)
    prev_pos = np.concatenate([c + np.arange(n) for c, n in zip(ctx, n_prev)]).astype(np.int64)
    nblk = [(c + n + K - 1 + BS - 1) // BS for c, n in zip(ctx, n_prev)]
    ids = rng.permutation(sum(nblk))
    table = np.full((B, max(nblk)), -1, np.int32)
    o = 0
    for r in range(B):
        table[r, :nblk[r]] = ids[o:o + nblk[r]]
        o += nblk[r]
    return qsl, prev_tok, prev_pos, np.array(accepted, np.int32), bonus, table


def _check(qsl, prev_tok, prev_pos, accepted, bonus, table, K):
    m = O.prepare_metadata(qsl, prev_tok, prev_pos, accepted, bonus, table, K, MASK, BS)
    B = len(accepted)
    n = np.diff(qsl)
    ctx = prev_pos[qsl[:-1]]
    T_out = m["T_out"]
    assert T_out == qsl[-1] + B * (K - 1)
    assert np.array_equal(np.diff(m["out_qsl"]), n + K - 1)
    # masked rows: exactly K-1 per request, MASK token, no hidden source, never rejected
    masked = m["is_masked"].astype(bool)
    rejected = m["is_rejected"].astype(bool)
    assert masked.sum() == B * (K - 1)
    assert np.all(m["tok"][masked] == MASK) and np.all(m["hidden_src"][masked] == -1)
    assert not np.any(masked & rejected)
    # rejected rows: one per draft past the accepted prefix; they write nothing
    assert rejected.sum() == int(np.sum(n - 1 - accepted))
    assert np.all(m["slot"][rejected] == -1)
    assert np.all(m["slot"][~rejected] >= 0)
    # slots: distinct across the whole batch
    live = m["slot"][~rejected]
    assert len(np.unique(live)) == len(live)
    valid_expected = []
    for r in range(B):
        rows = np.arange(m["out_qsl"][r], m["out_qsl"][r + 1])
        live_rows = [o for o in rows if not rejected[o]]
        valid_expected += live_rows
        c, a = int(ctx[r]), int(accepted[r])
        # the live positions are exactly c .. c+a+K-1, each once
        assert sorted(m["pos"][live_rows].tolist()) == list(range(c, c + a + K))
        for o in live_rows:
            p = int(m["pos"][o])
            blk = int(m["slot"][o]) // BS
            # the slot is in one of r's own blocks, at the position's offset, and the
            # block is the table entry for that position's block index
            assert blk in table[r] and int(m["slot"][o]) % BS == p % BS
            assert list(table[r]).index(blk) == p // BS
        # the NTP row: live, not masked, at position c+a, carries the bonus token
        ntp = [o for o in live_rows if not masked[o] and m["pos"][o] == c + a]
        assert len(ntp) == 1 and m["tok"][ntp[0]] == bonus[r]
        assert m["hidden_src"][ntp[0]] == qsl[r] + a
        # the other copied rows: hidden state of their own position, token of the next one
        for o in rows:
            if masked[o] or o == ntp[0]:
                continue
            j = int(m["pos"][o]) - c
            assert m["hidden_src"][o] == qsl[r] + j
            if j + 1 < n[r]:
                assert m["tok"][o] == prev_tok[qsl[r] + j + 1]
        # sample rows: NTP row then the MASK rows, positions c+a .. c+a+K-1
        s = m["sample_idx"][r * K:(r + 1) * K]
        assert s[0] == ntp[0] and all(masked[s[1:]])
        assert list(m["pos"][s]) == list(range(c + a, c + a + K))
        assert m["seq_len"][r] == c + a + K
    assert m["n_valid"] == int(np.sum(accepted + K)) == len(valid_expected)
    assert list(m["valid_rows"][:m["n_valid"]]) == sorted(valid_expected)
    assert np.all(m["valid_rows"][m["n_valid"]:] == -1)
    assert np.array_equal(np.diff(m["valid_qsl"]), accepted + K)
    return m


@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_metadata_all_accept_vectors_two_requests(K):
    rng = np.random.default_rng(K)
    ctxs = [0, 1, BS - 1, BS, BS + 1]
    count = 0
    for n0, n1 in itertools.product(range(1, K + 3), repeat=2):
        for a0, a1 in itertools.product(range(n0), range(n1)):
            c0, c1 = ctxs[(a0 + n1) % 5], ctxs[(a1 + 2 * n0) % 5]
            _check(*_batch([n0, n1], [c0, c1], [a0, a1], K, rng), K)
            count += 1
    assert count > 0


def test_metadata_every_context_and_accept_single_request():
    rng = np.random.default_rng(11)
    for K in (1, 2, 4):
        for n in range(1, K + 3):
            for a in range(n):
                for c in (0, 1, BS - 1, BS, BS + 1, 3 * BS + 2):
                    _check(*_batch([n], [c], [a], K, rng), K)


def test_metadata_three_requests_random_sample():
    rng = np.random.default_rng(12)
    for _ in range(1500):
        K = int(rng.integers(1, 5))
        n = [int(rng.integers(1, K + 3)) for _ in range(3)]
        a = [int(rng.integers(0, x)) for x in n]
        c = [int(rng.choice([0, 1, BS - 1, BS, BS + 1, 37])) for _ in range(3)]
        _check(*_batch(n, c, a, K, rng), K)


def test_k1_is_plain_shifted_eagle_batch():
    # K = 1: no MASK rows; the drafter batch is the verify batch with tokens
    # shifted by one, the bonus token at the accepted row, and nothing appended.
    rng = np.random.default_rng(13)
    qsl, tok, pos, acc, bonus, table = _batch([5, 3], [9, 2], [2, 2], 1, rng)
    m = _check(qsl, tok, pos, acc, bonus, table, 1)
    assert m["T_out"] == qsl[-1] and not m["is_masked"].any()
    assert list(m["tok"][:5]) == [tok[1], tok[2], bonus[0], tok[4], bonus[0]]
    assert list(m["slot"][:5] >= 0) == [True, True, True, False, False]
