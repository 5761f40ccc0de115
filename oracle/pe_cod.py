"""CPU oracle of the COD sample indices and the asymmetric attention mask.
TEST INFRASTRUCTURE ONLY: the tests, the package's smoke check and the
benchmark's CPU leg import it; the library never does, and it shares no code
with the CUDA sources.

Source: "[RFC]: Add random anchor for p-eagle first position".
  * Motivation: COD sampling predicts the next token from every starting
    position of a sample, then the token after that for a share of those
    positions (70 % in the example), the third token for that share of the
    share, and so on; with 4 speculative tokens the queries number
    sequence length x sum_{n=0..4} 0.7^n.
  * Proposed change: max_anchors caps the chain starting points; when set, a
    random max_anchors of the loss_mask = 1 positions are the depth-0 set.  The
    mask is asymmetric: its queries are the COD-sampled tokens, its keys and
    values the whole original sequence plus the deeper (depth >= 1) COD tokens.
  * Reply (orestis-z), "Depth > 0 attention": deeper queries see the original
    sequence, not only their own chain.
  * Ablation sections: the retained share is called the drop rate there (at a
    rate of 0.15 only 15 % of positions reach depth 1).

Readings where the page is silent (each is listed in the design notes):
  * Per sequence b of length L_b the candidates are the positions i < L_b with
    loss_mask[i] != 0.  With max_anchors A > 0 and more than A candidates, the
    anchors are the A candidates with the smallest random key (u_anchor[i], i):
    a uniform draw of A of them without replacement.  Otherwise every
    candidate is an anchor.
  * Depth k >= 1 keeps the anchors of depth k-1 whose own draw u_keep[k-1][a]
    is below the retained share rho, and whose position a + k lies inside the
    sequence (a + k < L_b): each chain continues independently (Bernoulli).
  * The chain at anchor a predicts token a + k + 1 at depth k; its depth-k
    query stands at position a + k.
  * Query rows: depth-major (all depth-0 anchors, then depth 1, ...), anchors
    ascending inside a depth.  Key columns: the L_b original positions, then
    the depth >= 1 tokens in the same depth-major order.
  * A query (a, k) sees original position j iff j <= a (the context up to its
    anchor; the tokens after a are what the chain predicts), and chain token
    (a', k') iff a' == a and k' <= k (its own chain's earlier depths and
    itself).  This is the visibility a MASK row of the parallel-draft step has
    at inference: the context, then its request's earlier draft positions.

The random draws are inputs (u_anchor[L], u_keep[D-1][L], float32 in [0, 1)),
so the oracle and the kernels decide on the same numbers; the comparisons
u_keep < rho are taken in float32 on both sides.
"""

from __future__ import annotations

import numpy as np


def cod_sample_indices(loss_mask, n_depth, retain, max_anchors, u_anchor, u_keep):
    """COD index lists of one sequence (length len(loss_mask)).

    Returns a list of n_depth int64 arrays: I_k = anchor positions whose chain
    reaches depth k, ascending.  ("[RFC]: Add random anchor for p-eagle first
    position", Motivation and Proposed change.)"""
    L = len(loss_mask)
    cand = np.nonzero(np.asarray(loss_mask[:L]) != 0)[0]
    if max_anchors > 0 and len(cand) > max_anchors:
        keys = np.asarray(u_anchor, dtype=np.float32)[cand]
        order = np.lexsort((cand, keys))  # by u, then by position
        anchors = np.sort(cand[order[:max_anchors]])
    else:
        anchors = cand
    rho = np.float32(retain)
    levels = [anchors.astype(np.int64)]
    for k in range(1, n_depth):
        prev = levels[-1]
        draws = np.asarray(u_keep[k - 1], dtype=np.float32)[prev] if len(prev) else np.zeros(0, np.float32)
        keep = (draws < rho) & (prev + k < L)
        levels.append(prev[keep])
    return levels


def cod_sizes(levels, L):
    """(Q, KV): query rows and key columns of the asymmetric mask.
    Q = sum_k |I_k|; KV = L + sum_{k>=1} |I_k|."""
    q = int(sum(len(x) for x in levels))
    return q, int(L + q - len(levels[0]))


def cod_rows(levels):
    """(anchor, depth) of each query row, depth-major."""
    if not levels:  # one depth only: no deeper tokens
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    a = np.concatenate(levels)
    k = np.concatenate([np.full(len(x), d, np.int64) for d, x in enumerate(levels)])
    return a.astype(np.int64), k


def cod_mask(levels, L):
    """Dense boolean mask [Q][KV] of one sequence: True where the query may
    attend the key ("[RFC]: Add random anchor for p-eagle first position",
    Proposed change and the reply's "Depth > 0 attention")."""
    qa, qk = cod_rows(levels)
    ca, ck = cod_rows(levels[1:])
    ck = ck + 1
    Q, KV = cod_sizes(levels, L)
    m = np.zeros((Q, KV), dtype=bool)
    for q in range(Q):
        a, k = qa[q], qk[q]
        m[q, :a + 1] = True                      # original positions 0..a
        m[q, L:] = (ca == a) & (ck <= k)         # own chain, depths 1..k
    return m


def cod_batch(seq_len, loss_mask, n_depth, retain, max_anchors, u_anchor, u_keep):
    """Per sequence of a batch: the index lists.  loss_mask[B][S_max],
    u_anchor[B][S_max], u_keep[B][D-1][S_max]; positions >= seq_len[b] are not
    part of sequence b."""
    out = []
    for b, L in enumerate(np.asarray(seq_len)):
        L = int(L)
        out.append(cod_sample_indices(loss_mask[b, :L], n_depth, retain, max_anchors,
                                      u_anchor[b, :L], u_keep[b, :, :L] if n_depth > 1 else []))
    return out
