"""GPU parity of the COD index lists and the asymmetric mask against the oracle.

"[RFC]: Add random anchor for p-eagle first position": COD sampling, the
max_anchors cap and the asymmetric mask.  Integer work: every list, count and
mask byte must match bit for bit; bytes outside each sequence's written region
must keep their sentinel.
"""

import dataclasses

import numpy as np
import pytest

from oracle import pe_cod as C
from parity import built, cuda_or_skip
from speculative_drafting_gb300 import binding, runner, workloads as W

pytestmark = pytest.mark.gpu

SENTINEL = 0xAB


def _oracle(b):
    return C.cod_batch(b["seq_len"], b["loss_mask"], b["n_depth"], b["retain"], b["max_anchors"],
                       b["u_anchor"], b["u_keep"])


def _run(b, q_cap=None, ld=None, guard=64):
    torch = cuda_or_skip()
    built()
    r = runner.CodRunner(b, q_cap=q_cap, ld=ld, guard=guard)
    r.mask.fill_(SENTINEL)
    r.run()
    torch.cuda.synchronize()
    return r


def _check(b, r, levels, full_mask=True):
    idx, counts = r.idx.cpu().numpy(), r.counts.cpu().numpy()
    for s, lv in enumerate(levels):
        L = int(np.clip(b["seq_len"][s], 0, b["S_max"]))
        np.testing.assert_array_equal(counts[s], [len(x) for x in lv], err_msg=f"counts {s}")
        for k, x in enumerate(lv):
            np.testing.assert_array_equal(idx[s, k, :len(x)], x, err_msg=f"list {s}/{k}")
        if not full_mask:
            continue
        Q, KV = C.cod_sizes(lv, L)
        width = (KV + 15) // 16 * 16
        got = r.mask_of(s).cpu().numpy()
        want = np.zeros((Q, width), np.uint8)
        want[:, :KV] = C.cod_mask(lv, L)
        np.testing.assert_array_equal(got[:Q, :width], want, err_msg=f"mask {s}")
        assert (got[:Q, width:] == SENTINEL).all(), f"bytes past row {s}"
        assert (got[Q:] == SENTINEL).all(), f"rows past Q {s}"
    assert (r.mask[r.B * r.mask_stride:].cpu().numpy() == SENTINEL).all()


@pytest.mark.parametrize("name", ["cod_tiny", "cod_small", "cod_s4096_nocap", "cod_s8192_a1024"])
def test_cod_matches_oracle(name):
    b = W.make_cod_batch(W.get_cod(name))
    r = _run(b)
    assert r.status()[0] == 0
    _check(b, r, _oracle(b))


VARIANTS = [
    {"retain": 1.0, "max_anchors": 0},            # every chain runs to the sequence end
    {"retain": 0.0},                              # depth 0 only
    {"n_depth": 1},                               # no u_keep at all
    {"n_depth": 16, "retain": 0.9},               # the most depths
    {"max_anchors": 1},                           # one anchor per sequence
    {"max_anchors": 100000},                      # a cap that never binds
    {"seed": 7, "prompt_span": (1, 3), "response_span": (1, 3)},  # fragmented loss mask
]


@pytest.mark.parametrize("over", VARIANTS)
def test_cod_variants(over):
    b = W.make_cod_batch(W.get_cod("cod_small", **over))
    r = _run(b)
    assert r.status()[0] == 0
    _check(b, r, _oracle(b))


def test_cod_equal_draws_break_ties_by_position():
    # draws quantised to 1/8: many candidates share the threshold key
    b = W.make_cod_batch(W.get_cod("cod_small", seed=3))
    b["u_anchor"] = (np.floor(b["u_anchor"] * 8) / 8).astype(np.float32)
    r = _run(b)
    assert r.status()[0] == 0
    _check(b, r, _oracle(b))


def test_cod_all_loss_long_sequence():
    # one 30000-token sequence with a loss at every position: the select runs
    # over 30000 keys and the lists over 30 chunks of 1024 positions
    wl = W.get_cod("cod_tiny", batch=1, seq_len=30000, s_max=30000, n_depth=6, retain=0.6,
                   max_anchors=4097, prompt_span=(1, 1), response_span=(40000, 40000))
    b = W.make_cod_batch(wl)
    b["loss_mask"][:] = 1
    r = _run(b, q_cap=11000)  # about 4097 x 2.38 rows expected
    assert r.status()[0] == 0
    _check(b, r, _oracle(b))


def test_cod_capacity_is_reported_and_respected():
    b = W.make_cod_batch(W.get_cod("cod_small"))
    levels = _oracle(b)
    sizes = [C.cod_sizes(lv, int(L)) for lv, L in zip(levels, b["seq_len"])]
    q_small = max(q for q, _ in sizes) // 2
    r = _run(b, q_cap=q_small)
    assert r.status()[0] & binding.PE_ST_CAPACITY
    # the rows that fit are right; nothing is written past the block
    for s, (lv, (Q, KV)) in enumerate(zip(levels, sizes)):
        L = int(b["seq_len"][s])
        width = (KV + 15) // 16 * 16
        n = min(Q, q_small)
        got = r.mask_of(s).cpu().numpy()
        want = np.zeros((Q, width), np.uint8)
        want[:, :KV] = C.cod_mask(lv, L)
        np.testing.assert_array_equal(got[:n, :width], want[:n])
    assert (r.mask[r.B * r.mask_stride:].cpu().numpy() == SENTINEL).all()


def test_cod_seq_len_out_of_range_is_clamped():
    b = W.make_cod_batch(W.get_cod("cod_tiny"))
    b["seq_len"] = b["seq_len"].copy()
    b["seq_len"][1] = b["S_max"] + 5
    b["seq_len"][2] = -3
    r = _run(b)
    assert r.status()[0] & binding.PE_ST_CAPACITY
    clamped = dict(b, seq_len=np.clip(b["seq_len"], 0, b["S_max"]).astype(np.int32))
    _check(clamped, r, _oracle(clamped))


def test_cod_graph_replay():
    torch = cuda_or_skip()
    built()
    b = W.make_cod_batch(W.get_cod("cod_small"))
    r = runner.CodRunner(b)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        r.run(stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        r.run(stream=s)
    r.mask.fill_(SENTINEL)
    r.idx.fill_(-1)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    s.synchronize()
    assert r.status()[0] == 0
    _check(b, r, _oracle(b))


def test_cod_empty_batch():
    cuda_or_skip()
    b = W.make_cod_batch(dataclasses.replace(W.get_cod("cod_tiny"), batch=2, seq_len=(0, 0)))
    r = _run(b)
    assert r.status()[0] == 0
    _check(b, r, _oracle(b))
