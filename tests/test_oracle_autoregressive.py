"""Pins of the oracle's autoregressive K-pass drafting (CPU only).

"P-EAGLE: parallel speculative decoding in vLLM", Solving the autoregressive
drafting bottleneck: an EAGLE-style drafter makes K draft tokens with K
sequential forward passes.  "Attention Drift", sections 3 and 4.1: after the
first step it consumes its own hidden state.

* An independently written drafter below (one row at a time, dict caches,
  complex-rotation RoPE, scipy softmax and expit) run as a K-pass loop gives the
  oracle's logits, pre- and post-norm, with random gains (so that feeding back
  y or the normalised output are told apart).
* The first pass is the parallel step's NTP row: same first draft, z and logits.
* K = 1 is the parallel step with K = 1.
* In bf16 mode the stored tensors are bf16 values and the logits track the
  unrounded definition within the step's tolerance.
* Mistakes planted in the oracle (the wrong hidden state fed back, a position
  off by one, the previous pass's KV not kept) each fail the first pin.
"""

import dataclasses

import numpy as np
import pytest
import scipy.special

from oracle import pe_oracle as O
from speculative_drafting_gb300 import workloads as W


def _setup(name, random_gains=False, **over):
    wl = W.get(name, **over)
    b = W.make_batch(wl)
    w = W.make_weights(wl)
    if random_gains:
        assert wl.dims.dtype == "f32"
        g = np.random.default_rng(77)
        for key in ("gamma_stream", "gamma_in", "gamma_post", "gamma_final"):
            if key in w:
                w[key] = (0.5 + g.random(w[key].shape)).astype(np.float32)
    kc, vc = W.make_kv_cache(wl, b["num_blocks"])
    return wl, b, w, kc, vc


def _f64(a, dt):
    if dt == "bf16":
        return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, np.float64)


def _norm(v, g, eps):
    return v * g / np.sqrt(np.dot(v, v) / v.shape[-1] + eps)


def _rot(x, p, theta):
    hd = x.shape[-1]
    h = hd // 2
    c = (x[:h] + 1j * x[h:]) * np.exp(1j * p * theta ** (-np.arange(0, hd, 2) / hd))
    return np.concatenate([c.real, c.imag])


class RowDrafter:
    """One row at a time: its KV goes into the dict caches, then it attends to
    every cached position at or before its own.  Returns (logits, hidden)."""

    def __init__(self, dm, w):
        self.dm = dm
        self.P = {k: _f64(v, dm.dtype) for k, v in w.items() if not isinstance(v, list)}

    def row(self, keys, vals, streams, e, p):
        dm, P = self.dm, self.P
        H, G, hd = dm.n_heads, dm.n_kv_heads, dm.head_dim
        inp = np.concatenate([_norm(streams[s], P["gamma_stream"][s], dm.eps) for s in range(3)] + [e])
        x = P["w_fc"].dot(inp)
        u = x if dm.post_norm else _norm(x, P["gamma_in"], dm.eps)
        qkv = P["w_qkv"].dot(u)
        q = [_rot(qkv[h * hd:(h + 1) * hd], p, dm.rope_theta) for h in range(H)]
        keys[p] = [_rot(qkv[(H + g) * hd:(H + g + 1) * hd], p, dm.rope_theta) for g in range(G)]
        vals[p] = [qkv[(H + G + g) * hd:(H + G + g + 1) * hd] for g in range(G)]
        seen = sorted(t for t in keys if t <= p)
        heads = []
        for h in range(H):
            g = h * G // H
            s = np.array([keys[t][g].dot(q[h]) for t in seen]) / np.sqrt(hd)
            heads.append(scipy.special.softmax(s).dot(np.array([vals[t][g] for t in seen])))
        att = P["w_o"].dot(np.concatenate(heads))

        def mlp(m):
            gate = P["w_gate"].dot(m)
            return P["w_down"].dot(gate * scipy.special.expit(gate) * P["w_up"].dot(m))

        if dm.post_norm:
            a = _norm(x + att, P["gamma_post"], dm.eps)
            hidden = _norm(a + mlp(a), P["gamma_final"], dm.eps)
            z = hidden
        else:
            a = x + att
            hidden = a + mlp(_norm(a, P["gamma_post"], dm.eps))
            z = _norm(hidden, P["gamma_final"], dm.eps)
        return P["w_lm"].dot(z), hidden


def independent_chain(dm, w, b, kc, vc, r):
    """The K-pass chain of request r written out: the verify rows up to the NTP
    row, then K-1 rows of (own hidden state x3, embedding of the last draft)."""
    dt, bs = dm.dtype, dm.block_size
    D = RowDrafter(dm, w)
    q0 = int(b["qsl"][r])
    a = int(b["accepted"][r])
    keys, vals = {}, {}
    for p in range(int(b["prev_pos"][q0])):
        blk = b["block_table"][r][p // bs]
        keys[p] = list(_f64(kc[blk, :, p % bs, :], dt))
        vals[p] = list(_f64(vc[blk, :, p % bs, :], dt))
    emb = _f64(w["emb"], dt)
    Ht = _f64(b["H_tgt"], dt)
    for j in range(a + 1):
        nxt = int(b["bonus"][r]) if j == a else int(b["prev_tok"][q0 + j + 1])
        lg, hid = D.row(keys, vals, Ht[q0 + j], emb[nxt], int(b["prev_pos"][q0 + j]))
    out = [lg]
    p0 = int(b["prev_pos"][q0 + a])
    for k in range(2, dm.K + 1):
        t = int(np.argmax(lg))
        lg, hid = D.row(keys, vals, np.stack([hid] * 3), emb[t], p0 + k - 1)
        out.append(lg)
    return np.stack(out)


@pytest.mark.parametrize("post_norm", [False, True])
def test_matches_independent_chain(post_norm):
    wl, b, w, kc, vc = _setup("tiny_fp32", random_gains=True, post_norm=post_norm)
    res = O.draft_autoregressive(wl.dims, w, b, kc, vc)
    for r in range(wl.batch):
        ref = independent_chain(wl.dims, w, b, kc, vc, r)
        np.testing.assert_allclose(res["req"][r]["logits"], ref, rtol=0, atol=1e-11)
        np.testing.assert_array_equal(res["req"][r]["draft"], np.argmax(ref, axis=-1))


@pytest.mark.parametrize("name", ["tiny_fp32", "small_prenorm", "small_postnorm_hd128"])
def test_first_pass_is_the_parallel_ntp_row(name):
    wl, b, w, kc, vc = _setup(name)
    ar = O.draft_autoregressive(wl.dims, w, b, kc, vc)
    par = O.draft_step(wl.dims, w, b, kc, vc)
    for r in range(wl.batch):
        assert ar["req"][r]["draft"][0] == par["req"][r]["draft"][0]
        np.testing.assert_allclose(ar["req"][r]["logits"][0], par["req"][r]["logits"][0],
                                   rtol=0, atol=1e-10)
        # every later pass sits at the position of the parallel step's MASK row
        np.testing.assert_array_equal(ar["req"][r]["pos"],
                                      par["meta"]["pos"][par["meta"]["sample_idx"][r * wl.dims.K:
                                                                                   (r + 1) * wl.dims.K]])


def test_k1_is_the_parallel_step():
    wl, b, w, kc, vc = _setup("small_prenorm", K=1)
    ar = O.draft_autoregressive(wl.dims, w, b, kc, vc)
    par = O.draft_step(wl.dims, w, b, kc, vc)
    for r in range(wl.batch):
        np.testing.assert_array_equal(ar["req"][r]["logits"], par["req"][r]["logits"])
        np.testing.assert_array_equal(ar["req"][r]["z"], par["req"][r]["z"])


@pytest.mark.parametrize("name", ["small_prenorm", "small_postnorm_hd128"])
def test_bf16_stores_and_tracking(name):
    wl, b, w, kc, vc = _setup(name)
    res = O.draft_autoregressive(wl.dims, w, b, kc, vc)
    res64 = O.draft_autoregressive(wl.dims, w, b, kc, vc, round_stores=False)
    for r in range(wl.batch):
        z = res["req"][r]["z"]
        assert np.array_equal(O.bf16_round(z), z)
        h = res["req"][r]["hidden"]
        assert not np.array_equal(O.bf16_round(h), h)
        # the chains agree as long as they draft the same tokens
        d, d64 = res["req"][r]["draft"], res64["req"][r]["draft"]
        same = int(np.argmax(np.append(d != d64, True)))
        n = min(same + 1, len(d))
        diff = np.abs(res["req"][r]["logits"][:n] - res64["req"][r]["logits"][:n]).max()
        assert diff <= 2e-2, diff


def _planted(monkeypatch, mistake):
    """A copy of the oracle's layer with one mistake planted."""
    real = O.decoder_layer

    def layer(dims, Pl, h_in, pos, att_rows, Kseq, Vseq, R, last):
        if mistake == "position" and len(pos) == 1:
            pos = pos - 1
        if mistake == "no_kv_kept" and len(pos) == 1:
            Kseq, Vseq = Kseq.copy(), Vseq.copy()
        out = real(dims, Pl, h_in, pos, att_rows, Kseq, Vseq, R, last)
        if mistake == "feed_z":
            out = dict(out, hidden=out["out"])
        return out

    monkeypatch.setattr(O, "decoder_layer", layer)


@pytest.mark.parametrize("mistake", ["feed_z", "position", "no_kv_kept"])
def test_planted_mistakes_fail_the_chain_pin(monkeypatch, mistake):
    wl, b, w, kc, vc = _setup("tiny_fp32", random_gains=True)
    _planted(monkeypatch, mistake)
    res = O.draft_autoregressive(wl.dims, w, b, kc, vc)
    worst = max(np.abs(res["req"][r]["logits"] - independent_chain(wl.dims, w, b, kc, vc, r)).max()
                for r in range(wl.batch))
    assert worst > 1e-6, (mistake, worst)
