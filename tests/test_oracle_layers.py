"""Pins of the oracle's N-layer drafter (CPU only).

"P-EAGLE: parallel speculative decoding in vLLM", Parallel drafting: all
positions pass through the N transformer layers and the LM head at once.  Every
layer but the last needs every valid row (the next layer's keys and values come
from them), and each layer has its own KV cache.

The checks: an independently written row-by-row N-layer drafter (dict caches,
complex-rotation RoPE, scipy softmax) gives the same logits; a pre-norm layer
whose O and down projections are zero is the identity; appending draft
positions leaves the earlier ones unchanged through every layer.
"""

import dataclasses

import numpy as np
import pytest
import scipy.special

from oracle import pe_oracle as O
from speculative_drafting_gb300 import workloads as W
from test_oracle_step import _explicit_rows, _f64, _norm, _rot


def _setup(name, **over):
    wl = W.get(name, **over)
    b = W.make_batch(wl)
    w = W.make_weights(wl)
    kc, vc = W.make_kv_cache(wl, b["num_blocks"])
    return wl, b, w, kc, vc


def _prior_layer(b, kc, vc, dm, r):
    c = int(b["prev_pos"][b["qsl"][r]])
    pk, pv = {}, {}
    for p in range(c):
        blk = b["block_table"][r][p // dm.block_size]
        pk[p] = _f64(kc[blk, :, p % dm.block_size, :], dm.dtype)
        pv[p] = _f64(vc[blk, :, p % dm.block_size, :], dm.dtype)
    return pk, pv


def plain_layers(dm, w, rows, priors):
    """rows: (streams[3][d], emb[d], position) per input row; priors: one
    (keys, values) pair of position -> [G][hd] dicts per layer.  Returns the
    logits of every row."""
    dt = dm.dtype
    top = {k: _f64(v, dt) for k, v in w.items() if k != "layers"}
    layers = [top] + [{k: (np.asarray(v, np.float64) if k == "attn_sink" else _f64(v, dt))
                       for k, v in lw.items()} for lw in w.get("layers", [])]
    if "attn_sink" in w:
        layers[0]["attn_sink"] = np.asarray(w["attn_sink"], np.float64)
    H, G, hd = dm.n_heads, dm.n_kv_heads, dm.head_dim
    hs = []
    for streams, e, p in rows:
        inp = np.concatenate([_norm(streams[s], top["gamma_stream"][s], dm.eps) for s in range(3)] + [e])
        hs.append(top["w_fc"].dot(inp))
    for li, P in enumerate(layers):
        keys, vals = dict(priors[li][0]), dict(priors[li][1])
        qs = []
        for (_, _, p), x in zip(rows, hs):
            u = x if dm.post_norm else _norm(x, P["gamma_in"], dm.eps)
            qkv = P["w_qkv"].dot(u)
            qs.append(np.stack([_rot(qkv[h * hd:(h + 1) * hd], p, dm.rope_theta) for h in range(H)]))
            keys[p] = np.stack([_rot(qkv[(H + g) * hd:(H + g + 1) * hd], p, dm.rope_theta)
                                for g in range(G)])
            vals[p] = np.stack([qkv[(H + G + g) * hd:(H + G + g + 1) * hd] for g in range(G)])
        nxt = []
        for (_, _, p), x, q in zip(rows, hs, qs):
            ps = sorted(t for t in keys if t <= p)
            Kt = np.stack([keys[t] for t in ps])
            Vt = np.stack([vals[t] for t in ps])
            o = []
            for h in range(H):
                g = h * G // H
                sc = Kt[:, g, :].dot(q[h]) / np.sqrt(hd)
                if "attn_sink" in P:
                    pr = scipy.special.softmax(np.concatenate([sc, [P["attn_sink"][h]]]))[:-1]
                else:
                    pr = scipy.special.softmax(sc)
                o.append(pr.dot(Vt[:, g, :]))
            att = P["w_o"].dot(np.concatenate(o))

            def mlp(m):
                gate = P["w_gate"].dot(m)
                return P["w_down"].dot(gate * scipy.special.expit(gate) * P["w_up"].dot(m))

            if dm.post_norm:
                a = _norm(x + att, P["gamma_post"], dm.eps)
                nxt.append(_norm(a + mlp(a), P["gamma_final"], dm.eps))
            else:
                a = x + att
                nxt.append(a + mlp(_norm(a, P["gamma_post"], dm.eps)))
        hs = nxt
    z = hs if dm.post_norm else [_norm(y, layers[-1]["gamma_final"], dm.eps) for y in hs]
    return np.stack([top["w_lm"].dot(v) for v in z])


@pytest.mark.parametrize("post_norm", [False, True])
@pytest.mark.parametrize("sinks", [False, True])
def test_layers_match_independent_drafter(post_norm, sinks):
    wl, b, w, kc, vc = _setup("tiny_fp32", post_norm=post_norm, n_layers=3, sinks=sinks)
    dm = wl.dims
    # distinct gains in every layer, so that a gain taken from the wrong layer shows
    g = np.random.default_rng(7)
    for lw in [w] + w["layers"]:
        for name in ("gamma_in", "gamma_post", "gamma_final"):
            lw[name] = g.uniform(0.5, 1.5, dm.d).astype(np.float32)
    res = O.draft_step(dm, w, b, kc, vc)
    for r in range(wl.batch):
        rows = _explicit_rows(dm, b, w, r)
        priors = [_prior_layer(b, kc[li], vc[li], dm, r) for li in range(dm.n_layers)]
        ref = plain_layers(dm, w, rows, priors)
        np.testing.assert_allclose(res["req"][r]["logits"], ref[-dm.K:], rtol=0, atol=1e-10)


@pytest.mark.parametrize("name", ["tiny_fp32", "small_prenorm"])
def test_zero_output_layer_is_identity(name):
    """Pre-norm: a second layer whose O and down projections are zero adds
    nothing to the residual stream, so z and the logits equal the one-layer
    drafter's, in either precision mode."""
    wl, b, w, kc, vc = _setup(name, n_layers=2)
    w["layers"][0]["w_o"] = np.zeros_like(w["layers"][0]["w_o"])
    w["layers"][0]["w_down"] = np.zeros_like(w["layers"][0]["w_down"])
    res2 = O.draft_step(wl.dims, w, b, kc, vc)
    one = dataclasses.replace(wl.dims, n_layers=1)
    w1 = {k: v for k, v in w.items() if k != "layers"}
    res1 = O.draft_step(one, w1, b, kc[0], vc[0])
    for r in range(wl.batch):
        np.testing.assert_array_equal(res2["req"][r]["z"], res1["req"][r]["z"])
        np.testing.assert_array_equal(res2["req"][r]["k"], res1["req"][r]["k"])


@pytest.mark.parametrize("post_norm", [False, True])
def test_appending_draft_positions_through_layers(post_norm):
    wl, b, w, kc, vc = _setup("small_prenorm", n_layers=2, post_norm=post_norm)
    K = wl.dims.K
    res = O.draft_step(wl.dims, w, b, kc, vc)
    wl2 = dataclasses.replace(wl, dims=dataclasses.replace(wl.dims, K=K + 2))
    b2 = W.make_batch(wl2)
    kc2, vc2 = W.make_kv_cache(wl2, b2["num_blocks"])
    bs = wl.dims.block_size
    for r in range(wl.batch):
        for p in range(int(b["prev_pos"][b["qsl"][r]])):
            blk1 = b["block_table"][r][p // bs]
            blk2 = b2["block_table"][r][p // bs]
            kc2[:, blk2, :, p % bs] = kc[:, blk1, :, p % bs]
            vc2[:, blk2, :, p % bs] = vc[:, blk1, :, p % bs]
    res2 = O.draft_step(wl2.dims, w, b2, kc2, vc2)
    for r in range(wl.batch):
        np.testing.assert_array_equal(res2["req"][r]["z"][:K], res["req"][r]["z"])
        for li in range(2):
            n = len(res["req"][r]["k_layers"][li])
            np.testing.assert_array_equal(res2["req"][r]["k_layers"][li][:n - K],
                                          res["req"][r]["k_layers"][li][:n - K])
