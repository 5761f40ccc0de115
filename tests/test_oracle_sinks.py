"""Pins of the oracle's attention sinks (CPU only).

"Attention Drift", section 3 ("What if the verifier has no attention sinks?"):
the GPT-oss attention adds a learned per-head bias logit to the softmax
denominator, an explicit option for a head to attend to nothing.  The oracle
reads it as one more logit whose value row is zero.  The checks: a sink at -inf
is no sink at all; closed forms for one key and for all-ones values; a huge
sink silences the head; and in the whole step a sink changes its own head only.
"""

import dataclasses

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import pe_oracle as O
from speculative_drafting_gb300 import workloads as W


def test_sink_at_minus_infinity_is_no_sink():
    g = np.random.default_rng(0)
    q, K, V = g.standard_normal(16), g.standard_normal((9, 16)), g.standard_normal((9, 16))
    np.testing.assert_allclose(O.attend(q, K, V, -np.inf), O.attend(q, K, V), rtol=1e-15, atol=0)


@pytest.mark.parametrize("sink", [-3.0, 0.0, 0.7, 4.0])
def test_one_key_closed_form(sink):
    g = np.random.default_rng(1)
    q, k, v = g.standard_normal(16), g.standard_normal(16), g.standard_normal(16)
    s = q @ k / 4.0  # sqrt(16)
    want = v / (1.0 + np.exp(sink - s))
    np.testing.assert_allclose(O.attend(q, k[None], v[None], sink), want, rtol=1e-13)


@pytest.mark.parametrize("sink", [-2.0, 1.5])
def test_weights_sum_below_one(sink):
    """With every value row equal to ones the output is the mass the real keys
    keep: Z / (Z + e^sink), Z the sum of their exponentials."""
    g = np.random.default_rng(2)
    q, K = g.standard_normal(32), g.standard_normal((20, 32))
    s = K @ q / np.sqrt(32)
    want = 1.0 / (1.0 + np.exp(sink - logsumexp(s)))
    got = O.attend(q, K, np.ones((20, 32)), sink)
    np.testing.assert_allclose(got, np.full(32, want), rtol=1e-13)


def test_huge_sink_silences_the_head():
    g = np.random.default_rng(3)
    q, K, V = g.standard_normal(16), g.standard_normal((5, 16)), g.standard_normal((5, 16))
    assert np.abs(O.attend(q, K, V, 80.0)).max() < 1e-30


def test_step_sink_changes_its_own_head_only():
    wl = W.get("tiny_fp32", sinks=True)
    b = W.make_batch(wl)
    w = W.make_weights(wl)
    kc, vc = W.make_kv_cache(wl, b["num_blocks"])
    H, hd = wl.dims.n_heads, wl.dims.head_dim
    base = dict(w)
    base.pop("attn_sink")
    ref = O.draft_step(wl.dims, base, b, kc, vc, want_logits=False)
    only = dict(base)
    only["attn_sink"] = np.full(H, -np.inf, np.float32)
    only["attn_sink"][2] = 0.5
    got = O.draft_step(wl.dims, only, b, kc, vc, want_logits=False)
    for r in ref["req"]:
        a0 = ref["req"][r]["attn"].reshape(-1, H, hd)
        a1 = got["req"][r]["attn"].reshape(-1, H, hd)
        for h in range(H):
            if h == 2:
                assert np.abs(a1[:, h] - a0[:, h]).max() > 1e-6
            else:
                np.testing.assert_array_equal(a1[:, h], a0[:, h])
