"""Pins of the oracle's numeric primitives against closed forms, hand-worked
examples and independent library routines (CPU only)."""

import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import pe_oracle as O


# --- bf16 rounding ---------------------------------------------------------


@pytest.mark.parametrize("x, want", [
    (1.0, 1.0),
    (1.0 + 2.0 ** -8, 1.0),                        # halfway, 1.0 is the even neighbour
    (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),        # halfway, 1+2^-6 is the even neighbour
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 1.0 + 2.0 ** -7),  # just above halfway rounds up
    (3.14159265358979, 3.140625),                  # 0x4049
    (-2.5, -2.5),
    (0.0, 0.0),
    (65536.0 * 1.00390625, 65536.0),               # 1+2^-8 scaled: tie to even again
    (1e-3, 0.00099945068359375),                 # 0x3A83
])
def test_bf16_round_worked_values(x, want):
    assert O.bf16_round(np.float64(x)) == want


def test_bf16_round_matches_torch_on_float32_inputs():
    # For values that are exact float32 numbers, nearest-even bf16 from fp64 and
    # torch's float32 -> bfloat16 conversion are the same rounding.
    g = np.random.default_rng(1)
    v = np.concatenate([g.standard_normal(20000) * s for s in (1e-3, 1.0, 1e3)]).astype(np.float32)
    # add exact ties: bf16 value + half an ulp
    b = torch.tensor(v[:1000]).to(torch.bfloat16).to(torch.float32).numpy()
    ulp = np.abs(b) * 2.0 ** -7
    ties = (b + np.sign(b) * ulp / 2 * (np.abs(b) >= 2.0 ** -120)).astype(np.float32)
    v = np.concatenate([v, ties])
    ref = torch.tensor(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_round(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_decode():
    bits = np.array([0x3F80, 0xC000, 0x4049, 0x0000, 0x8000, 0x3A83], dtype=np.uint16)
    assert list(O.bf16_decode(bits)) == [1.0, -2.0, 3.140625, 0.0, -0.0, 0.00099945068359375]


# --- RMS / RMSNorm ---------------------------------------------------------


def test_rms_definition():
    # ||x||_2 / sqrt(d): [3, 4] -> 5 / sqrt(2)
    assert O.rms([3.0, 4.0]) == pytest.approx(5.0 / math.sqrt(2.0), rel=1e-15)


def test_rmsnorm_worked_values():
    r = math.sqrt(12.5)
    np.testing.assert_allclose(O.rmsnorm([3.0, 4.0], np.array([1.0, 1.0]), 0.0),
                               [3 / r, 4 / r], rtol=1e-15)
    np.testing.assert_allclose(O.rmsnorm([3.0, 4.0], np.array([2.0, 0.5]), 0.0),
                               [6 / r, 2 / r], rtol=1e-15)
    # eps sits inside the square root, beside the mean square
    np.testing.assert_allclose(O.rmsnorm([1.0, 1.0], np.array([1.0, 1.0]), 1.0),
                               [1 / math.sqrt(2)] * 2, rtol=1e-15)
    assert np.all(O.rmsnorm(np.zeros(8), np.ones(8), 1e-6) == 0.0)


def test_rmsnorm_scale_invariance_and_unit_rms():
    g = np.random.default_rng(2)
    x = g.standard_normal(2880) * 16.0
    y = O.rmsnorm(x, np.ones(2880), 0.0)
    assert O.rms(y) == pytest.approx(1.0, rel=1e-14)
    np.testing.assert_allclose(O.rmsnorm(x * 37.0, np.ones(2880), 0.0), y, rtol=1e-13)


# --- linear ----------------------------------------------------------------


def test_linear_orientation():
    # W is [out][in]; y = x W^T.  A transposed operand would not even conform.
    x = np.array([[1.0, 2.0, 3.0]])
    W = np.array([[1.0, 0.0, 0.0], [0.0, 1.0, 1.0]])
    np.testing.assert_array_equal(O.linear(x, W), [[1.0, 5.0]])


# --- RoPE ------------------------------------------------------------------


def test_rope_hd2_is_rotation_by_position():
    for p in (0, 1, 7, 1000):
        got = O.rope(np.array([[[1.0, 0.0]]]), np.array([p]), 10000.0)[0, 0]
        np.testing.assert_allclose(got, [math.cos(p), math.sin(p)], atol=1e-15)


def test_rope_rotate_half_pairing_and_frequencies():
    # hd = 4: pairs (0, 2) at frequency 1 and (1, 3) at theta^(-1/2)
    th = 10000.0
    got = O.rope(np.array([[[1.0, 0.0, 0.0, 0.0]]]), np.array([1]), th)[0, 0]
    np.testing.assert_allclose(got, [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    got = O.rope(np.array([[[0.0, 1.0, 0.0, 0.0]]]), np.array([3]), th)[0, 0]
    f = th ** -0.5
    np.testing.assert_allclose(got, [0, math.cos(3 * f), 0, math.sin(3 * f)], atol=1e-15)
    got = O.rope(np.array([[[0.0, 0.0, 1.0, 0.0]]]), np.array([1]), th)[0, 0]
    np.testing.assert_allclose(got, [-math.sin(1), 0, math.cos(1), 0], atol=1e-15)


def test_rope_relative_position_property():
    g = np.random.default_rng(3)
    q = g.standard_normal((1, 1, 64))
    k = g.standard_normal((1, 1, 64))
    d1 = np.dot(O.rope(q, [100], 1e4)[0, 0], O.rope(k, [37], 1e4)[0, 0])
    d2 = np.dot(O.rope(q, [5100], 1e4)[0, 0], O.rope(k, [5037], 1e4)[0, 0])
    assert d1 == pytest.approx(d2, rel=1e-10)
    np.testing.assert_allclose(np.linalg.norm(O.rope(q, [12345], 1e4)), np.linalg.norm(q), rtol=1e-14)
    np.testing.assert_array_equal(O.rope(q, [0], 1e4), q)


# --- attention -------------------------------------------------------------


def test_attend_single_key_returns_value():
    g = np.random.default_rng(4)
    v = g.standard_normal((1, 16))
    np.testing.assert_allclose(O.attend(g.standard_normal(16), g.standard_normal((1, 16)), v)[None], v)


def test_attend_equal_scores_is_mean():
    g = np.random.default_rng(5)
    kk = np.tile(g.standard_normal(16), (9, 1))
    v = g.standard_normal((9, 16))
    np.testing.assert_allclose(O.attend(g.standard_normal(16), kk, v), v.mean(0), rtol=1e-13)


def test_attend_two_key_closed_form():
    # q = (1, 0), keys (0, 0) and (2, 0), hd = 2: scores 0 and 2/sqrt(2)
    p2 = 1.0 / (1.0 + math.exp(-math.sqrt(2.0)))
    got = O.attend(np.array([1.0, 0.0]), np.array([[0.0, 0.0], [2.0, 0.0]]),
                   np.array([[1.0, 0.0], [0.0, 1.0]]))
    np.testing.assert_allclose(got, [1 - p2, p2], rtol=1e-15)


def test_attend_matches_scipy_softmax():
    g = np.random.default_rng(6)
    q, K, V = g.standard_normal(64), g.standard_normal((300, 64)) * 3, g.standard_normal((300, 64))
    ref = scipy.special.softmax(K @ q / 8.0) @ V
    np.testing.assert_allclose(O.attend(q, K, V), ref, rtol=1e-12)


# --- SwiGLU / argmax -------------------------------------------------------


def test_silu_values():
    assert O.silu(0.0) == 0.0
    assert O.silu(1.0) == pytest.approx(0.7310585786300049, rel=1e-15)
    assert O.silu(-1.0) == pytest.approx(-0.2689414213699951, rel=1e-15)
    t = np.linspace(-30, 30, 101)
    np.testing.assert_allclose(O.silu(t), t * scipy.special.expit(t), rtol=1e-13, atol=1e-300)


def test_swiglu_worked_example():
    # m = [1, 2]; gate picks m0, up picks m1; down sums: silu(1) * 2
    m = np.array([[1.0, 2.0]])
    wg = np.array([[1.0, 0.0]])
    wu = np.array([[0.0, 1.0]])
    wd = np.array([[1.0], [3.0]])
    got = O.swiglu_mlp(m, wg, wu, wd)
    np.testing.assert_allclose(got, [[2 * O.silu(1.0), 6 * O.silu(1.0)]], rtol=1e-15)


def test_argmax_lowest_index_on_ties():
    np.testing.assert_array_equal(O.argmax_lowest(np.array([[1.0, 3.0, 3.0], [5.0, 5.0, 5.0]])), [1, 0])


# --- paged cache read --------------------------------------------------------


def test_request_kv_sequence_matches_elementwise_walk():
    g = np.random.default_rng(7)
    NB, G, bs, hd = 9, 2, 4, 3
    cache = g.standard_normal((NB, G, bs, hd)).astype(np.float32)
    table = np.array([[5, 2, 7, -1], [0, 8, 1, 3]], dtype=np.int32)
    for r, n in ((0, 11), (1, 16), (1, 1)):
        seq = O.request_kv_sequence(cache, table, r, n, bs, "f32")
        for p in range(n):
            for gg in range(G):
                np.testing.assert_array_equal(seq[p, gg], cache[table[r][p // bs], gg, p % bs])
