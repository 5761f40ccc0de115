"""Parity of pe_verify_greedy with the oracle's greedy verification.

Target tokens, accepted counts and bonus tokens are index results: they must be
bit-exact.  The oracle decodes the logits to fp64 (exact for fp32 and bf16), so
both sides compare the same values and the lowest-index tie rule decides equal
values the same way.  Cases: the seeded verify batches (small ragged ones whose
rows start off the 16-byte grid, and the full K=7 batches over a 201,088-token
vocabulary), exact ties, NaN and signed zeros, a one-token vocabulary, empty
requests, a logits pointer off the 16-byte grid, long requests, and a qsl the
kernel must clamp.
"""

import numpy as np
import pytest

from oracle import pe_oracle as O
from parity import built, cuda_or_skip, host
from speculative_drafting_gb300 import binding, workloads as W

pytestmark = pytest.mark.gpu


def _dtype_code(dtype):
    return binding.PE_DTYPE_BF16 if dtype == "bf16" else binding.PE_DTYPE_F32


def _run(qsl, tok, logits, dtype, offset=0):
    """Upload, call through the C-ABI, return (target, accepted, bonus, status).

    logits: [T_in][V] float32, or uint16 bf16 bits.  offset > 0 places the
    logits that many elements into a larger buffer (an unaligned base)."""
    torch = cuda_or_skip()
    built()
    B, T_in = len(qsl) - 1, len(tok)
    V = logits.shape[1]
    d_qsl = torch.from_numpy(np.ascontiguousarray(qsl, dtype=np.int32)).cuda()
    d_tok = torch.from_numpy(np.ascontiguousarray(tok, dtype=np.int32)).cuda()
    flat = np.ascontiguousarray(logits).reshape(-1)
    if dtype == "bf16":
        flat = flat.view(np.int16)
    host_buf = np.zeros(flat.size + offset + 8, dtype=flat.dtype)
    host_buf[offset:offset + flat.size] = flat
    d_buf = torch.from_numpy(host_buf).cuda()
    d_logits = d_buf[offset:]
    target = torch.full((max(T_in, 1),), -7, dtype=torch.int32, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    bon = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    ws = binding.verify_workspace(max(T_in, 1), V)
    binding.verify_greedy(B, T_in, d_qsl, d_tok, d_logits, V, _dtype_code(dtype), target, acc,
                          bon, ws)
    torch.cuda.synchronize()
    st, _ = binding.read_status_ws(ws)
    return host(target)[:T_in], host(acc), host(bon), st


def _oracle(qsl, tok, logits, dtype):
    return O.verify_greedy(qsl, tok, O.decode(logits, dtype))


def _check(qsl, tok, logits, dtype, offset=0, expect_status=0):
    got = _run(qsl, tok, logits, dtype, offset)
    ref = _oracle(qsl, tok, logits, dtype)
    for g, r, what in zip(got[:3], ref, ("target_tok", "accepted", "bonus")):
        np.testing.assert_array_equal(g, r, err_msg=what)
    assert got[3] == expect_status
    return got


@pytest.mark.parametrize("name", ["verify_small", "verify_small_bf16", "verify_b1_k7",
                                  "verify_b64_k7", "verify_b64_k7_bf16"])
def test_verify_batches(name):
    wl = W.get_verify(name)
    b = W.make_verify_batch(wl)
    t, a, bo, _ = _check(b["qsl"], b["tok"], b["logits"], wl.dtype)
    # the planted counts come back as well
    np.testing.assert_array_equal(a, b["planted_accepted"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 7, 1000, 4099])
def test_exact_ties_and_special_values(dtype, V):
    rng = np.random.default_rng(V)
    rows = []
    rows.append(np.zeros(V))                                    # all equal: index 0
    rows.append(rng.integers(-2, 3, V).astype(np.float64))      # many exact ties
    x = rng.integers(-2, 3, V).astype(np.float64)
    x[x == 0] = -0.0                                            # -0 and +0 tie
    x[::3] = 0.0
    rows.append(x)
    rows.append(np.full(V, -np.inf))                            # all -inf
    y = rng.standard_normal(V)
    y[V // 2] = np.nan                                          # a NaN wins
    y[-1] = np.nan
    rows.append(y)
    z = rng.standard_normal(V)
    z[-1] = np.inf                                              # the last element wins
    rows.append(z)
    lg = np.stack(rows).astype(np.float32)
    if dtype == "bf16":
        lg = W.f32_to_bf16_bits(lg)
    T = lg.shape[0]
    qsl = np.array([0, 2, 2, T], np.int32)                      # an empty request inside
    tok = rng.integers(0, V, T).astype(np.int32)
    for offset in (0, 1, 3):                                    # bases off the 16-byte grid
        _check(qsl, tok, lg, dtype, offset=offset)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_long_requests(dtype):
    """Requests of thousands of rows (a verified prefill) over a small vocabulary."""
    rng = np.random.default_rng(11)
    V, n = 50, (3000, 1, 777)
    T = sum(n)
    lg = rng.integers(-3, 4, (T, V)).astype(np.float32)
    tgt = O.target_argmax(lg)
    tok = rng.integers(0, V, T).astype(np.int32)
    tok[1:2500] = tgt[:2499]  # a long accepted prefix in the first request
    tok[2500] = (tgt[2499] + 1) % V
    qsl = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    if dtype == "bf16":
        lg = W.f32_to_bf16_bits(lg)
    _, a, _, _ = _check(qsl, tok, lg, dtype)
    assert a[0] == 2499


def test_empty_batch_rows():
    """T_in = 0: every request is empty (accepted 0, bonus -1)."""
    t, a, bo, st = _run(np.zeros(4, np.int32), np.zeros(0, np.int32), np.zeros((0, 10), np.float32),
                        "f32")
    assert list(a) == [0, 0, 0] and list(bo) == [-1, -1, -1] and st == 0


def test_bad_qsl_is_clamped_and_reported():
    rng = np.random.default_rng(5)
    V, T = 300, 12
    lg = rng.standard_normal((T, V)).astype(np.float32)
    tok = rng.integers(0, V, T).astype(np.int32)
    qsl = np.array([0, 5, 3, 40], np.int32)  # decreasing, then past T_in
    t, a, bo, st = _run(qsl, tok, lg, "f32")
    assert st & binding.PE_ST_ROWS_RANGE
    # request 1 clamps to no rows; request 2 to rows 3..11; request 0 is untouched
    ref = _oracle(np.array([0, 5, 5, 12], np.int32), tok, lg, "f32")
    assert a[0] == ref[1][0] and bo[0] == ref[2][0]
    assert a[1] == 0 and bo[1] == -1
    ref2 = _oracle(np.array([0, 9], np.int32), tok[3:], lg[3:], "f32")
    assert a[2] == ref2[1][0] and bo[2] == ref2[2][0]


def test_verify_replays_in_a_cuda_graph():
    """Captured once, replayed: the same results on every replay (the call holds
    no host state and allocates nothing)."""
    torch = cuda_or_skip()
    built()
    wl = W.get_verify("verify_small")
    b = W.make_verify_batch(wl)
    d = {k: torch.from_numpy(b[k]).cuda() for k in ("qsl", "tok", "logits")}
    target = torch.empty(b["T_in"], dtype=torch.int32, device="cuda")
    acc = torch.empty(b["B"], dtype=torch.int32, device="cuda")
    bon = torch.empty(b["B"], dtype=torch.int32, device="cuda")
    ws = binding.verify_workspace(b["T_in"], b["V"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        binding.verify_greedy(b["B"], b["T_in"], d["qsl"], d["tok"], d["logits"], b["V"],
                              binding.PE_DTYPE_F32, target, acc, bon, ws, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        binding.verify_greedy(b["B"], b["T_in"], d["qsl"], d["tok"], d["logits"], b["V"],
                              binding.PE_DTYPE_F32, target, acc, bon, ws, stream=s)
    ref = _oracle(b["qsl"], b["tok"], b["logits"], "f32")
    for _ in range(3):
        target.fill_(-9)
        acc.fill_(-9)
        bon.fill_(-9)
        g.replay()
        torch.cuda.synchronize()
        for got, want in zip((target, acc, bon), ref):
            np.testing.assert_array_equal(host(got), want)
