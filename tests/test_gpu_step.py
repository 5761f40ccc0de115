"""GPU parity of the whole parallel-draft step (pe_prepare_inputs ->
pe_draft_step -> pe_argmax) against the CPU oracle on every row, at sizes the
oracle finishes in seconds: every projection spans several 128-row tiles and a
ragged tail, contexts cross block boundaries, one request starts from an empty
context."""

import numpy as np
import pytest

from oracle import pe_oracle as O
from parity import (LOGIT_TOL, check_close_bf16, check_logits_and_draft, check_meta, check_z,
                    cuda_or_skip, f64, host, setup)

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny_fp32", {}),
    ("tiny_fp32", {"post_norm": True}),
    ("tiny_fp32", {"K": 1}),
    ("small_prenorm", {}),
    ("small_prenorm", {"accepted": (5, 0, 3)}),
    ("small_postnorm_hd128", {}),
    ("small_postnorm_hd128", {"post_norm": False, "accepted": (0, 2, 0, 8)}),
    ("small_prenorm", {"K": 1}),
    ("small_prenorm", {"batch": 12, "n_prev": 6, "ctx": ("uniform", 0, 700), "seed": 3}),
    # enough requests that attention splits merge through global memory: the
    # combine stops at each request's own last split
    ("small_prenorm", {"batch": 160, "n_prev": 6, "ctx": ("uniform", 0, 700), "seed": 5}),
    # per-head sink logits (GPT-oss attention) on every normalisation path: the
    # fp32 kernel, the in-cluster merge and the global combine
    ("tiny_fp32", {"sinks": True}),
    ("small_prenorm", {"sinks": True}),
    ("small_postnorm_hd128", {"sinks": True}),
    ("small_prenorm", {"batch": 12, "n_prev": 6, "ctx": ("uniform", 0, 700), "seed": 3, "sinks": True}),
    ("small_prenorm", {"batch": 160, "n_prev": 6, "ctx": ("uniform", 0, 700), "seed": 5,
                       "sinks": True}),
    # decode-sized steps (at most 16 token rows and 16 sample rows): the layer
    # runs as the two persistent kernels
    ("small_prenorm", {"batch": 2, "n_prev": 4, "K": 4, "ctx": (37, 150)}),
    ("small_prenorm", {"batch": 1, "n_prev": 8, "K": 7, "ctx": (300,)}),
    ("small_prenorm", {"batch": 2, "n_prev": (5, 2), "K": 4, "accepted": (4, 0), "ctx": (60, 9),
                       "sinks": True}),
    ("small_postnorm_hd128", {"batch": 2, "n_prev": (3, 1), "K": 5, "ctx": (17, 100)}),
    ("small_postnorm_hd128", {"batch": 1, "n_prev": 9, "K": 8, "ctx": (0,), "post_norm": False}),
    ("small_prenorm", {"batch": 16, "n_prev": 1, "K": 1, "ctx": ("uniform", 0, 400), "seed": 7}),
]


def _check_kv(wl, b, kc0, vc0, r, res):
    """Written slots hold the oracle's k / v; every other slot is untouched."""
    dt = wl.dims.dtype
    bs = wl.dims.block_size
    kc, vc = host(r.k_cache), host(r.v_cache)
    written = np.zeros(kc.shape[0] * bs, dtype=bool)
    for rr, out in res["req"].items():
        slots = out["slot"]
        assert (slots >= 0).all()
        written[slots] = True
        got_k = f64(kc[slots // bs, :, slots % bs, :], dt)
        got_v = f64(vc[slots // bs, :, slots % bs, :], dt)
        if dt == "bf16":
            check_close_bf16(got_k, out["k"], "k cache", max_ulps=1, min_exact=0.95)
            check_close_bf16(got_v, out["v"], "v cache", max_ulps=1, min_exact=0.95)
        else:
            np.testing.assert_allclose(got_k, out["k"], rtol=1e-5, atol=1e-6)
            np.testing.assert_allclose(got_v, out["v"], rtol=1e-5, atol=1e-6)
    w2 = written.reshape(kc.shape[0], bs)
    untouched = ~w2
    np.testing.assert_array_equal(kc.transpose(0, 2, 1, 3)[untouched], kc0.transpose(0, 2, 1, 3)[untouched])
    np.testing.assert_array_equal(vc.transpose(0, 2, 1, 3)[untouched], vc0.transpose(0, 2, 1, 3)[untouched])


@pytest.mark.parametrize("name,over", CASES)
def test_step_matches_oracle(name, over):
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup(name, **over)
    r.run()
    torch.cuda.synchronize()
    st, rc = r.status()
    assert st == 0, hex(st)
    res = O.draft_step(wl.dims, w, b, kc, vc)
    check_meta(r, res["meta"])
    K = wl.dims.K
    dt = wl.dims.dtype
    z = f64(host(r.z), dt)
    logits = host(r.logits)
    draft = host(r.draft)
    for rr, out in res["req"].items():
        sl = slice(rr * K, (rr + 1) * K)
        check_z(dt, z[sl], out["z"], where=f"request {rr}")
        check_logits_and_draft(dt, logits[sl], draft[sl], out["logits"], where=f"request {rr}")
    _check_kv(wl, b, kc, vc, r, res)


def test_step_is_repeatable_and_graph_capturable():
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup("small_prenorm")
    r.run()
    torch.cuda.synchronize()
    first = host(r.logits).copy()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        r.run(stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(r.logits), first)
    assert r.status()[0] == 0


@pytest.mark.parametrize("seed", range(12))
def test_random_steps(seed):
    """Random small steps (bf16, d=320, hd 64): batch 1-24, K 1-8, ragged verify
    rows, contexts 0-600, pre- or post-norm, with or without sinks, one or two
    layers: metadata bit-exact, z and logits within the step's tolerances."""
    torch = cuda_or_skip()
    g = np.random.default_rng(500 + seed)
    B = int(g.integers(1, 25))
    K = int(g.integers(1, 9))
    layers = int(g.integers(1, 3))
    top = K + 1 if layers > 1 else K + 3   # several layers: steady-state rows
    over = dict(batch=B, K=K, n_layers=layers, seed=seed,
                n_prev=tuple(int(x) for x in g.integers(1, top + 1, size=B)),
                ctx=tuple(int(x) for x in g.integers(0, 601, size=B)),
                post_norm=bool(g.integers(0, 2)), sinks=bool(g.integers(0, 2)))
    wl, b, w, kc, vc, r = setup("small_prenorm", **over)
    r.run()
    torch.cuda.synchronize()
    st, _ = r.status()
    assert st == 0, hex(st)
    res = O.draft_step(wl.dims, w, b, kc, vc)
    check_meta(r, res["meta"])
    z = f64(host(r.z), "bf16")
    logits, draft = host(r.logits), host(r.draft)
    for rr, out in res["req"].items():
        sl = slice(rr * K, (rr + 1) * K)
        check_z("bf16", z[sl], out["z"], where=f"request {rr}")
        check_logits_and_draft("bf16", logits[sl], draft[sl], out["logits"], where=f"request {rr}")


def test_bad_context_block_at_a_batch_of_several_waves():
    """A context block id out of range in one request of a batch whose attention
    grid runs several waves (160 requests x 2 KV heads, partials merged by the
    combine kernel): the status word flags it, the step completes, the keys of
    that block are skipped, and every other request still matches the oracle."""
    torch = cuda_or_skip()
    from speculative_drafting_gb300 import binding as Bnd

    wl, b, w, kc, vc, r = setup("small_prenorm", batch=160, n_prev=6,
                                ctx=("uniform", 100, 700), seed=11)
    bad = 37
    bs = wl.dims.block_size
    assert int(b["ctx"][bad]) >= 3 * bs
    # block 1 of the request holds context keys only: no row of this step writes
    # there, so the attention is the one kernel that reads it
    r.inp["block_table"][bad, 1] = int(b["num_blocks"]) + 5
    r.run()
    torch.cuda.synchronize()
    st, rc = r.status()
    assert st & Bnd.PE_ST_BLOCK_RANGE, hex(st)
    assert not st & Bnd.PE_ST_TIMEOUT, hex(st)
    assert rc == Bnd.PE_ERR_DEVICE_INPUT
    K = wl.dims.K
    logits, draft = host(r.logits), host(r.draft)
    others = [0, 1, bad - 1, bad + 1, 100, 159]
    res = O.draft_step(wl.dims, w, b, kc, vc, requests=others)
    for rr in others:
        sl = slice(rr * K, (rr + 1) * K)
        check_logits_and_draft("bf16", logits[sl], draft[sl], res["req"][rr]["logits"],
                               where=f"request {rr}")
    assert ((draft[bad * K:(bad + 1) * K] >= 0) & (draft[bad * K:(bad + 1) * K] < wl.dims.vocab)).all()


def test_batch_of_1100_requests():
    """1100 requests (past the drafter-input kernel's self-indexing limit, an
    attention grid of many waves).  Metadata bit-exact; a sample of requests (the
    first, the last and some between) matches the oracle."""
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup("small_prenorm", batch=1100, n_prev=2, ctx=("uniform", 0, 120),
                                seed=13)
    r.run()
    torch.cuda.synchronize()
    st, _ = r.status()
    assert st == 0, hex(st)
    K = wl.dims.K
    sample = [0, 1, 517, 1024, 1098, 1099]
    res = O.draft_step(wl.dims, w, b, kc, vc, requests=sample)
    check_meta(r, res["meta"])
    logits, draft = host(r.logits), host(r.draft)
    z = f64(host(r.z), "bf16")
    for rr in sample:
        sl = slice(rr * K, (rr + 1) * K)
        check_z("bf16", z[sl], res["req"][rr]["z"], where=f"request {rr}")
        check_logits_and_draft("bf16", logits[sl], draft[sl], res["req"][rr]["logits"],
                               where=f"request {rr}")
