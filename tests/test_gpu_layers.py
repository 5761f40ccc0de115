"""GPU parity of the N-layer drafter against the CPU oracle.

"P-EAGLE: parallel speculative decoding in vLLM", Parallel drafting: all
positions pass through the N layers and the LM head.  With several layers every
layer but the last runs over all non-rejected rows, each layer writes its own KV
cache, and the last layer's sample rows give the drafts.  Checked: all metadata
bit for bit, z and the logits within the step's tolerances, the drafts outside
the tie window, every layer's KV writes, and that no other cache slot changes.
"""

import numpy as np
import pytest

from oracle import pe_oracle as O
from parity import (check_close_bf16, check_logits_and_draft, check_meta, check_z, cuda_or_skip, f64,
                    host, setup)
from speculative_drafting_gb300 import binding

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny_fp32", {"n_layers": 2}),
    ("tiny_fp32", {"n_layers": 2, "K": 1, "n_prev": 2}),  # n_r = K + 1 verify rows
    ("tiny_fp32", {"n_layers": 3, "post_norm": True, "sinks": True}),
    ("small_prenorm", {"n_layers": 3}),
    ("small_postnorm_hd128", {"n_layers": 2}),
    ("small_postnorm_hd128", {"n_layers": 2, "post_norm": False, "sinks": True}),
    # the attention splits merge in a cluster / through global memory
    ("small_prenorm", {"n_layers": 2, "batch": 12, "n_prev": 6, "ctx": ("uniform", 0, 700),
                       "seed": 3}),
    ("small_prenorm", {"n_layers": 2, "batch": 160, "n_prev": 6, "ctx": ("uniform", 0, 700),
                       "seed": 5, "sinks": True}),
]


def _check_layers_kv(wl, kc0, vc0, r, res):
    dt, bs = wl.dims.dtype, wl.dims.block_size
    kc, vc = host(r.k_cache), host(r.v_cache)
    for li in range(wl.dims.n_layers):
        written = np.zeros(kc.shape[1] * bs, dtype=bool)
        for rr, out in res["req"].items():
            slots = out["slot"]
            written[slots] = True
            got_k = f64(kc[li][slots // bs, :, slots % bs, :], dt)
            got_v = f64(vc[li][slots // bs, :, slots % bs, :], dt)
            if dt == "bf16":
                check_close_bf16(got_k, out["k_layers"][li], f"layer {li} k", max_ulps=1, min_exact=0.95)
                check_close_bf16(got_v, out["v_layers"][li], f"layer {li} v", max_ulps=1, min_exact=0.95)
            else:
                np.testing.assert_allclose(got_k, out["k_layers"][li], rtol=1e-5, atol=1e-5)
                np.testing.assert_allclose(got_v, out["v_layers"][li], rtol=1e-5, atol=1e-5)
        untouched = ~written.reshape(kc.shape[1], bs)
        np.testing.assert_array_equal(kc[li].transpose(0, 2, 1, 3)[untouched],
                                      kc0[li].transpose(0, 2, 1, 3)[untouched])
        np.testing.assert_array_equal(vc[li].transpose(0, 2, 1, 3)[untouched],
                                      vc0[li].transpose(0, 2, 1, 3)[untouched])


@pytest.mark.parametrize("name,over", CASES)
def test_layers_match_oracle(name, over):
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup(name, **over)
    r.run()
    torch.cuda.synchronize()
    st, _ = r.status()
    assert st == 0, hex(st)
    res = O.draft_step(wl.dims, w, b, kc, vc)
    check_meta(r, res["meta"])
    K, dt = wl.dims.K, wl.dims.dtype
    z = f64(host(r.z), dt)
    logits = host(r.logits)
    draft = host(r.draft)
    for rr, out in res["req"].items():
        sl = slice(rr * K, (rr + 1) * K)
        check_z(dt, z[sl], out["z"], where=f"request {rr}")
        check_logits_and_draft(dt, logits[sl], draft[sl], out["logits"], where=f"request {rr}")
    _check_layers_kv(wl, kc, vc, r, res)


def test_prefill_sized_request_is_reported():
    """A request with more non-rejected rows than the layers carry sets
    PE_ST_ROWS_RANGE (no fault); the other requests still match the oracle."""
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup("small_prenorm", n_layers=2, n_prev=(20, 6, 6),
                                accepted=(19, 2, 5))
    r.run()
    torch.cuda.synchronize()
    st, _ = r.status()
    assert st & binding.PE_ST_ROWS_RANGE
    res = O.draft_step(wl.dims, w, b, kc, vc, requests=[1, 2])
    K = wl.dims.K
    logits = host(r.logits)
    draft = host(r.draft)
    for rr in (1, 2):
        sl = slice(rr * K, (rr + 1) * K)
        check_logits_and_draft("bf16", logits[sl], draft[sl], res["req"][rr]["logits"],
                               where=f"request {rr}")


def test_full_size_two_layers():
    """GPT-OSS-20B shape, B=64, K=7, post-norm, two layers with sinks: sampled
    requests against the oracle."""
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup("gptoss_b64_k7_postnorm", n_layers=2, sinks=True)
    r.run()
    torch.cuda.synchronize()
    st, _ = r.status()
    assert st == 0, hex(st)
    sample = [4, 41]
    res = O.draft_step(wl.dims, w, b, kc, vc, requests=sample)
    check_meta(r, res["meta"])
    K = wl.dims.K
    z = f64(host(r.z), "bf16")
    draft = host(r.draft)
    for rr in sample:
        sl = slice(rr * K, (rr + 1) * K)
        out = res["req"][rr]
        check_z("bf16", z[sl], out["z"], where=f"request {rr}")
        check_logits_and_draft("bf16", host(r.logits[sl]), draft[sl], out["logits"],
                               where=f"request {rr}")
