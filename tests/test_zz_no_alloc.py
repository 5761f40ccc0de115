"""pe_argmax_noalloc: the LM head + argmax for callers that cannot allocate
device memory (an engine that has reserved all of it, a runtime bound to a fixed
memory plan).  Its scratch is a static device array instead of a caller
workspace.  Through the C-ABI, two calls in a row must give what pe_argmax gives
on the same rows (the same plan, so the same draft tokens and logits), and at
the GPT-OSS vocabulary the drafts of the oracle."""

import re

import numpy as np
import pytest

from oracle import pe_oracle as O
from parity import LOGIT_TOL, TIE_WINDOW, check_drafts, cuda_or_skip, host, setup
from speculative_drafting_gb300 import binding

pytestmark = pytest.mark.gpu


def _max_rows():
    """PE_NOALLOC_MAX_ROWS as include/pe.h defines it."""
    text = open(binding.HEADER).read()
    return int(re.search(r"#define\s+PE_NOALLOC_MAX_ROWS\s+(\d+)", text).group(1))


@pytest.mark.parametrize("name", ["small_prenorm", "small_postnorm_hd128", "tiny_fp32"])
def test_noalloc_argmax_matches_argmax(name):
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup(name)
    r.run()  # pe_argmax with its workspace: the reference result
    torch.cuda.synchronize()
    assert r.status()[0] == 0
    ref_draft = host(r.draft).copy()
    ref_logits = host(r.logits).copy()
    n = r.B * wl.dims.K
    tol = LOGIT_TOL[wl.dims.dtype]
    for _ in range(2):  # the static scratch keeps the last call's contents
        draft = torch.full((n,), -7, dtype=torch.int32, device="cuda")
        logits = torch.full((n, wl.dims.vocab), float("nan"), dtype=torch.float32, device="cuda")
        r.drafter.argmax_noalloc(r.z, n, draft, logits=logits)
        torch.cuda.synchronize()
        got_logits = host(logits)
        got_draft = host(draft)
        assert np.abs(got_logits - ref_logits).max() <= tol
        top2 = np.sort(ref_logits, axis=-1)[:, -2:]
        clear = (top2[:, 1] - top2[:, 0]) >= TIE_WINDOW
        np.testing.assert_array_equal(got_draft[clear], ref_draft[clear])
        assert (got_draft >= 0).all() and (got_draft < wl.dims.vocab).all()
        # the same LM-head plan as pe_argmax: the same results bit for bit
        np.testing.assert_array_equal(got_logits, ref_logits)
        np.testing.assert_array_equal(got_draft, ref_draft)


def test_noalloc_argmax_at_the_gpt_oss_vocabulary():
    """V = 201,088 (the GPT-OSS-20B-shaped B=1 step): two calls in a row against
    pe_argmax and against the oracle's drafts of the same request."""
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup("gptoss_b1_k7", want_logits=False)
    r.run()
    torch.cuda.synchronize()
    assert r.status()[0] == 0
    ref_draft = host(r.draft).copy()
    n = r.B * wl.dims.K
    res = O.draft_step(wl.dims, w, b, kc, vc)
    for _ in range(2):
        draft = torch.full((n,), -7, dtype=torch.int32, device="cuda")
        r.drafter.argmax_noalloc(r.z, n, draft)
        torch.cuda.synchronize()
        got = host(draft)
        np.testing.assert_array_equal(got, ref_draft)
        check_drafts("bf16", got, res["req"][0]["logits"], where="noalloc request 0")


def test_noalloc_argmax_rejects_rows_beyond_its_array():
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup("tiny_fp32", want_logits=False)
    too_many = _max_rows() + 1
    z = torch.zeros(too_many, wl.dims.d, dtype=torch.float32, device="cuda")
    out = torch.zeros(too_many, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.PeError) as e:
        r.drafter.argmax_noalloc(z, too_many, out)
    assert e.value.code == binding.PE_ERR_ARG
