"""pe_argmax_noalloc: the LM head + argmax for callers that cannot allocate
device memory (an engine that has reserved all of it, code running during
another component's CUDA-graph capture, a fixed memory plan).  Its scratch is a
static device array instead of a caller workspace.  Through the C-ABI, two calls
in a row must give what pe_argmax gives on the same rows: the same draft tokens
and logits within the parity tolerance of the other tests."""

import numpy as np
import pytest

from parity import LOGIT_TOL, TIE_WINDOW, cuda_or_skip, host, setup
from speculative_drafting_gb300 import binding

pytestmark = pytest.mark.gpu


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


def test_noalloc_argmax_rejects_rows_beyond_its_array():
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup("tiny_fp32", want_logits=False)
    too_many = 4097
    z = torch.zeros(too_many, wl.dims.d, dtype=torch.float32, device="cuda")
    out = torch.zeros(too_many, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.PeError) as e:
        r.drafter.argmax_noalloc(z, too_many, out)
    assert e.value.code == binding.PE_ERR_ARG
