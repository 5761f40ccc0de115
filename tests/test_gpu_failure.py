"""Failure detection without a GPU fault.

Every wait inside the kernels (mbarrier waits on TMA stages, TMEM hand-offs,
cluster partners) gives up after a time limit instead of spinning forever, then
records PE_ST_TIMEOUT in the status word and returns.  The test hook runs one
kernel whose barrier nothing ever arrives on: the wait must run out, the status
must say so, and the next step on the same context must still match the
oracle.  A request whose captured hidden states are NaN must not disturb the
other requests of the batch (nothing mixes rows of different requests).
"""

import ctypes
import re
import time

import numpy as np
import pytest

from oracle import pe_oracle as O
from parity import check_logits_and_draft, cuda_or_skip, host, setup
from speculative_drafting_gb300 import binding

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_the_context_survives():
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup("tiny_fp32")
    lib = binding.load()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    t0 = time.perf_counter()
    rc = lib.pe_test_bounded_wait(ctypes.c_void_p(ws.data_ptr()), 256, ctypes.c_void_p(s.cuda_stream))
    assert rc == binding.PE_OK
    st, code = binding.read_status_ws(ws)
    waited = time.perf_counter() - t0
    assert st == binding.PE_ST_TIMEOUT and code == binding.PE_ERR_TIMEOUT
    assert 1.5 < waited < 30.0  # the 2 s limit, not a hang
    # the context is still usable: a whole step still matches the oracle
    r.run()
    torch.cuda.synchronize()
    assert r.status()[0] == 0
    res = O.draft_step(wl.dims, w, b, kc, vc)
    K = wl.dims.K
    logits, draft = host(r.logits), host(r.draft)
    for rr, out in res["req"].items():
        sl = slice(rr * K, (rr + 1) * K)
        check_logits_and_draft("f32", logits[sl], draft[sl], out["logits"], where=f"request {rr}")


def test_decode_layer_barrier_runs_out_and_the_context_survives():
    """The persistent decode layer's grid barriers are bounded waits too: with the
    first kernel's launch count set far ahead of its arrival counters, its first
    barrier can never complete.  The wait runs out, every CTA of both layer
    kernels leaves, the status says so, and after clearing the workspace header
    the next step matches the oracle."""
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup("small_prenorm", batch=1, n_prev=8, K=7, ctx=(300,))
    text = open(binding.TESTING_HEADER).read()
    off = int(re.search(r"#define\s+PE_TEST_DECODE_EPOCH_BYTE\s+(\d+)u", text).group(1))
    r.prepare()
    torch.cuda.synchronize()
    r.ws[off:off + 4].view(torch.int32).fill_(1 << 20)
    t0 = time.perf_counter()
    r.step()
    r.argmax()
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    st, code = r.status(clear=True)
    assert st & binding.PE_ST_TIMEOUT and code == binding.PE_ERR_TIMEOUT
    assert 1.5 < waited < 30.0  # the 2 s limit, not a hang
    # the same workspace, cleared: a whole step matches the oracle
    r.run()
    torch.cuda.synchronize()
    assert r.status()[0] == 0
    res = O.draft_step(wl.dims, w, b, kc, vc)
    K = wl.dims.K
    logits, draft = host(r.logits), host(r.draft)
    for rr, out in res["req"].items():
        sl = slice(rr * K, (rr + 1) * K)
        check_logits_and_draft("bf16", logits[sl], draft[sl], out["logits"], where=f"request {rr}")


def test_nan_hidden_states_stay_in_their_request():
    torch = cuda_or_skip()
    from speculative_drafting_gb300 import runner, workloads as W

    wl = W.get("small_prenorm")
    b = W.make_batch(wl)
    q0, q1 = int(b["qsl"][1]), int(b["qsl"][2])
    b["H_tgt"][q0:q1] = np.uint16(0x7FC0)  # bf16 NaN in every stream of request 1
    w = W.make_weights(wl)
    kc, vc = W.make_kv_cache(wl, b["num_blocks"])
    r = runner.StepRunner(wl, b, w, kc, vc, want_logits=True)
    r.run()
    torch.cuda.synchronize()
    assert r.status()[0] == 0
    res = O.draft_step(wl.dims, w, b, kc, vc, requests=[0, 2])
    K = wl.dims.K
    logits, draft = host(r.logits), host(r.draft)
    for rr in (0, 2):
        sl = slice(rr * K, (rr + 1) * K)
        check_logits_and_draft("bf16", logits[sl], draft[sl], res["req"][rr]["logits"],
                               where=f"request {rr}")
    # the poisoned request still yields token ids in range (a NaN logit counts as
    # the greatest, lowest index first)
    assert ((draft[K:2 * K] >= 0) & (draft[K:2 * K] < wl.dims.vocab)).all()
