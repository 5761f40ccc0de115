"""The speculative loop on the device: verification feeds the next draft step.

pe_verify_greedy writes its accepted counts and bonus tokens straight into the
buffers pe_prepare_inputs reads, with no host round trip, and the draft step
runs on them ("Attention Drift", section 2: the target keeps the longest
accepted prefix; "P-EAGLE: parallel speculative decoding in vLLM", Parallel
drafting: the NTP row carries the new token).  The oracle runs the same chain
on the host: its verification, then its step on the counts it found.
"""

import dataclasses

import numpy as np
import pytest

from oracle import pe_oracle as O
from parity import built, check_logits_and_draft, check_meta, check_z, cuda_or_skip, f64, host
from speculative_drafting_gb300 import binding, runner, workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,logit_dtype", [("small_prenorm", "f32"),
                                              ("small_postnorm_hd128", "bf16")])
def test_verify_then_draft(name, logit_dtype):
    torch = cuda_or_skip()
    built()
    wl = W.get(name)
    b = W.make_batch(wl)
    w = W.make_weights(wl)
    kc, vc = W.make_kv_cache(wl, b["num_blocks"])
    # the target's logits over the step's verify rows; their tokens are the rows' tokens
    vwl = dataclasses.replace(W.get_verify("verify_small"), batch=wl.batch,
                              n_rows=tuple(int(n) for n in np.diff(b["qsl"])), vocab=wl.dims.vocab,
                              dtype=logit_dtype, seed=11)
    vb = W.make_verify_batch(vwl)
    assert np.array_equal(vb["qsl"], b["qsl"])
    b = dict(b, prev_tok=vb["tok"])
    r = runner.StepRunner(wl, b, w, kc, vc, want_logits=True)
    # verification writes into the step's own input buffers
    lg = torch.from_numpy(vb["logits"].view(np.int16) if logit_dtype == "bf16" else vb["logits"]).cuda()
    target = torch.empty(vb["T_in"], dtype=torch.int32, device="cuda")
    vws = binding.verify_workspace(vb["T_in"], vb["V"])
    code = binding.PE_DTYPE_BF16 if logit_dtype == "bf16" else binding.PE_DTYPE_F32
    r.inp["accepted"].fill_(-5)
    r.inp["bonus"].fill_(-5)
    binding.verify_greedy(vb["B"], vb["T_in"], r.inp["qsl"], r.inp["prev_tok"], lg, vb["V"], code,
                          target, r.inp["accepted"], r.inp["bonus"], vws)
    r.run()
    torch.cuda.synchronize()
    assert binding.read_status_ws(vws)[0] == 0
    assert r.status()[0] == 0
    # the same chain on the host
    t_ref, acc_ref, bon_ref = O.verify_greedy(vb["qsl"], vb["tok"], O.decode(vb["logits"], logit_dtype))
    np.testing.assert_array_equal(host(target), t_ref)
    np.testing.assert_array_equal(host(r.inp["accepted"]), acc_ref)
    np.testing.assert_array_equal(host(r.inp["bonus"]), bon_ref)
    res = O.draft_step(wl.dims, w, dict(b, accepted=acc_ref, bonus=bon_ref), kc, vc)
    check_meta(r, res["meta"])
    K, dt = wl.dims.K, wl.dims.dtype
    logits, draft = host(r.logits), host(r.draft)
    z = f64(host(r.z), dt)
    for rr, out in res["req"].items():
        sl = slice(rr * K, (rr + 1) * K)
        check_z(dt, z[sl], out["z"], where=f"request {rr}")
        check_logits_and_draft(dt, logits[sl], draft[sl], out["logits"], where=f"request {rr}")
