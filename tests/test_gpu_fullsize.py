"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times: the whole batch runs on the GPU; all metadata is compared with
the oracle bit for bit, and the oracle recomputes the layer for a sample of
requests (requests are independent given the weights) for logits, draft tokens,
final hidden states and KV writes.  Properties that hold at any size are checked
on every row."""

import numpy as np
import pytest

from oracle import pe_oracle as O
from parity import (check_close_bf16, check_logits_and_draft, check_meta, check_z, cuda_or_skip, f64,
                    host, setup)

pytestmark = pytest.mark.gpu

CASES = [
    ("gptoss_b1_k7", [0], {}),
    ("gptoss_b64_k7_postnorm", [0, 37, 63], {}),
    ("llama8b_b32_k8_32k", [5, 31], {}),
    # the GPT-oss attention with per-head sink logits
    ("gptoss_b64_k7_postnorm", [11, 50], {"sinks": True}),
]


@pytest.mark.parametrize("name,sample,over", CASES)
def test_full_size_step(name, sample, over):
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup(name, **over)
    r.run()
    torch.cuda.synchronize()
    st, rc = r.status()
    assert st == 0, hex(st)
    dm = wl.dims
    K, bs = dm.K, dm.block_size
    res = O.draft_step(dm, w, b, kc, vc, requests=sample)
    check_meta(r, res["meta"])
    logits = r.logits
    draft = host(r.draft)
    # every row: the draft token is the argmax of the logits the kernel produced
    assert ((draft >= 0) & (draft < dm.vocab)).all()
    gmax = logits.max(dim=1).values
    picked = logits.gather(1, r.draft.long().view(-1, 1)).view(-1)
    assert torch.equal(picked, gmax)
    # sampled requests against the oracle
    z = f64(host(r.z), dm.dtype)
    for rr in sample:
        out = res["req"][rr]
        sl = slice(rr * K, (rr + 1) * K)
        check_z(dm.dtype, z[sl], out["z"], where=f"request {rr}")
        check_logits_and_draft(dm.dtype, host(logits[sl]), draft[sl], out["logits"], where=f"request {rr}")
        slots = torch.from_numpy(out["slot"]).to("cuda")
        got_k = f64(host(r.k_cache[slots // bs, :, slots % bs, :]), dm.dtype)
        got_v = f64(host(r.v_cache[slots // bs, :, slots % bs, :]), dm.dtype)
        check_close_bf16(got_k, out["k"], f"k cache r{rr}", max_ulps=1, min_exact=0.95)
        check_close_bf16(got_v, out["v"], f"v cache r{rr}", max_ulps=1, min_exact=0.95)
    # slots no valid row writes keep their prior contents (a sample of blocks)
    live = res["meta"]["slot"][res["meta"]["slot"] >= 0]
    touched = np.zeros(b["num_blocks"], dtype=bool)
    touched[live // bs] = True
    g = np.random.default_rng(0)
    cand = np.nonzero(~touched)[0]
    pick = g.choice(cand, size=min(64, len(cand)), replace=False)
    idx = torch.from_numpy(pick).to("cuda")
    np.testing.assert_array_equal(host(r.k_cache[idx]), kc[pick])
    np.testing.assert_array_equal(host(r.v_cache[idx]), vc[pick])
