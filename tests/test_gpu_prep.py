"""GPU parity of steps (1)-(3): fused metadata kernel, hidden-state map /
placeholder broadcast, and the per-stream-RMSNorm drafter input, through the
C-ABI (pe_prepare_inputs) against the CPU oracle."""

import numpy as np
import pytest

from oracle import pe_oracle as O
from parity import check_close_bf16, check_meta, cuda_or_skip, f64, host, setup

pytestmark = pytest.mark.gpu

CASES = [
    ("tiny_fp32", {}),
    ("tiny_fp32", {"K": 1}),
    ("small_prenorm", {}),
    ("small_postnorm_hd128", {}),
    ("meta_prep_b64", {}),                                   # the full B=64, d=2880 preparation
    ("small_prenorm", {"accepted": (5, 0, 3)}),              # prefill-like, all-rejected, middle
    ("small_postnorm_hd128", {"accepted": (0, 2, 0, 8)}),    # n_r = 1 and full acceptance
    ("small_prenorm", {"batch": 1, "n_prev": 1, "ctx": (0,), "accepted": (0,)}),  # first step
]


@pytest.mark.parametrize("name,over", CASES)
def test_prepare_inputs_matches_oracle(name, over):
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup(name, want_G=True, want_E=True, want_logits=False, kv=False, **over)
    r.prepare()
    torch.cuda.synchronize()
    st, rc = r.status()
    assert st == 0, hex(st)
    meta, G, E, A = O.prepare_inputs(wl.dims, w, b)
    check_meta(r, meta)
    dt = wl.dims.dtype
    # the hidden-state map and the embedding rows are plain copies: bit-exact
    np.testing.assert_array_equal(f64(host(r.G), dt), G)
    np.testing.assert_array_equal(f64(host(r.E), dt), E)
    # A: drafter input of the non-rejected rows, in valid_rows order
    nv = meta["n_valid"]
    A_ref = A[meta["valid_rows"][:nv]]
    A_got = f64(host(r.A)[:nv], dt)
    if dt == "bf16":
        check_close_bf16(A_got, A_ref, "A", max_ulps=1, min_exact=0.995)
    else:
        np.testing.assert_allclose(A_got, A_ref, rtol=2e-6, atol=1e-7)
    # all MASK rows carry identical inputs
    mrows = np.nonzero(meta["is_masked"])[0]
    if len(mrows):
        pos = {o: i for i, o in enumerate(meta["valid_rows"][:nv])}
        Am = A_got[[pos[o] for o in mrows]]
        assert (Am == Am[0]).all()


def test_status_flags_bad_inputs_without_faulting():
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup("small_prenorm", want_logits=False, kv=False)
    # accepted count past the verify rows, a block id out of range where request
    # 0's NTP row writes, a bonus token past V
    r.inp["accepted"][1] = 99
    p_ntp = int(b["prev_pos"][b["qsl"][0] + b["accepted"][0]])
    r.inp["block_table"][0, p_ntp // wl.dims.block_size] = b["num_blocks"] + 5
    r.inp["bonus"][0] = wl.dims.vocab + 3
    r.prepare()
    torch.cuda.synchronize()
    st, rc = r.status()
    from speculative_drafting_gb300 import binding as B
    assert st & B.PE_ST_ACCEPTED_RANGE and st & B.PE_ST_BLOCK_RANGE and st & B.PE_ST_TOKEN_RANGE, hex(st)
    assert rc == B.PE_ERR_DEVICE_INPUT
    # the context is still usable and a clean batch reports nothing
    r2 = setup("small_prenorm", want_logits=False, kv=False)[-1]
    r2.prepare()
    torch.cuda.synchronize()
    assert r2.status()[0] == 0


def test_preparation_only_handle_refuses_layer_calls():
    """A handle made without the layer's weights (they are NULL) prepares inputs
    and refuses the layer's calls on the host, before anything is enqueued."""
    torch = cuda_or_skip()
    from speculative_drafting_gb300 import binding
    wl, b, w, kc, vc, r = setup("meta_prep_b64", want_logits=False, kv=False)
    assert "w_lm" not in r.drafter.weights
    z = torch.zeros(8, wl.dims.d, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(8, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.PeError) as e:
        r.drafter.argmax_noalloc(z, 8, out)
    assert e.value.code == binding.PE_ERR_ARG
    with pytest.raises(binding.PeError) as e:
        r.drafter.test_projection(5, z, 8, torch.zeros(8, 4, device="cuda"))
    assert e.value.code == binding.PE_ERR_ARG
    r.prepare()
    torch.cuda.synchronize()
    st, _ = r.status()
    assert st == 0


@pytest.mark.parametrize("seed", range(40))
def test_metadata_random_batches(seed):
    """Random ragged batches (1-40 requests, K 1-9, 1..K+3 verify rows each,
    contexts 0-300 across block boundaries, block sizes 1, 4 and 16): every
    metadata tensor bit-exact against the oracle, A within one bf16 step."""
    torch = cuda_or_skip()
    g = np.random.default_rng(1000 + seed)
    B = int(g.integers(1, 41))
    K = int(g.integers(1, 10))
    n_prev = tuple(int(x) for x in g.integers(1, K + 4, size=B))
    ctx = tuple(int(x) for x in g.integers(0, 301, size=B))
    bs = int(g.choice([1, 4, 16]))
    wl, b, w, kc, vc, r = setup("tiny_fp32", want_logits=False, kv=False, batch=B, n_prev=n_prev,
                                ctx=ctx, K=K, block_size=bs, seed=seed, has_drafter=False)
    r.prepare()
    torch.cuda.synchronize()
    st, _ = r.status()
    assert st == 0, hex(st)
    meta, G, E, A = O.prepare_inputs(wl.dims, w, b)
    check_meta(r, meta)
    nv = meta["n_valid"]
    np.testing.assert_allclose(f64(host(r.A)[:nv], "f32"), A[meta["valid_rows"][:nv]], rtol=2e-6,
                               atol=1e-7)
