"""Shared helpers of the GPU parity tests: run a workload through the C-ABI and
compare against the CPU oracle on the same seeded inputs."""

from __future__ import annotations

import functools

import numpy as np
import pytest

from oracle import pe_oracle as O
from speculative_drafting_gb300 import build, runner, workloads as W

# Tolerances of the step (written here, used by every parity test):
#   metadata / index tensors / the G and E copies: bit-exact
#   fp32 mode: logits max-abs <= 1e-5
#   bf16 mode: logits max-abs <= 2e-2, and the greedy token agrees unless the
#   oracle's two best logits are within 1e-3 of each other.
LOGIT_TOL = {"f32": 1e-5, "bf16": 2e-2}
TIE_WINDOW = 1e-3


def cuda_or_skip():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch


@functools.lru_cache(maxsize=None)
def built():
    return build.build()


def setup(name, want_G=False, want_E=False, want_logits=True, kv=True, **over):
    """Generate a workload, upload it and return (wl, batch, weights, kc, vc, runner)."""
    built()
    wl = W.get(name, **over)
    b = W.make_batch(wl)
    w = W.make_weights(wl)
    kc = vc = None
    if kv and wl.has_drafter:
        kc, vc = W.make_kv_cache(wl, b["num_blocks"])
    r = runner.StepRunner(wl, b, w, kc, vc, want_G=want_G, want_E=want_E,
                          want_logits=want_logits and wl.has_drafter)
    return wl, b, w, kc, vc, r


def host(t):
    return runner.to_host_bits(t)


def check_meta(r, ref):
    """Every metadata tensor bit-exact."""
    m = {k: host(v) for k, v in r.meta.t.items()}
    for k in ("out_qsl", "tok", "pos", "is_rejected", "is_masked", "hidden_src", "slot",
              "valid_qsl", "valid_rows", "sample_idx", "seq_len"):
        np.testing.assert_array_equal(m[k], ref[k], err_msg=k)
    assert int(m["n_valid"][0]) == ref["n_valid"]


def f64(a, dtype):
    return O.decode(a, dtype)


def check_logits_and_draft(dtype, got_logits, got_draft, ref_logits, where=""):
    """Logit tolerance, then argmax agreement outside the tie window."""
    tol = LOGIT_TOL[dtype]
    diff = np.abs(got_logits.astype(np.float64) - ref_logits)
    print(f"[parity] {where}: logits max-abs {diff.max():.3g} (tolerance {tol})")
    assert diff.max() <= tol, f"{where} logits max-abs {diff.max():.3g} > {tol}"
    top2 = np.sort(ref_logits, axis=-1)[:, -2:]
    gap = top2[:, 1] - top2[:, 0]
    ref_draft = O.argmax_lowest(ref_logits)
    for i in range(len(got_draft)):
        if gap[i] >= TIE_WINDOW:
            assert got_draft[i] == ref_draft[i], f"{where} row {i}: draft {got_draft[i]} != {ref_draft[i]}"
        else:
            # inside the window: any token whose oracle logit is within the window is valid
            assert ref_logits[i, got_draft[i]] >= top2[i, 1] - TIE_WINDOW - tol, f"{where} row {i}"
    return diff.max()


def check_drafts(dtype, got_draft, ref_logits, where=""):
    """Draft tokens alone (no logits stored): equal to the oracle's argmax where
    its two best logits are at least TIE_WINDOW apart; inside the window, a token
    whose oracle logit is within the window (plus the logit tolerance) of the top."""
    tol = LOGIT_TOL[dtype]
    top2 = np.sort(ref_logits, axis=-1)[:, -2:]
    gap = top2[:, 1] - top2[:, 0]
    ref_draft = O.argmax_lowest(ref_logits)
    n_window = 0
    for i in range(len(got_draft)):
        assert 0 <= got_draft[i] < ref_logits.shape[1], f"{where} row {i}: token {got_draft[i]}"
        if gap[i] >= TIE_WINDOW:
            assert got_draft[i] == ref_draft[i], f"{where} row {i}: draft {got_draft[i]} != {ref_draft[i]}"
        else:
            n_window += 1
            assert ref_logits[i, got_draft[i]] >= top2[i, 1] - TIE_WINDOW - tol, f"{where} row {i}"
    return n_window


# z, the LM head's operand, is stored in bf16 by both sides: within one bf16 step
# (at the value or at the tensor's RMS) of the oracle, and mostly bit-identical.
# The rest are rounding flips: z = bf16(RMSNorm(y)) where the kernel's y differs
# from the oracle's by fp32 accumulation and by the flips of the bf16 tensors
# before it (A, q/k/v, the attention output).  A relative difference e of y
# flips about e / 2^-9 of the roundings; the post-norm GPT-OSS step at B=64
# (e ~ 2e-4) measured 0.87-0.96 bit-identical per request, the B=1 pre-norm
# step 0.992.
Z_MIN_EXACT = 0.8


def check_z(dtype, got, ref, where=""):
    if dtype == "bf16":
        ex = check_close_bf16(got, ref, f"{where} z", max_ulps=1, min_exact=Z_MIN_EXACT)
        print(f"[parity] {where}: z {ex:.4f} bit-identical")
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5, err_msg=f"{where} z")


def bf16_ulps(a, b):
    """|a - b| in units of the bf16 spacing at max(|a|, |b|) (a, b fp64 arrays)."""
    m = np.maximum(np.abs(a), np.abs(b))
    _, e = np.frexp(np.where(m == 0, 1.0, m))
    ulp = np.ldexp(1.0, e - 8)
    return np.abs(a - b) / ulp


def check_close_bf16(got, ref, what, max_ulps=1, min_exact=0.99):
    """Stored bf16 values: nearly all bit-equal, the rest within max_ulps of the
    bf16 spacing at the larger of the value and the tensor's RMS (a value that
    comes out of a cancellation carries the error of the terms it came from)."""
    scale = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    u = bf16_ulps(got, ref)
    u_scale = np.abs(got - ref) / (2.0 ** -8 * max(scale, 1e-30))
    err = np.minimum(u, u_scale)
    exact = float(np.mean(got == ref))
    assert err.max() <= max_ulps, f"{what}: max {err.max():.3g} ulps"
    assert exact >= min_exact, f"{what}: only {exact:.4f} bit-exact"
    return exact
