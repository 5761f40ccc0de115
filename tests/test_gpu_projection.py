"""The step's projection kernel (tcgen05 GEMM for bf16, SIMT for fp32) alone,
against a float64 matrix product of the same bf16 operands."""

import numpy as np
import pytest

from oracle import pe_oracle as O
from parity import cuda_or_skip, f64, host, setup
from speculative_drafting_gb300 import runner

pytestmark = pytest.mark.gpu

PROJ = {"fc": 0, "qkv": 1, "o": 2, "swiglu": 3, "down": 4, "lm": 5}


def _shape(dm, which):
    H = dm.n_heads * dm.head_dim
    return {"fc": (dm.d, 4 * dm.d, "w_fc"), "qkv": (dm.qkv_rows, dm.d, "w_qkv"), "o": (dm.d, H, "w_o"),
            "swiglu": (dm.inter, dm.d, "w_gate"), "down": (dm.d, dm.inter, "w_down"),
            "lm": (dm.vocab, dm.d, "w_lm")}[which]


@pytest.mark.parametrize("name", ["small_prenorm", "small_postnorm_hd128", "tiny_fp32"])
@pytest.mark.parametrize("which", list(PROJ))
@pytest.mark.parametrize("n", [1, 7, 16, 100, 300])
def test_projection_matches_matmul(name, which, n):
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup(name, want_logits=False, kv=False)
    dm = wl.dims
    M, Kd, wname = _shape(dm, which)
    g = np.random.default_rng(n * 31 + PROJ[which])
    X = g.standard_normal((n, Kd)).astype(np.float32)
    if dm.dtype == "bf16":
        from speculative_drafting_gb300.workloads import f32_to_bf16_bits
        Xh = f32_to_bf16_bits(X)
    else:
        Xh = X
    Xd = runner.to_device(Xh, dm.dtype)
    out_dt = (torch.bfloat16 if dm.dtype == "bf16" else torch.float32) if which == "swiglu" else torch.float32
    out = torch.full((n, M), float("nan"), dtype=out_dt, device="cuda")
    ws = r.drafter.test_projection(PROJ[which], Xd, n, out)
    torch.cuda.synchronize()
    st, _ = r.drafter.read_status(ws)
    assert st == 0, hex(st)
    x64 = f64(Xh, dm.dtype)
    if which == "swiglu":
        ref = O.bf16_round(O.silu(O.linear(x64, f64(w["w_gate"], dm.dtype))) *
                           O.linear(x64, f64(w["w_up"], dm.dtype))) if dm.dtype == "bf16" else \
            O.silu(O.linear(x64, f64(w["w_gate"], dm.dtype))) * O.linear(x64, f64(w["w_up"], dm.dtype))
        got = f64(host(out), dm.dtype)
        tol = 2 ** -7 * np.abs(ref) + 1e-6 if dm.dtype == "bf16" else 1e-5 * (1 + np.abs(ref))
    else:
        ref = O.linear(x64, f64(w[wname], dm.dtype))
        got = host(out).astype(np.float64)
        # fp32 accumulation of K products of magnitude ~|x||w|
        tol = 1e-5 * np.sqrt(Kd) * 0.02 * 4 + 1e-5 * np.abs(ref)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"max err {err.max():.3g}"


# PE_PROJ_PERSISTENT / PE_PROJ_PAIR (pe_testing.h)
PERSISTENT, PAIR = 0x100, 0x200


@pytest.mark.parametrize("name", ["small_prenorm", "small_postnorm_hd128"])
@pytest.mark.parametrize("which", list(PROJ))
@pytest.mark.parametrize("n", [100, 256, 300, 513])
@pytest.mark.parametrize("flags", [PERSISTENT, PAIR, PERSISTENT | PAIR])
def test_projection_schedules_and_pairs(name, which, n, flags):
    """The persistent schedule (several CTAs per SM for narrow token tiles, the
    ragged last round split over K) and bf16-pair operands, against the float64
    product of the operand the kernel was given."""
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup(name, want_logits=False, kv=False)
    dm = wl.dims
    M, Kd, wname = _shape(dm, which)
    from speculative_drafting_gb300.workloads import f32_to_bf16_bits
    g = np.random.default_rng(n * 37 + PROJ[which] + flags)
    X = g.standard_normal((n, Kd)).astype(np.float32)
    hi = f32_to_bf16_bits(X)
    x64 = f64(hi, "bf16")
    Xh = hi
    if flags & PAIR:
        lo = f32_to_bf16_bits((X.astype(np.float64) - x64).astype(np.float32))
        x64 = x64 + f64(lo, "bf16")
        Xh = np.concatenate([hi, lo], axis=0)
    Xd = runner.to_device(Xh, "bf16")
    out_dt = torch.bfloat16 if which == "swiglu" else torch.float32
    out = torch.full((n, M), float("nan"), dtype=out_dt, device="cuda")
    ws = r.drafter.test_projection(PROJ[which] | flags, Xd, n, out)
    torch.cuda.synchronize()
    st, _ = r.drafter.read_status(ws)
    assert st == 0, hex(st)
    if which == "swiglu":
        ref = O.bf16_round(O.silu(O.linear(x64, f64(w["w_gate"], "bf16"))) *
                           O.linear(x64, f64(w["w_up"], "bf16")))
        got = f64(host(out), "bf16")
        tol = 2 ** -7 * np.abs(ref) + 1e-6
    else:
        ref = O.linear(x64, f64(w[wname], "bf16"))
        got = host(out).astype(np.float64)
        tol = 1e-5 * np.sqrt(Kd) * 0.02 * 4 + 1e-5 * np.abs(ref)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"max err {err.max():.3g}"


PARTIAL = 0x400  # PE_PROJ_PARTIAL (pe_testing.h)


@pytest.mark.parametrize("name", ["small_prenorm", "small_postnorm_hd128", "tiny_fp32"])
@pytest.mark.parametrize("which", ["fc", "qkv", "o", "down", "lm"])
@pytest.mark.parametrize("n", [1, 7, 16, 100, 300])
@pytest.mark.parametrize("pair", [False, True])
def test_projection_partial_sums(name, which, n, pair):
    """K splits that store their own partial sums: the tiles add up to the
    float64 product (tiles past the split count stay zero)."""
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup(name, want_logits=False, kv=False)
    dm = wl.dims
    if pair and dm.dtype != "bf16":
        pytest.skip("pair operands are bf16 only")
    M, Kd, wname = _shape(dm, which)
    g = np.random.default_rng(n * 41 + PROJ[which] + 7 * pair)
    X = g.standard_normal((n, Kd)).astype(np.float32)
    if dm.dtype == "bf16":
        from speculative_drafting_gb300.workloads import f32_to_bf16_bits
        hi = f32_to_bf16_bits(X)
        x64 = f64(hi, "bf16")
        Xh = hi
        if pair:
            lo = f32_to_bf16_bits((X.astype(np.float64) - x64).astype(np.float32))
            x64 = x64 + f64(lo, "bf16")
            Xh = np.concatenate([hi, lo], axis=0)
    else:
        Xh, x64 = X, X.astype(np.float64)
    Xd = runner.to_device(Xh, dm.dtype)
    out = torch.zeros((16, n, M), dtype=torch.float32, device="cuda")
    ws = r.drafter.test_projection(PROJ[which] | PARTIAL | (PAIR if pair else 0), Xd, n, out)
    torch.cuda.synchronize()
    st, _ = r.drafter.read_status(ws)
    assert st == 0, hex(st)
    ref = O.linear(x64, f64(w[wname], dm.dtype))
    parts = host(out).astype(np.float64)
    got = parts.sum(axis=0)
    tol = 1e-5 * np.sqrt(Kd) * 0.02 * 4 + 1e-5 * np.abs(ref)
    assert np.all(np.isfinite(parts))
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"max err {err.max():.3g}"


ARGMAX = 0x2000  # pe_testing.h


@pytest.mark.parametrize("name", ["small_prenorm", "small_postnorm_hd128"])
@pytest.mark.parametrize("n", [1, 7, 100, 300, 448, 513])
def test_lm_head_argmax(name, n):
    """The LM head with its argmax epilogue: the logits match the float64
    product, each row's index is the first maximum of the logits the kernel
    produced, and it is the float64 argmax wherever the top two logits are apart
    by more than the accumulation error."""
    torch = cuda_or_skip()
    wl, b, w, kc, vc, r = setup(name, want_logits=False, kv=False)
    M, Kd, wname = _shape(wl.dims, "lm")
    from speculative_drafting_gb300.workloads import f32_to_bf16_bits
    g = np.random.default_rng(n * 47)
    hi = f32_to_bf16_bits(g.standard_normal((n, Kd)).astype(np.float32))
    Xd = runner.to_device(hi, "bf16")
    out = torch.full((n, M), float("nan"), dtype=torch.float32, device="cuda")
    ws = r.drafter.test_projection(PROJ["lm"] | ARGMAX, Xd, n, out)
    torch.cuda.synchronize()
    st, _ = r.drafter.read_status(ws)
    assert st == 0, hex(st)
    off = 256 + (n * 8 + 255) // 256 * 256  # PE_PROJ_ARGMAX_TOKENS_OFFSET(n)
    tok = host(ws[off:off + 4 * n]).view(np.int32)
    logits = host(out).astype(np.float64)
    ref = O.linear(f64(hi, "bf16"), f64(w[wname], "bf16"))
    tol = 1e-5 * np.sqrt(Kd) * 0.02 * 4 + 1e-5 * np.abs(ref)
    assert np.all(np.abs(logits - ref) <= tol)
    np.testing.assert_array_equal(tok, logits.argmax(axis=1))
    top2 = np.sort(ref, axis=1)[:, -2:]
    clear = top2[:, 1] - top2[:, 0] > 2 * tol.max()
    np.testing.assert_array_equal(tok[clear], ref.argmax(axis=1)[clear])


def test_gemms_read_the_callers_packed_copy():
    """A bf16 handle's GEMMs read the caller's tile-packed buffer: packing the
    negated matrices into it (pe_pack_weights, no new handle) negates every
    projection, and writing the row-major matrices afterwards changes nothing."""
    torch = cuda_or_skip()
    import ctypes

    from speculative_drafting_gb300 import binding
    wl, b, w, kc, vc, r = setup("small_prenorm", want_logits=False, kv=False)
    dm = wl.dims
    n = 40
    from speculative_drafting_gb300.workloads import f32_to_bf16_bits
    X = runner.to_device(f32_to_bf16_bits(
        np.random.default_rng(3).standard_normal((n, 4 * dm.d)).astype(np.float32)), "bf16")
    out = torch.empty(n, dm.d, dtype=torch.float32, device="cuda")
    r.drafter.test_projection(PROJ["fc"], X, n, out)
    torch.cuda.synchronize()
    first = out.clone()
    neg = {k: -t for k, t in r.w.items() if k.startswith("w_")}
    cw = binding.PeWeights.from_buffer_copy(r.drafter.cw)
    for k, t in neg.items():
        setattr(cw, k, t.data_ptr())
    r.drafter.pack(weights=cw)
    torch.cuda.synchronize()
    r.drafter.test_projection(PROJ["fc"], X, n, out)
    torch.cuda.synchronize()
    assert torch.equal(out, -first)
    # the row-major matrices are not what the kernels read
    r.w["w_fc"].zero_()
    r.drafter.test_projection(PROJ["fc"], X, n, out)
    torch.cuda.synchronize()
    assert torch.equal(out, -first)
