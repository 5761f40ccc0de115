"""The C-ABI library builds for sm_103a, loads, and exports every function the
headers declare; host-side argument checks answer without touching a GPU."""

import ctypes
import shutil

import pytest

from speculative_drafting_gb300 import binding, build

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not __import__("os").path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="needs nvcc to build libpe.so")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_exports_every_declared_function(lib):
    names = binding.declared_functions(binding.HEADER) + binding.declared_functions(binding.TESTING_HEADER)
    assert {"pe_create", "pe_destroy", "pe_workspace_bytes", "pe_prepare_inputs", "pe_draft_step",
            "pe_argmax", "pe_read_status", "pe_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(0, 7):
        assert isinstance(binding.status_string(code), str)
    assert binding.status_string(0) == "ok"


def test_host_argument_checks(lib):
    h = ctypes.c_void_p()
    w = binding.PeWeights()
    good = binding.PeDims(d=64, n_streams=3, n_heads=4, n_kv_heads=2, head_dim=16, inter=128, vocab=512,
                          K=4, block_size=4, mask_id=0, post_norm=0, dtype=binding.PE_DTYPE_F32,
                          eps=1e-6, rope_theta=1e4)
    # null handle output / null dims / null weights
    assert lib.pe_create(ctypes.byref(good), ctypes.byref(w), None) == binding.PE_ERR_ARG
    assert lib.pe_create(None, ctypes.byref(w), ctypes.byref(h)) == binding.PE_ERR_ARG
    assert lib.pe_create(ctypes.byref(good), ctypes.byref(w), ctypes.byref(h)) == binding.PE_ERR_ARG
    assert not h.value
    # unsupported dims are refused before any device call
    for field, value in (("n_streams", 2), ("d", 60), ("head_dim", 256), ("n_kv_heads", 3), ("K", 0),
                         ("dtype", 7)):
        bad = binding.PeDims.from_buffer_copy(good)
        setattr(bad, field, value)
        assert lib.pe_create(ctypes.byref(bad), ctypes.byref(w), ctypes.byref(h)) == \
            binding.PE_ERR_UNSUPPORTED, field
    bf = binding.PeDims.from_buffer_copy(good)
    bf.dtype = binding.PE_DTYPE_BF16  # bf16 attention needs head_dim 64 or 128
    assert lib.pe_create(ctypes.byref(bf), ctypes.byref(w), ctypes.byref(h)) == binding.PE_ERR_UNSUPPORTED
    assert lib.pe_workspace_bytes(None, 1, 1, 1) == 0
    assert lib.pe_prepare_inputs(None, 1, 1, *([None] * 6), 1, 1, None, None, None, None, None, None,
                                 0, None) == binding.PE_ERR_ARG
    assert lib.pe_argmax(None, None, 1, None, None, None, 0, None) == binding.PE_ERR_ARG


def test_packed_weights_host_checks(lib):
    """The tile-packed weight copy: its size from the dims alone, and a bf16
    handle with a layer refused without it (answered on the host)."""
    gpt = binding.PeDims(d=2880, n_streams=3, n_heads=64, n_kv_heads=8, head_dim=64, inter=7680,
                         vocab=201088, K=7, block_size=16, mask_id=0, post_norm=0,
                         dtype=binding.PE_DTYPE_BF16, eps=1e-6, rope_theta=1e4, n_layers=1)

    def packed(M, K):  # blocks of 128 rows x 64 columns of 2-byte elements, 256-aligned
        b = -(-M // 128) * -(-K // 64) * 128 * 64 * 2
        return -(-b // 256) * 256

    d, H, G, hd, I, V = 2880, 64, 8, 64, 7680, 201088
    one = (packed(d, 4 * d) + packed((H + 2 * G) * hd, d) + packed(d, H * hd) + 2 * packed(I, d)
           + packed(d, I) + packed(V, d))
    assert lib.pe_packed_weights_bytes(ctypes.byref(gpt)) == one
    four = binding.PeDims.from_buffer_copy(gpt)
    four.n_layers = 4
    per_layer = packed((H + 2 * G) * hd, d) + packed(d, H * hd) + 2 * packed(I, d) + packed(d, I)
    assert lib.pe_packed_weights_bytes(ctypes.byref(four)) == one + 3 * per_layer
    f32 = binding.PeDims.from_buffer_copy(gpt)
    f32.dtype = binding.PE_DTYPE_F32
    assert lib.pe_packed_weights_bytes(ctypes.byref(f32)) == 0
    assert lib.pe_packed_weights_bytes(None) == 0
    # fake, never dereferenced device addresses: every case fails on the host
    fake = [ctypes.c_void_p((1 << 30) + 256 * i) for i in range(len(binding.WEIGHT_FIELDS))]
    w = binding.PeWeights(**{k: fake[i] for i, k in enumerate(binding.WEIGHT_FIELDS)})
    w.attn_sink = None
    h = ctypes.c_void_p()
    assert lib.pe_create(ctypes.byref(gpt), ctypes.byref(w), ctypes.byref(h)) == binding.PE_ERR_ARG
    w.packed, w.packed_bytes = ctypes.c_void_p(1 << 40), one - 1          # too small
    assert lib.pe_create(ctypes.byref(gpt), ctypes.byref(w), ctypes.byref(h)) == binding.PE_ERR_ARG
    w.packed, w.packed_bytes = ctypes.c_void_p((1 << 40) + 128), one      # misaligned
    assert lib.pe_create(ctypes.byref(gpt), ctypes.byref(w), ctypes.byref(h)) == binding.PE_ERR_ARG
    assert not h.value
    pack = lib.pe_pack_weights
    assert pack(ctypes.byref(f32), ctypes.byref(w), ctypes.c_void_p(1 << 40), one, None) == \
        binding.PE_ERR_UNSUPPORTED
    assert pack(ctypes.byref(gpt), ctypes.byref(w), None, one, None) == binding.PE_ERR_ARG
    assert pack(ctypes.byref(gpt), ctypes.byref(w), ctypes.c_void_p(1 << 40), one - 1, None) == \
        binding.PE_ERR_ARG
    w.w_lm = None
    assert pack(ctypes.byref(gpt), ctypes.byref(w), ctypes.c_void_p(1 << 40), one, None) == \
        binding.PE_ERR_ARG


def test_verify_host_checks(lib):
    # 256-byte header, then one 8-byte key per (row, 1024-element chunk)
    assert lib.pe_verify_workspace_bytes(512, 201088) == 256 + 512 * 197 * 8
    assert lib.pe_verify_workspace_bytes(-1, 10) == 0
    assert lib.pe_verify_workspace_bytes(1, 0) == 0
    call = lib.pe_verify_greedy
    # an empty batch is a no-op; a bad dtype or null outputs are refused on the host
    assert call(0, 0, *([None] * 3), 10, binding.PE_DTYPE_F32, *([None] * 4), 0, None) == binding.PE_OK
    assert call(1, 1, *([None] * 3), 10, 7, *([None] * 4), 0, None) == binding.PE_ERR_UNSUPPORTED
    assert call(1, 1, *([None] * 3), 10, binding.PE_DTYPE_F32, *([None] * 4), 0, None) == \
        binding.PE_ERR_ARG
    assert call(0, 3, *([None] * 3), 10, binding.PE_DTYPE_F32, *([None] * 4), 0, None) == \
        binding.PE_ERR_ARG
    assert call(-1, 0, *([None] * 3), 10, binding.PE_DTYPE_F32, *([None] * 4), 0, None) == \
        binding.PE_ERR_ARG


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes structs the binding marshals have the header's sizes."""
    gxx = shutil.which("g++") or shutil.which("gcc")
    if gxx is None:
        pytest.skip("needs a host C++ compiler")
    src = tmp_path / "sizes.cc"
    src.write_text('#include <cstdio>\n#include "pe.h"\nint main(){std::printf("%zu %zu %zu %zu",'
                   ' sizeof(pe_dims), sizeof(pe_weights), sizeof(pe_layer_weights), sizeof(pe_meta));}\n')
    exe = tmp_path / "sizes"
    import subprocess

    subprocess.run([gxx, "-x", "c++", "-I", __import__("os").path.dirname(binding.HEADER), str(src),
                    "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert got == [ctypes.sizeof(binding.PeDims), ctypes.sizeof(binding.PeWeights),
                   ctypes.sizeof(binding.PeLayerWeights), ctypes.sizeof(binding.PeMeta)]


def test_cod_host_checks(lib):
    # 256-byte header, then one int32 place per (sequence, depth >= 1, position)
    assert lib.pe_cod_workspace_bytes(16, 8192, 8) == 256 + 16 * 7 * 8192 * 4
    assert lib.pe_cod_workspace_bytes(4, 100, 1) == 256
    for bad in ((-1, 10, 2), (1, -1, 2), (1, 10, 0), (1, 10, binding.PE_COD_MAX_DEPTH + 1)):
        assert lib.pe_cod_workspace_bytes(*bad) == 0
    # fake, never dereferenced addresses: every case fails on the host
    ws, p = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21)
    big = 1 << 30
    sample = lib.pe_cod_sample_indices
    assert sample(1, 10, p, p, 0, 0.5, 0, p, p, p, p, ws, big, None) == binding.PE_ERR_ARG    # D = 0
    assert sample(1, 10, p, p, 17, 0.5, 0, p, p, p, p, ws, big, None) == binding.PE_ERR_ARG   # D > 16
    assert sample(1, 10, p, p, 4, float("nan"), 0, p, p, p, p, ws, big, None) == binding.PE_ERR_ARG
    assert sample(1, 10, p, p, 4, 0.5, -1, p, p, p, p, ws, big, None) == binding.PE_ERR_ARG  # cap < 0
    assert sample(1, 10, p, p, 4, 0.5, 0, p, None, p, p, ws, big, None) == binding.PE_ERR_ARG  # no u_keep
    assert sample(1, 10, p, p, 4, 0.5, 0, p, p, p, p, None, big, None) == binding.PE_ERR_ARG   # no ws
    assert sample(1, 10, p, p, 4, 0.5, 0, p, p, p, p, ctypes.c_void_p((1 << 20) + 16), big, None) == \
        binding.PE_ERR_ARG                                                                     # ws misaligned
    assert sample(2, 10, p, p, 4, 0.5, 0, p, p, p, p, ws, 256, None) == binding.PE_ERR_ARG     # ws too small
    assert sample(70000, 1, p, p, 1, 0.5, 0, p, p, p, p, ws, big, None) == binding.PE_ERR_UNSUPPORTED
    mask = lib.pe_cod_mask
    assert mask(1, 10, p, 4, p, p, p, 8, 15, 1 << 12, ws, big, None) == binding.PE_ERR_ARG     # ld % 16
    assert mask(1, 10, p, 4, p, p, p, 8, 0, 1 << 12, ws, big, None) == binding.PE_ERR_ARG      # ld = 0
    assert mask(1, 10, p, 4, p, p, p, 8, 32, 200, ws, big, None) == binding.PE_ERR_ARG         # stride < q_cap * ld
    assert mask(1, 10, p, 4, p, p, p, 8, 32, 264, ws, big, None) == binding.PE_ERR_ARG         # stride % 16
    assert mask(1, 10, p, 4, p, p, ctypes.c_void_p((1 << 21) + 8), 8, 32, 256, ws, big, None) == \
        binding.PE_ERR_ARG                                                                     # mask misaligned
    assert mask(1, 10, p, 4, p, p, p, 1 << 62, 32, 1 << 12, ws, big, None) == binding.PE_ERR_ARG  # overflow


def test_cod_mask_empty_calls_are_no_ops(lib):
    # B = 0 or q_cap = 0: nothing to write, answered on the host (no device call)
    ws, p = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21)
    assert lib.pe_cod_mask(0, 10, None, 4, None, None, None, 8, 32, 256, ws, 1 << 30, None) == binding.PE_OK
    assert lib.pe_cod_mask(2, 10, p, 4, p, p, p, 0, 32, 0, ws, 1 << 30, None) == binding.PE_OK
