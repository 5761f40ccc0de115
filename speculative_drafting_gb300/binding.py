"""ctypes binding of ``libpe.so`` (include/pe.h), with the same call names.

Argument marshalling only: every step of the draft path runs in the library's
CUDA kernels.  PyTorch supplies device memory (tensor data pointers) and
streams; the helpers below allocate the caller-owned buffers the C-ABI expects.
There is no fallback: loading fails loudly when the library is missing.
"""

from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

PE_OK = 0
PE_ERR_ARG = 1
PE_ERR_UNSUPPORTED = 2
PE_ERR_CUDA = 3
PE_ERR_DEVICE_INPUT = 4
PE_ERR_TIMEOUT = 5
PE_ST_ACCEPTED_RANGE = 0x1
PE_ST_BLOCK_RANGE = 0x2
PE_ST_TOKEN_RANGE = 0x4
PE_ST_ROWS_RANGE = 0x8
PE_ST_TIMEOUT = 0x10
PE_ST_CAPACITY = 0x20
PE_COD_MAX_DEPTH = 16
PE_DTYPE_F32 = 0
PE_DTYPE_BF16 = 1

HEADER = os.path.join(_build.ROOT, "include", "pe.h")
TESTING_HEADER = os.path.join(_build.ROOT, "include", "pe_testing.h")


class PeError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"{what}: {status_string(code)} (code {code})")
        self.code = code


class PeDims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("n_streams", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("K", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("mask_id", ctypes.c_int32), ("post_norm", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("n_layers", ctypes.c_int32)]


WEIGHT_FIELDS = ["emb", "emb_mask", "h_shared", "gamma_stream", "w_fc", "gamma_in", "w_qkv", "w_o",
                 "gamma_post", "w_gate", "w_up", "w_down", "gamma_final", "w_lm", "attn_sink"]
LAYER_FIELDS = ["gamma_in", "w_qkv", "w_o", "gamma_post", "w_gate", "w_up", "w_down", "gamma_final",
                "attn_sink"]


class PeLayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_FIELDS]


class PeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS] + \
        [("more_layers", ctypes.POINTER(PeLayerWeights)), ("packed", ctypes.c_void_p),
         ("packed_bytes", ctypes.c_size_t)]


META_FIELDS = ["out_qsl", "tok", "pos", "is_rejected", "is_masked", "hidden_src", "slot",
               "valid_qsl", "valid_rows", "n_valid", "sample_idx", "seq_len"]


class PeMeta(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in META_FIELDS]


_lib = None
_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load libpe.so (built by ``build.build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run speculative_drafting_gb300.build.build()")
    lib = ctypes.CDLL(path)
    lib.pe_create.argtypes = [ctypes.POINTER(PeDims), ctypes.POINTER(PeWeights), ctypes.POINTER(_vp)]
    lib.pe_create.restype = _i32
    lib.pe_destroy.argtypes = [_vp]
    lib.pe_destroy.restype = None
    lib.pe_packed_weights_bytes.argtypes = [ctypes.POINTER(PeDims)]
    lib.pe_packed_weights_bytes.restype = _sz
    lib.pe_pack_weights.argtypes = [ctypes.POINTER(PeDims), ctypes.POINTER(PeWeights), _vp, _sz, _vp]
    lib.pe_pack_weights.restype = _i32
    lib.pe_workspace_bytes.argtypes = [_vp, _i32, _i32, _i32]
    lib.pe_workspace_bytes.restype = _sz
    lib.pe_prepare_inputs.argtypes = [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp,
                                      ctypes.POINTER(PeMeta), _vp, _vp, _vp, _vp, _sz, _vp]
    lib.pe_prepare_inputs.restype = _i32
    lib.pe_draft_step.argtypes = [_vp, _i32, _i32, ctypes.POINTER(PeMeta), _vp, _vp, _i32, _i32, _vp,
                                  _vp, _vp, _vp, _sz, _vp]
    lib.pe_draft_step.restype = _i32
    lib.pe_argmax.argtypes = [_vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp]
    lib.pe_argmax.restype = _i32
    lib.pe_read_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint32), _i32, _vp]
    lib.pe_read_status.restype = _i32
    lib.pe_status_string.argtypes = [_i32]
    lib.pe_status_string.restype = ctypes.c_char_p
    lib.pe_autoregressive_workspace_bytes.argtypes = [_vp, _i32, _i32, _i32]
    lib.pe_autoregressive_workspace_bytes.restype = _sz
    lib.pe_draft_autoregressive.argtypes = [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                            _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
    lib.pe_draft_autoregressive.restype = _i32
    lib.pe_argmax_noalloc.argtypes = [_vp, _vp, _i32, _vp, _vp, _vp]
    lib.pe_argmax_noalloc.restype = _i32
    lib.pe_test_projection_workspace.argtypes = [_vp, _i32, _i32]
    lib.pe_test_projection_workspace.restype = _sz
    lib.pe_test_projection.argtypes = [_vp, _i32, _vp, _i32, _vp, _vp, _sz, _vp]
    lib.pe_test_projection.restype = _i32
    lib.pe_test_bounded_wait.argtypes = [_vp, _sz, _vp]
    lib.pe_test_bounded_wait.restype = _i32
    lib.pe_verify_workspace_bytes.argtypes = [_i32, _i32]
    lib.pe_verify_workspace_bytes.restype = _sz
    lib.pe_verify_greedy.argtypes = [_i32, _i32, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp,
                                     _sz, _vp]
    lib.pe_verify_greedy.restype = _i32
    lib.pe_cod_workspace_bytes.argtypes = [_i32, _i32, _i32]
    lib.pe_cod_workspace_bytes.restype = _sz
    lib.pe_cod_sample_indices.argtypes = [_i32, _i32, _vp, _vp, _i32, ctypes.c_float, _i32, _vp,
                                          _vp, _vp, _vp, _vp, _sz, _vp]
    lib.pe_cod_sample_indices.restype = _i32
    lib.pe_cod_mask.argtypes = [_i32, _i32, _vp, _i32, _vp, _vp, _vp, ctypes.c_int64,
                                ctypes.c_int64, ctypes.c_int64, _vp, _sz, _vp]
    lib.pe_cod_mask.restype = _i32
    _lib = lib
    return lib


def declared_functions(header: str = HEADER):
    """Names of the functions include/pe.h declares."""
    src = open(header).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pe_[a-z_]+)\s*\(", src)))


def status_string(code: int) -> str:
    return load().pe_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc, what):
    if rc != PE_OK:
        raise PeError(rc, what)


def make_dims(dm) -> PeDims:
    """PeDims from any object with the Dims attributes (workloads.Dims)."""
    return PeDims(d=dm.d, n_streams=3, n_heads=dm.n_heads, n_kv_heads=dm.n_kv_heads,
                  head_dim=dm.head_dim, inter=dm.inter, vocab=dm.vocab, K=dm.K,
                  block_size=dm.block_size, mask_id=dm.mask_id, post_norm=int(bool(dm.post_norm)),
                  dtype=PE_DTYPE_BF16 if dm.dtype == "bf16" else PE_DTYPE_F32,
                  eps=dm.eps, rope_theta=dm.rope_theta, n_layers=getattr(dm, "n_layers", 1))


class Meta:
    """Caller-owned metadata buffers for a batch of B requests and T_in rows."""

    def __init__(self, B: int, T_in: int, K: int, device="cuda"):
        import torch

        T_out = T_in + B * (K - 1)
        i32, i64, u8 = torch.int32, torch.int64, torch.uint8
        self.B, self.T_in, self.T_out, self.K = B, T_in, T_out, K
        self.t = {
            "out_qsl": torch.empty(B + 1, dtype=i32, device=device),
            "tok": torch.empty(T_out, dtype=i32, device=device),
            "pos": torch.empty(T_out, dtype=i64, device=device),
            "is_rejected": torch.empty(T_out, dtype=u8, device=device),
            "is_masked": torch.empty(T_out, dtype=u8, device=device),
            "hidden_src": torch.empty(T_out, dtype=i32, device=device),
            "slot": torch.empty(T_out, dtype=i64, device=device),
            "valid_qsl": torch.empty(B + 1, dtype=i32, device=device),
            "valid_rows": torch.empty(T_out, dtype=i32, device=device),
            "n_valid": torch.empty(1, dtype=i32, device=device),
            "sample_idx": torch.empty(B * K, dtype=i32, device=device),
            "seq_len": torch.empty(B, dtype=i32, device=device),
        }
        self.c = PeMeta(**{k: v.data_ptr() for k, v in self.t.items()})

    def __getitem__(self, k):
        return self.t[k]


class Drafter:
    """One drafter handle: ``pe_create`` over device weight tensors (borrowed).
    A bf16 drafter's projection matrices are first tile-packed (pe_pack_weights)
    into a buffer this object owns and the handle borrows."""

    def __init__(self, dims, weights: dict, stream=None):
        import torch

        self.lib = load()
        self.dims = dims
        self.weights = weights  # keep the tensors alive for the handle's lifetime
        cw = PeWeights(**{k: (weights[k].data_ptr() if weights.get(k) is not None else None)
                          for k in WEIGHT_FIELDS})
        more = weights.get("layers") or []
        if more:
            # host array of the later layers' device pointers (read by pe_create)
            arr = (PeLayerWeights * len(more))()
            for i, lw in enumerate(more):
                for k in LAYER_FIELDS:
                    setattr(arr[i], k, lw[k].data_ptr() if lw.get(k) is not None else None)
            cw.more_layers = arr
        self.cw = cw
        h = ctypes.c_void_p()
        self.cdims = make_dims(dims)
        self.packed = None
        n = int(self.lib.pe_packed_weights_bytes(ctypes.byref(self.cdims)))
        if n and weights.get("w_fc") is not None:
            dev = weights["w_fc"].device
            self.packed = torch.empty(n, dtype=torch.uint8, device=dev)
            self.pack(stream)
            # the handle may be used on any stream: let the packing finish first
            (stream or torch.cuda.current_stream()).synchronize()
            cw.packed = self.packed.data_ptr()
            cw.packed_bytes = n
        _check(self.lib.pe_create(ctypes.byref(self.cdims), ctypes.byref(cw), ctypes.byref(h)), "pe_create")
        self.h = h

    def pack(self, stream=None, weights=None):
        """pe_pack_weights into this drafter's packed buffer (from `weights`, a
        PeWeights, when given: the tests pack other matrices into it)."""
        _check(self.lib.pe_pack_weights(ctypes.byref(self.cdims), ctypes.byref(weights or self.cw),
                                        _ptr(self.packed), self.packed.numel(), _stream(stream)),
               "pe_pack_weights")

    def close(self):
        if self.h:
            self.lib.pe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_bytes(self, max_batch: int, max_rows_in: int, max_blocks: int) -> int:
        return int(self.lib.pe_workspace_bytes(self.h, max_batch, max_rows_in, max_blocks))

    def workspace(self, max_batch: int, max_rows_in: int, max_blocks: int, device="cuda"):
        import torch

        n = self.workspace_bytes(max_batch, max_rows_in, max_blocks)
        if n == 0:
            raise PeError(PE_ERR_ARG, "pe_workspace_bytes")
        return torch.zeros(n, dtype=torch.uint8, device=device)

    def prepare_inputs(self, B, T_in, qsl, prev_tok, prev_pos, accepted, bonus, block_table,
                       num_blocks, H_tgt, meta: Meta, ws, G=None, E=None, A=None, stream=None):
        rc = self.lib.pe_prepare_inputs(
            self.h, B, T_in, _ptr(qsl), _ptr(prev_tok), _ptr(prev_pos), _ptr(accepted), _ptr(bonus),
            _ptr(block_table), block_table.shape[1], num_blocks, _ptr(H_tgt), ctypes.byref(meta.c),
            _ptr(G), _ptr(E), _ptr(A), _ptr(ws), ws.numel(), _stream(stream))
        _check(rc, "pe_prepare_inputs")

    def draft_step(self, B, T_in, meta: Meta, A, block_table, num_blocks, k_cache, v_cache, z_out,
                   ws, stream=None):
        rc = self.lib.pe_draft_step(self.h, B, T_in, ctypes.byref(meta.c), _ptr(A), _ptr(block_table),
                                    block_table.shape[1], num_blocks, _ptr(k_cache), _ptr(v_cache),
                                    _ptr(z_out), _ptr(ws), ws.numel(), _stream(stream))
        _check(rc, "pe_draft_step")

    def argmax(self, z, n_rows, draft_tokens, ws, logits=None, stream=None):
        rc = self.lib.pe_argmax(self.h, _ptr(z), n_rows, _ptr(draft_tokens), _ptr(logits), _ptr(ws),
                                ws.numel(), _stream(stream))
        _check(rc, "pe_argmax")

    def autoregressive_workspace(self, max_batch: int, max_rows_in: int, max_blocks: int,
                                 device="cuda"):
        import torch

        n = int(self.lib.pe_autoregressive_workspace_bytes(self.h, max_batch, max_rows_in,
                                                           max_blocks))
        if n == 0:
            raise PeError(PE_ERR_ARG, "pe_autoregressive_workspace_bytes")
        return torch.zeros(n, dtype=torch.uint8, device=device)

    def draft_autoregressive(self, B, T_in, qsl, prev_tok, prev_pos, accepted, bonus, block_table,
                             num_blocks, H_tgt, k_cache, v_cache, draft_tokens, ws, logits=None,
                             hidden=None, stream=None):
        """pe_draft_autoregressive: K sequential one-token passes (the baseline)."""
        rc = self.lib.pe_draft_autoregressive(
            self.h, B, T_in, _ptr(qsl), _ptr(prev_tok), _ptr(prev_pos), _ptr(accepted), _ptr(bonus),
            _ptr(block_table), block_table.shape[1], num_blocks, _ptr(H_tgt), _ptr(k_cache),
            _ptr(v_cache), _ptr(draft_tokens), _ptr(logits), _ptr(hidden), _ptr(ws), ws.numel(),
            _stream(stream))
        _check(rc, "pe_draft_autoregressive")

    def argmax_noalloc(self, z, n_rows, draft_tokens, logits=None, stream=None):
        """pe_argmax without a workspace (its scratch is a static device array)."""
        rc = self.lib.pe_argmax_noalloc(self.h, _ptr(z), n_rows, _ptr(draft_tokens), _ptr(logits),
                                        _stream(stream))
        _check(rc, "pe_argmax_noalloc")

    def test_projection(self, which, X, n_rows, out, stream=None):
        """One drafter projection through the step's GEMM kernel (pe_testing.h)."""
        import torch

        n = int(self.lib.pe_test_projection_workspace(self.h, which, n_rows))
        if n == 0:
            raise PeError(PE_ERR_ARG, "pe_test_projection_workspace")
        ws = torch.zeros(n, dtype=torch.uint8, device=X.device)
        rc = self.lib.pe_test_projection(self.h, which, _ptr(X), n_rows, _ptr(out), _ptr(ws), n,
                                         _stream(stream))
        _check(rc, "pe_test_projection")
        return ws

    def read_status(self, ws, clear=True, stream=None):
        v = ctypes.c_uint32(0)
        rc = self.lib.pe_read_status(self.h, _ptr(ws), ctypes.byref(v), int(clear), _stream(stream))
        if rc not in (PE_OK, PE_ERR_DEVICE_INPUT, PE_ERR_TIMEOUT):
            raise PeError(rc, "pe_read_status")
        return int(v.value), rc


# ----------------------------------------------------------------------------- verification


def verify_workspace_bytes(max_rows_in: int, vocab: int) -> int:
    n = int(load().pe_verify_workspace_bytes(int(max_rows_in), int(vocab)))
    if n == 0:
        raise PeError(PE_ERR_ARG, "pe_verify_workspace_bytes")
    return n


def verify_workspace(max_rows_in: int, vocab: int, device="cuda"):
    """A device workspace for pe_verify_greedy (torch allocates it 256-byte aligned)."""
    import torch

    return torch.zeros(verify_workspace_bytes(max_rows_in, vocab), dtype=torch.uint8,
                       device=device)


def verify_greedy(B, T_in, qsl, tok, logits, vocab, dtype, target_tok, accepted, bonus, ws,
                  stream=None):
    """pe_verify_greedy on device tensors; dtype is PE_DTYPE_F32 or PE_DTYPE_BF16."""
    rc = load().pe_verify_greedy(int(B), int(T_in), _ptr(qsl), _ptr(tok), _ptr(logits),
                                 int(vocab), int(dtype), _ptr(target_tok), _ptr(accepted),
                                 _ptr(bonus), _ptr(ws), int(ws.numel()), _stream(stream))
    _check(rc, "pe_verify_greedy")


def read_status_ws(ws, clear=True, stream=None):
    """pe_read_status without a handle (the verification call has none)."""
    v = ctypes.c_uint32(0)
    rc = load().pe_read_status(None, _ptr(ws), ctypes.byref(v), int(clear), _stream(stream))
    if rc not in (PE_OK, PE_ERR_DEVICE_INPUT, PE_ERR_TIMEOUT):
        raise PeError(rc, "pe_read_status")
    return int(v.value), rc


# ----------------------------------------------------------------------------- COD training indices


def cod_workspace_bytes(B: int, S_max: int, n_depth: int) -> int:
    n = int(load().pe_cod_workspace_bytes(int(B), int(S_max), int(n_depth)))
    if n == 0:
        raise PeError(PE_ERR_ARG, "pe_cod_workspace_bytes")
    return n


def cod_workspace(B: int, S_max: int, n_depth: int, device="cuda"):
    """A device workspace for the two COD calls (torch allocates it 256-byte aligned)."""
    import torch

    return torch.zeros(cod_workspace_bytes(B, S_max, n_depth), dtype=torch.uint8, device=device)


def cod_sample_indices(B, S_max, seq_len, loss_mask, n_depth, retain, max_anchors, u_anchor, u_keep,
                       idx, counts, ws, stream=None):
    """pe_cod_sample_indices on device tensors."""
    rc = load().pe_cod_sample_indices(int(B), int(S_max), _ptr(seq_len), _ptr(loss_mask),
                                      int(n_depth), float(retain), int(max_anchors), _ptr(u_anchor),
                                      _ptr(u_keep), _ptr(idx), _ptr(counts), _ptr(ws),
                                      int(ws.numel()), _stream(stream))
    _check(rc, "pe_cod_sample_indices")


def cod_mask(B, S_max, seq_len, n_depth, idx, counts, mask, q_cap, ld, mask_stride, ws, stream=None):
    """pe_cod_mask on device tensors; mask is a uint8 buffer of B * mask_stride bytes."""
    rc = load().pe_cod_mask(int(B), int(S_max), _ptr(seq_len), int(n_depth), _ptr(idx), _ptr(counts),
                            _ptr(mask), int(q_cap), int(ld), int(mask_stride), _ptr(ws),
                            int(ws.numel()), _stream(stream))
    _check(rc, "pe_cod_mask")
