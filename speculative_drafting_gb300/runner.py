"""Device-side setup of one step workload and the three C-ABI calls in order.

Uploads host arrays (from ``workloads``) to the GPU, allocates the caller-owned
buffers the C-ABI expects and runs pe_prepare_inputs -> pe_draft_step ->
pe_argmax on a stream.  No arithmetic of the step happens here.
"""

from __future__ import annotations

import numpy as np

from . import binding


def to_device(arr, dtype: str, device="cuda"):
    """Host array -> torch tensor on device (bf16 bit patterns become bfloat16)."""
    import torch

    if dtype == "bf16" and arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def to_host_bits(t):
    """torch tensor -> numpy (bfloat16 as uint16 bit patterns)."""
    import torch

    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


class StepRunner:
    """One batch of one workload, resident on the device."""

    def __init__(self, wl, batch: dict, weights: dict, k_cache=None, v_cache=None, device="cuda",
                 max_batch=None, max_rows_in=None, want_G=False, want_E=False, want_logits=False):
        import torch

        self.wl, self.dims = wl, wl.dims
        dt = wl.dims.dtype
        self.device = device
        self.B, self.T_in = int(batch["B"]), int(batch["T_in"])
        self.num_blocks = int(batch["num_blocks"])
        K = wl.dims.K
        self.T_out = self.T_in + self.B * (K - 1)
        self.w = {k: to_device(v, dt, device) for k, v in weights.items() if k != "layers"}
        if weights.get("layers"):
            self.w["layers"] = [{k: to_device(v, dt, device) for k, v in lw.items()}
                                for lw in weights["layers"]]
        self.inp = {k: to_device(batch[k], dt, device) for k in
                    ("qsl", "prev_tok", "prev_pos", "accepted", "bonus", "block_table", "H_tgt")}
        self.drafter = binding.Drafter(wl.dims, self.w) if wl.has_drafter else None
        if self.drafter is None:
            # metadata + preparation only: the layer's weights are left out (NULL)
            self.drafter = binding.Drafter(wl.dims, self.w)
        self.meta = binding.Meta(self.B, self.T_in, K, device)
        edt = torch.bfloat16 if dt == "bf16" else torch.float32
        d = wl.dims.d
        self.A = torch.empty(self.T_out, 4 * d, dtype=edt, device=device)
        self.G = torch.empty(self.T_out, 3, d, dtype=edt, device=device) if want_G else None
        self.E = torch.empty(self.T_out, d, dtype=edt, device=device) if want_E else None
        self.z = torch.empty(self.B * K, d, dtype=edt, device=device)
        self.draft = torch.empty(self.B * K, dtype=torch.int32, device=device)
        self.logits = (torch.empty(self.B * K, wl.dims.vocab, dtype=torch.float32, device=device)
                       if want_logits else None)
        self.k_cache = to_device(k_cache, dt, device) if k_cache is not None else None
        self.v_cache = to_device(v_cache, dt, device) if v_cache is not None else None
        mb = self.inp["block_table"].shape[1]
        self.ws = self.drafter.workspace(max_batch or self.B, max_rows_in or self.T_in, mb, device)

    def prepare(self, stream=None, A=True):
        i = self.inp
        self.drafter.prepare_inputs(self.B, self.T_in, i["qsl"], i["prev_tok"], i["prev_pos"],
                                    i["accepted"], i["bonus"], i["block_table"], self.num_blocks,
                                    i["H_tgt"], self.meta, self.ws, G=self.G, E=self.E,
                                    A=self.A if A else None, stream=stream)

    def step(self, stream=None):
        self.drafter.draft_step(self.B, self.T_in, self.meta, self.A, self.inp["block_table"],
                                self.num_blocks, self.k_cache, self.v_cache, self.z, self.ws,
                                stream=stream)

    def argmax(self, stream=None):
        self.drafter.argmax(self.z, self.B * self.dims.K, self.draft, self.ws, logits=self.logits,
                            stream=stream)

    def run(self, stream=None):
        self.prepare(stream)
        self.step(stream)
        self.argmax(stream)

    def autoregressive(self, draft, ws, logits=None, hidden=None, stream=None):
        """The K-pass autoregressive drafting of the same batch (the baseline):
        draft [B][K] int32, ws from Drafter.autoregressive_workspace; optional
        logits [B][K][V] and per-pass hidden states [B][K][d] (fp32)."""
        i = self.inp
        self.drafter.draft_autoregressive(self.B, self.T_in, i["qsl"], i["prev_tok"], i["prev_pos"],
                                          i["accepted"], i["bonus"], i["block_table"],
                                          self.num_blocks, i["H_tgt"], self.k_cache, self.v_cache,
                                          draft, ws, logits=logits, hidden=hidden, stream=stream)

    def status(self, clear=True):
        return self.drafter.read_status(self.ws, clear=clear)


def cod_capacity(S_max: int, n_depth: int, max_anchors: int):
    """(q_cap, ld) that hold any COD mask of a sequence of at most S_max tokens:
    at most n_depth * anchors rows and S_max + (n_depth - 1) * anchors columns,
    anchors = max_anchors (or S_max without a cap)."""
    anchors = min(max_anchors, S_max) if max_anchors > 0 else S_max
    q_cap = max(1, n_depth * anchors)
    ld = max(16, (S_max + (n_depth - 1) * anchors + 15) // 16 * 16)
    return q_cap, ld


class CodRunner:
    """One COD batch resident on the device: the index call, then the mask call."""

    def __init__(self, batch: dict, device="cuda", q_cap=None, ld=None, guard=0):
        import torch

        self.B, self.S, self.D = int(batch["B"]), int(batch["S_max"]), int(batch["n_depth"])
        self.retain, self.max_anchors = float(batch["retain"]), int(batch["max_anchors"])
        self.inp = {k: torch.from_numpy(np.ascontiguousarray(batch[k])).to(device)
                    for k in ("seq_len", "loss_mask", "u_anchor", "u_keep")}
        cq, cl = cod_capacity(self.S, self.D, self.max_anchors)
        self.q_cap = cq if q_cap is None else int(q_cap)
        self.ld = cl if ld is None else int(ld)
        self.mask_stride = self.q_cap * self.ld
        self.idx = torch.full((self.B, self.D, self.S), -1, dtype=torch.int32, device=device)
        self.counts = torch.full((self.B, self.D), -1, dtype=torch.int32, device=device)
        # `guard` extra bytes after the last sequence's block (tests check them)
        self.mask = torch.zeros(self.B * self.mask_stride + guard, dtype=torch.uint8, device=device)
        self.ws = binding.cod_workspace(self.B, self.S, self.D, device)

    def sample(self, stream=None):
        i = self.inp
        binding.cod_sample_indices(self.B, self.S, i["seq_len"], i["loss_mask"], self.D, self.retain,
                                   self.max_anchors, i["u_anchor"], i["u_keep"] if self.D > 1 else None,
                                   self.idx, self.counts, self.ws, stream=stream)

    def build_mask(self, stream=None):
        binding.cod_mask(self.B, self.S, self.inp["seq_len"], self.D, self.idx, self.counts, self.mask,
                         self.q_cap, self.ld, self.mask_stride, self.ws, stream=stream)

    def run(self, stream=None):
        self.sample(stream)
        self.build_mask(stream)

    def status(self, clear=True):
        return binding.read_status_ws(self.ws, clear=clear)

    def mask_of(self, b):
        """Sequence b's mask block as a [q_cap][ld] uint8 view."""
        return self.mask[b * self.mask_stride:(b + 1) * self.mask_stride].view(self.q_cap, self.ld)
