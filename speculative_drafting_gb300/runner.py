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

    def status(self, clear=True):
        return self.drafter.read_status(self.ws, clear=clear)
