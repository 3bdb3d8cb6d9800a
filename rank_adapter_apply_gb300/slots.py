"""PyTorch-side owner of the device memory and streams a context needs.

PyTorch allocates; the compiled library computes. Nothing here does arithmetic
on activations or weights.
"""
from __future__ import annotations

import torch

from . import binding as B


class LoraSlots:
    """Slot pools for a set of injected layers plus the C context.

    layers: list of (d_in, d_out). dtype: torch.bfloat16 or torch.float32.
    """

    def __init__(self, layers, max_loras, max_lora_rank, max_tokens, dtype=torch.bfloat16,
                 max_layers_per_call=None, device="cuda:0", compute_stream=None,
                 upload_stream=None):
        if not torch.cuda.is_available():
            raise RuntimeError("LoraSlots needs a CUDA device")
        B.load()
        self.device = torch.device(device)
        self.dtype = dtype
        self.cdtype = B.LORA_DTYPE_BF16 if dtype == torch.bfloat16 else B.LORA_DTYPE_F32
        self.layers = list(layers)
        self.S, self.R, self.max_tokens = max_loras, max_lora_rank, max_tokens
        self.max_layers = max_layers_per_call or min(8, len(self.layers))
        self.A = [torch.zeros((max_loras, max_lora_rank, di), dtype=dtype, device=self.device)
                  for di, _ in self.layers]
        self.B = [torch.zeros((max_loras, do, max_lora_rank), dtype=dtype, device=self.device)
                  for _, do in self.layers]
        self.scale = torch.zeros(max_loras, dtype=torch.float32, device=self.device)
        self.rank = torch.zeros(max_loras, dtype=torch.int32, device=self.device)
        nbytes = B.lora_workspace_bytes(max_loras, max_lora_rank, max_tokens, self.max_layers)
        self.ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.ws.data_ptr()) % 256
        self.ws_ptr, self.ws_bytes = self.ws.data_ptr() + off, nbytes
        self.compute = compute_stream or torch.cuda.Stream(device=self.device)
        self.upload = upload_stream or torch.cuda.Stream(device=self.device)
        self.ctx = B.lora_slots_init(
            max_loras, max_lora_rank, max_tokens, self.max_layers, self.cdtype,
            [(di, do, a.data_ptr(), b.data_ptr()) for (di, do), a, b in zip(self.layers, self.A, self.B)],
            self.scale.data_ptr(), self.rank.data_ptr(), self.ws_ptr, self.ws_bytes,
            self.compute.cuda_stream, self.upload.cuda_stream)

    # --- slot table ------------------------------------------------------------
    def load_slot(self, slot, A_host, B_host, rank, alpha):
        """A_host/B_host: per-layer host tensors [rank, d_in] / [d_out, rank] (pinned)."""
        self._keep = getattr(self, "_keep", {})
        self._keep[slot] = (A_host, B_host)          # keep alive until the copy completes
        B.lora_load_slot(self.ctx, slot, [a.data_ptr() for a in A_host],
                         [b.data_ptr() for b in B_host], rank, alpha)

    def load_slots(self, slots, adapters, ranks, alphas):
        """Several adapters in one call: adapters[i] = (A_host list, B_host list)
        per layer, as for load_slot."""
        self._keep = getattr(self, "_keep", {})
        A_ptrs, B_ptrs = [], []
        for s, (A_host, B_host) in zip(slots, adapters):
            self._keep[s] = (A_host, B_host)
            A_ptrs += [a.data_ptr() for a in A_host]
            B_ptrs += [b.data_ptr() for b in B_host]
        B.lora_load_slots(self.ctx, slots, A_ptrs, B_ptrs, ranks, alphas)

    def assign(self, adapter_id, rank):
        return B.lora_assign(self.ctx, adapter_id, rank)

    def lookup(self, adapter_id):
        return B.lora_lookup(self.ctx, adapter_id)

    def acquire(self, slot):
        return B.lora_acquire(self.ctx, slot)

    def release(self, slot):
        return B.lora_release(self.ctx, slot)

    def evict_lru(self):
        return B.lora_evict_lru(self.ctx)

    def sync_uploads(self):
        B.lora_sync_uploads(self.ctx)

    def stats(self):
        return B.lora_stats(self.ctx)

    # --- apply -----------------------------------------------------------------
    def apply(self, layer, x, y, idx):
        B.lora_apply(self.ctx, layer, x.data_ptr(), y.data_ptr(), idx.data_ptr(), int(idx.shape[0]))

    def apply_multi(self, layers, xs, ys, idx):
        B.lora_apply_multi(self.ctx, list(layers), [x.data_ptr() for x in xs],
                           [y.data_ptr() for y in ys], idx.data_ptr(), int(idx.shape[0]))

    def close(self):
        if getattr(self, "ctx", None) is not None:
            B.lora_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
