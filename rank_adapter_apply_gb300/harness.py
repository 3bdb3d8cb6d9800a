"""Run a synthetic Workload through the library: device buffers, slot uploads
and apply calls. Used by the tests, the smoke check and the benchmark. It moves
data and calls the C ABI; it computes nothing itself."""
from __future__ import annotations

import numpy as np
import torch

from . import workloads as wl
from .slots import LoraSlots


def to_torch(arr: np.ndarray, dtype_code: int) -> torch.Tensor:
    """Host tensor sharing the numpy buffer (uint16 bf16 bits -> torch.bfloat16)."""
    a = np.ascontiguousarray(arr)
    if dtype_code == wl.DTYPE_BF16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def from_torch(t: torch.Tensor) -> np.ndarray:
    """Device/host tensor -> numpy (bf16 as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


class DeviceWorkload:
    """A Workload resident on the GPU with every adapter uploaded to its slot."""

    def __init__(self, w: wl.Workload, device="cuda:0", max_tokens=None, pin=True,
                 prefill_min_tokens=None, small_batch_tokens=None):
        self.w = w
        self.device = torch.device(device)
        tdt = torch.bfloat16 if w.dtype == wl.DTYPE_BF16 else torch.float32
        self.layer_index = {ly.name: i for i, ly in enumerate(w.layers)}
        self.slots = LoraSlots([(ly.d_in, ly.d_out) for ly in w.layers], w.max_loras,
                               w.max_lora_rank, max_tokens or max(1, w.n_tokens), dtype=tdt,
                               max_layers_per_call=min(8, len(w.layers)), device=device)
        from . import binding as B
        if prefill_min_tokens is not None:
            B.lora_set_prefill_min_tokens(self.slots.ctx, prefill_min_tokens)
        if small_batch_tokens is not None:
            B.lora_set_small_batch_tokens(self.slots.ctx, small_batch_tokens)
        self.host_adapters = []
        for s, ad in enumerate(w.adapters):
            if ad is None:
                continue
            A = [to_torch(ad[ly.name][0], w.dtype) for ly in w.layers]
            Bm = [to_torch(ad[ly.name][1], w.dtype) for ly in w.layers]
            if pin:
                A = [a.pin_memory() for a in A]
                Bm = [b.pin_memory() for b in Bm]
            self.host_adapters.append((A, Bm))
            self.slots.load_slot(s, A, Bm, int(w.ranks[s]), float(w.alphas[s]))
        self.slots.sync_uploads()
        self.xs = {k: to_torch(v, w.dtype).to(self.device) for k, v in w.xs.items()}
        self.y_in = {k: to_torch(v, w.dtype).to(self.device) for k, v in w.ys.items()}
        self.idx = torch.from_numpy(w.token_slot_idx).to(self.device)
        self.ys = {}
        self.reset()

    def reset(self):
        for k, v in self.y_in.items():
            self.ys[k] = v.clone()
        torch.cuda.synchronize(self.device)

    def run(self, layer_names=None, multi=True):
        names = layer_names or [ly.name for ly in self.w.layers]
        torch.cuda.synchronize(self.device)
        if multi:
            lys = [self.layer_index[n] for n in names]
            xs = [self.xs[self.w.layers[i].x_key] for i in lys]
            ys = [self.ys[n] for n in names]
            self.slots.apply_multi(lys, xs, ys, self.idx)
        else:
            for n in names:
                i = self.layer_index[n]
                self.slots.apply(i, self.xs[self.w.layers[i].x_key], self.ys[n], self.idx)
        self.slots.compute.synchronize()
        return {n: from_torch(self.ys[n]) for n in names}

    def close(self):
        self.slots.close()
