"""Adapter capacity formula (test infrastructure only).

The "Multi-LoRA 适配器缓存生产实战" page, section "Adapter 容量不能只按「个数」规划",
estimates an adapter's size as the sum over every injected linear layer of
(d_in + d_out) * rank * bytes_per_param. For a LoRA pair A [r, d_in] and
B [d_out, r] that sum is the exact count of weight bytes the slot upload moves.
"""


def adapter_bytes(layers, rank: int, bytes_per_param: int) -> int:
    """layers: iterable of (d_in, d_out) for the injected linears."""
    return sum((int(d_in) + int(d_out)) * int(rank) * int(bytes_per_param)
               for d_in, d_out in layers)
