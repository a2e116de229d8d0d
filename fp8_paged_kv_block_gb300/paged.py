"""Device-side construction of FP8 decode inputs with the library's kernels.

Given float K/V of whole sequences (concatenated, with cu_seqlens) and each
token's physical slot, build the paged E4M3 cache the way the GLM-4.5 paged
FP8 page quantises it: K per (token, head) with scale amax/448, V per channel
with one scale per sequence, head and channel (max over the sequence). Query
rows are quantised per (token, head). All arithmetic runs in the library.
"""
from __future__ import annotations

from dataclasses import dataclass

from . import (LAYOUT_BNBD, LAYOUT_BSND, cache_quant_scatter, quantize_rows,
               value_channel_scale)


@dataclass
class PagedFP8:
    k_cache: "torch.Tensor"      # uint8, layout-shaped
    v_cache: "torch.Tensor"
    k_scale: "torch.Tensor"      # float32, cache shape without D
    v_scale: "torch.Tensor"      # float32 [B, NKV, D]
    layout: int


def empty_cache(num_blocks: int, NKV: int, D: int, layout: int, device, block_size: int = 128):
    import torch
    if layout == LAYOUT_BSND:
        shape = (num_blocks, block_size, NKV, D)
    else:
        shape = (num_blocks, NKV, block_size, D)
    kc = torch.zeros(shape, dtype=torch.uint8, device=device)
    vc = torch.zeros(shape, dtype=torch.uint8, device=device)
    ks = torch.zeros(shape[:3], dtype=torch.float32, device=device)
    return kc, vc, ks


def build_cache(k, v, cu_seqlens, slots, token_batch, num_blocks: int, layout: int,
                block_size: int = 128, stream=None) -> PagedFP8:
    """k, v float32/bfloat16 [Ttot, NKV, D] on the device; cu_seqlens int64
    [B+1], slots int64 [Ttot] (physical slot of each token), token_batch int32
    [Ttot], all on the device."""
    import torch
    T, NKV, D = k.shape
    B = cu_seqlens.shape[0] - 1
    kc, vc, ks = empty_cache(num_blocks, NKV, D, layout, k.device, block_size)
    vs = torch.empty((B, NKV, D), dtype=torch.float32, device=k.device)
    value_channel_scale(v, cu_seqlens, vs, stream=stream)
    if T > 0:
        cache_quant_scatter(k, v, kc, vc, slots, ks, vs, token_batch, layout=layout, stream=stream)
    return PagedFP8(kc, vc, ks, vs, layout)


def quantize_queries(q, stream=None):
    """q float32/bfloat16 [B*S1, NQ, D] -> (codes uint8, scale float32 [B*S1, NQ])."""
    import torch
    codes = torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    scale = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    quantize_rows(q, codes, scale, stream=stream)
    return codes, scale


__all__ = ["PagedFP8", "empty_cache", "build_cache", "quantize_queries", "LAYOUT_BSND",
           "LAYOUT_BNBD"]
