"""TurboQuant KV-cache hot path on GB300: fused quantising store and split-K
decode attention over a packed paged cache, behind the C ABI in include/tq.h.

`TQCache` bundles the per-layer constants (codebook, signs) and a paged
cache; `_lib` holds the raw C-ABI binding.
"""
from __future__ import annotations

from . import _lib
from ._lib import (PRESETS, TQ_2BIT_NC, TQ_3BIT_NC, TQ_4BIT_NC, TQ_LAYOUT_SOA, TQ_BF16, TQ_F16, TQ_F32, TQ_K3V4_NC,
                   TQ_K8V4, TQError, decode_attention, dequant, load, store, tq_build_codebook,
                   tq_decode_attention, tq_decode_kernel_kind, tq_decode_pick_splits, tq_decode_workspace_bytes,
                   tq_decode_attention_sparse_v, tq_dequant, tq_get_layout, tq_make_signs, tq_status_string, tq_store, tq_version)

__all__ = ["PRESETS", "TQ_K8V4", "TQ_4BIT_NC", "TQ_K3V4_NC", "TQ_3BIT_NC", "TQ_2BIT_NC", "TQ_LAYOUT_SOA", "TQ_F16", "TQ_BF16",
           "TQ_F32", "TQError", "TQCache", "load", "store", "decode_attention", "dequant", "tq_store",
           "tq_decode_attention", "tq_decode_attention_sparse_v", "tq_dequant", "tq_decode_kernel_kind", "tq_get_layout", "tq_build_codebook", "tq_make_signs",
           "tq_decode_workspace_bytes", "tq_decode_pick_splits", "tq_status_string", "tq_version"]

SIGN_SEED = 42          # per-layer seed = 42 + 1337 * layer
LAYER_SEED_STRIDE = 1337


class TQCache:
    """One layer's packed paged cache plus the device constants its kernels read.

    Holds device tensors only; every operation is one C-ABI call.
    """

    def __init__(self, preset, num_blocks: int, block_size: int, num_kv_heads: int,
                 head_dim: int = 128, layer: int = 0, device="cuda"):
        import torch
        self.preset = PRESETS[preset] if isinstance(preset, str) else int(preset)
        self.layout = tq_get_layout(self.preset, head_dim)
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.num_kv_heads, self.head_dim = int(num_kv_heads), int(head_dim)
        self.device = torch.device(device)
        self.cache = torch.zeros((num_blocks, block_size, num_kv_heads,
                                  self.layout["slot_size_aligned"]), dtype=torch.uint8,
                                 device=self.device)
        self.signs = torch.from_numpy(
            tq_make_signs(head_dim, SIGN_SEED + LAYER_SEED_STRIDE * layer)).to(self.device)
        if self.layout["key_fp8"]:
            self.centroids = self.midpoints = None
        else:
            c, m = tq_build_codebook(head_dim, self.layout["key_bits"])
            self.centroids = torch.from_numpy(c).to(self.device)
            self.midpoints = torch.from_numpy(m).to(self.device)

    def store(self, key, value, slot_mapping, stream=None):
        store(self.preset, key, value, slot_mapping, self.cache, self.block_size, self.signs,
              self.centroids, self.midpoints, stream)

    def workspace(self, batch: int, num_q_heads: int, num_splits: int):
        import torch
        nbytes = tq_decode_workspace_bytes(batch, num_q_heads, num_splits, self.head_dim)
        return torch.empty(max(16, nbytes), dtype=torch.uint8, device=self.device)

    def dequant(self, slot_mapping, key_out, value_out, stream=None):
        """K and V of the slots slot_mapping names, in the original space."""
        dequant(self.preset, slot_mapping, self.cache, self.num_kv_heads, self.block_size,
                self.signs, self.centroids, key_out, value_out, stream)

    def decode(self, query, block_table, seq_lens, max_seq_len, out, lse, workspace,
               num_splits=0, softmax_scale=None, stream=None, v_threshold=0.0):
        decode_attention(self.preset, query, self.cache, block_table, seq_lens, max_seq_len,
                         self.num_kv_heads, self.block_size, self.signs, self.centroids, out,
                         lse, workspace, num_splits, softmax_scale, stream, v_threshold)
