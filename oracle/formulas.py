"""KV-cache size formulas -- TEST INFRASTRUCTURE ONLY (part of the oracle).

Page 1 ("大模型推理优化全攻略" §2.2), page 3 ("KV Cache 的显存计算") and page 4
("cs336 lecture 10", KV Cache 的内存占用) all state the same product: the
factor 2 counts K and V, times layers, KV heads, head dimension, sequence
length, batch and bytes per element. Page 4 also writes it with d_model in
place of KV heads x head dimension (the MHA case).
"""
from __future__ import annotations

import math


def kv_cache_bytes(num_layers: int, num_kv_heads: int, head_dim: int,
                   seq_len: int, batch: int, dtype_bytes: int) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * seq_len * batch * dtype_bytes


def kv_cache_bytes_dmodel(num_layers: int, d_model: int, seq_len: int,
                          dtype_bytes: int) -> int:
    """Page 4's form: 2 x L x d_model x S x dtype_size (MHA: d_model = heads x head_dim)."""
    return 2 * num_layers * d_model * seq_len * dtype_bytes


def paged_bytes(num_layers: int, num_kv_heads: int, head_dim: int,
                seq_lens, dtype_bytes: int, block_size: int = 16) -> int:
    """Bytes a paged pool holds for these sequences: whole blocks only
    (page 1 §2.3: the only waste is the unfilled tail of the last block)."""
    tokens = sum(block_size * math.ceil(L / block_size) for L in seq_lens)
    return kv_cache_bytes(num_layers, num_kv_heads, head_dim, tokens, 1, dtype_bytes)
