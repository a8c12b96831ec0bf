"""Algorithmic byte counts used for the roofline and the benchmark metric.

KV bytes per token per layer = 2 * n_kv * head_dim * dtype_bytes (the
tiniestgpt notes, section 0, and the CS336 lecture-10 guide's KV-cache size
formula M_KV = 2 L S n_kv d_h s); the worked example on the CS336 page
(n_kv=64, d_h=128, bf16: 32 KiB per token per layer; S=100,000 and L=80:
about 244 GiB) pins ``kv_cache_bytes``.

A decode launch must read, once, every KV row in each sequence's window,
their int8 scales, and Q, and write the output.  K and V stored as one
tensor count once; prefix blocks shared by several sequences count once
(unique physical slots).  Block-granular over-read, split partials and the
block table are not algorithmic and are not counted.
"""
from __future__ import annotations

import numpy as np


def kv_cache_bytes(layers: int, seq_len: int, n_kv: int, head_dim: int, dtype_bytes: int,
                   kv_tensors: int = 2) -> int:
    """Bytes of a dense KV cache: kv_tensors * L * S * n_kv * d_h * s."""
    return kv_tensors * layers * seq_len * n_kv * head_dim * dtype_bytes


def bytes_per_key(num_kv_heads: int, head_dim: int, kv: str, alias: bool) -> int:
    """Bytes one cached token contributes to a decode read, scales included."""
    es = 2 if kv == "bf16" else 1
    tensors = 1 if alias else 2
    b = tensors * num_kv_heads * head_dim * es
    if kv == "int8_token":
        b += tensors * 4
    return b


def window_slots(seq_lens: np.ndarray, block_table: np.ndarray, window: int, P: int = 16,
                 ring_blocks: int = 0):
    """Physical slot ids of every key a decode reads (keys [lo, pos]); for a
    ring layout key j sits in table entry (j mod W) / P, W = ring_blocks * P."""
    out = []
    for b, L in enumerate(np.asarray(seq_lens, np.int64)):
        if L <= 0:
            continue
        pos = L - 1
        lo = max(0, pos - window) if window > 0 else 0
        j = np.arange(lo, pos + 1, dtype=np.int64)
        entry = (j % (ring_blocks * P)) // P if ring_blocks else j // P
        out.append(block_table[b, entry].astype(np.int64) * P + j % P)
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def decode_bytes(spec, seq_lens, block_table, out_bytes_per_elem: int = 2) -> dict:
    """Algorithmic bytes of one decode of one layer."""
    slots = window_slots(seq_lens, block_table, spec.window, spec.block_size,
                         getattr(spec, "ring_blocks", 0))
    uniq = int(np.unique(slots).size)
    kv = uniq * bytes_per_key(spec.num_kv_heads, spec.head_dim, spec.kv, spec.alias)
    if spec.kv == "int8_head":
        kv += (1 if spec.alias else 2) * spec.num_kv_heads * 4
    B = len(seq_lens)
    q = B * spec.num_q_heads * spec.head_dim * 2
    out = B * spec.num_q_heads * spec.head_dim * out_bytes_per_elem
    return {"kv": kv, "q": q, "out": out, "keys": int(slots.size), "unique_keys": uniq}


def append_bytes(spec, num_tokens: int) -> int:
    """Read the new bf16 K/V rows, write them (or their int8 codes and scales)."""
    tensors = 1 if spec.alias else 2
    row = spec.num_kv_heads * spec.head_dim
    read = num_tokens * tensors * row * 2 + num_tokens * 8
    es = 2 if spec.kv == "bf16" else 1
    write = num_tokens * tensors * row * es
    if spec.kv == "int8_token":
        write += num_tokens * tensors * 4
    return read + write
