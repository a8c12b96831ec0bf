"""Seeded synthetic workloads for paged-KV decode attention.

This module only draws random numbers and lays out blocks: lengths, block
tables, slot ids, bf16 values, static scales chosen by the caller and poison
for slots that must never be read.  It holds none of the method's arithmetic
(no attention, no quantisation), so both the CUDA path and the CPU oracle can
take their inputs from it.

The five workloads follow the shapes the pages describe: a tiny global layer;
a Gemma4-12B sliding-window layer (H_q=16, H_kv=8, head_dim=256, w=1024) and
global layer (H_kv=1, K and V one tensor), from the Lab5-Gemma4 page's
sections on sliding windows, GQA and weight sharing; a Llama-2-13B-like MHA
layer (40 heads of 128) with int8 KV, from the CS336 lecture-10 guide's
Llama 2 13B example and int8 section (outliers: values ~0.1% of which are
large); and a continuous-batching step with ragged lengths, a 5:1
sliding:global layer pattern ("1 global per 6 layers") and shared prefix
blocks (the tiniestgpt notes' prefix caching and the CS336 guide's vLLM
section).  The pages publish no dataset for this kernel; these seeded inputs
stand in for the request traces they mention.

bf16 values are carried as uint16 bit patterns (numpy has no bf16).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional, Tuple

import numpy as np

BF16_NAN = np.uint16(0x7FC0)   # poison for bf16 slots that must never be read
INT8_POISON = np.int8(127)     # poison for int8 slots
F32_NAN = np.float32("nan")    # poison for per-token scales of unread slots


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even) via torch's CPU cast."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Spec:
    """One attention layer's workload.

    lens: ("fixed", (l0, l1, ...)) | ("uniform", lo, hi) | ("const", n) |
          ("lognormal", median, sigma, lo, hi)
    kv:   "bf16" | "int8_token" | "int8_head"
    """
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    lens: tuple
    block_size: int = 16
    window: int = 0
    kv: str = "bf16"
    alias: bool = False
    pool_factor: float = 1.25
    pool_blocks: Optional[int] = None
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    shared_prefix_blocks: int = 0
    shared_prefix_seqs: int = 0
    shared_min_len: int = 0
    split_tokens: int = 0
    seed: int = 1234
    # 0: paged layout (the block table lists every logical block); > 0: ring
    # layout of a sliding layer, each sequence owning a ring of this many
    # blocks (only the blocks its length reaches are allocated)
    ring_blocks: int = 0

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


# The workloads.  Seeds are 1234 + workload index.
C1 = Spec("c1_tiny_global", batch=4, num_q_heads=4, num_kv_heads=2, head_dim=64,
          lens=("fixed", (1, 7, 16, 33)), pool_blocks=16, seed=1235)
C2 = Spec("c2_gemma4_sliding", batch=64, num_q_heads=16, num_kv_heads=8, head_dim=256,
          lens=("uniform", 512, 8192), window=1024, seed=1236)
C3 = Spec("c3_gemma4_global_kv_shared", batch=32, num_q_heads=16, num_kv_heads=1, head_dim=256,
          lens=("uniform", 4096, 32768), alias=True, split_tokens=1024, seed=1237)
C4 = Spec("c4_llama2_13b_mha_int8_token", batch=64, num_q_heads=40, num_kv_heads=40,
          head_dim=128, lens=("const", 2048), kv="int8_token", outlier_frac=0.01,
          outlier_mult=8.0, seed=1238)
C5_SLIDING = Spec("c5_step_sliding", batch=256, num_q_heads=16, num_kv_heads=8, head_dim=256,
                  lens=("lognormal", 1500.0, 1.0, 1, 65536), window=1024, kv="int8_head",
                  shared_prefix_blocks=8, shared_prefix_seqs=64, shared_min_len=130, seed=1239)
C5_GLOBAL = replace(C5_SLIDING, name="c5_step_global", num_kv_heads=1, window=0, kv="bf16")
C5_LAYERS = ("S", "S", "S", "S", "S", "G")

# Ring-KV variants of the sliding layers (Lab5-Gemma4, Ring KV Cache): each
# sequence's keys live in a ring of W = ring_blocks * 16 slots, W >= w + 1 so
# that the inclusive window [pos - w, pos] fits.
def ring_blocks_for(window: int, block_size: int = 16) -> int:
    return -(-(window + 1) // block_size)


C2_RING = replace(C2, name="c2_gemma4_sliding_ring", ring_blocks=ring_blocks_for(C2.window))
C5_SLIDING_RING = replace(C5_SLIDING, name="c5_step_sliding_ring", shared_prefix_blocks=0,
                          shared_prefix_seqs=0, ring_blocks=ring_blocks_for(C5_SLIDING.window))

CONFIGS = {"c1": C1, "c2": C2, "c3": C3, "c4": C4, "c5s": C5_SLIDING, "c5g": C5_GLOBAL,
           "c2r": C2_RING, "c5sr": C5_SLIDING_RING}


@dataclass
class Layout:
    """Sequence lengths and the block structure shared by the layers of a step."""
    seq_lens: np.ndarray        # [B] int32, includes the token appended this step
    block_table: np.ndarray     # [B, max_blocks] int32 (unused entries -1)
    num_blocks: int
    owner_first: np.ndarray     # [num_blocks] bool: block's content comes from this seq's history
    shared_seqs: np.ndarray     # [B] bool: the seq's first blocks are the shared prefix


@dataclass
class Workload:
    spec: Spec
    layout: Layout
    q: np.ndarray                        # [B, H_q, D] uint16
    hist_k: np.ndarray                   # [T, H_kv, D] uint16, tokens present before the step
    hist_v: Optional[np.ndarray]
    hist_slots: np.ndarray               # [T] int64
    new_k: np.ndarray                    # [B, H_kv, D] uint16, the step's token (position len-1)
    new_v: Optional[np.ndarray]
    new_slots: Optional[np.ndarray]      # [B] int64 (paged layouts; None for rings)
    k_head_scale: Optional[np.ndarray] = None   # [H_kv] fp32 (int8_head only)
    v_head_scale: Optional[np.ndarray] = None
    hist_seq: Optional[np.ndarray] = None       # [T] int32 sequence of each history token
    hist_pos: Optional[np.ndarray] = None       # [T] int64 its absolute position

    @property
    def seq_lens(self):
        return self.layout.seq_lens

    @property
    def block_table(self):
        return self.layout.block_table


def sample_lens(spec: Spec, rng: np.random.Generator) -> np.ndarray:
    kind = spec.lens[0]
    if kind == "fixed":
        lens = np.array(spec.lens[1], dtype=np.int64)
        assert len(lens) == spec.batch
    elif kind == "uniform":
        lens = rng.integers(spec.lens[1], spec.lens[2] + 1, size=spec.batch)
    elif kind == "const":
        lens = np.full(spec.batch, spec.lens[1], dtype=np.int64)
    elif kind == "lognormal":
        median, sigma, lo, hi = spec.lens[1:]
        lens = np.rint(rng.lognormal(math.log(median), sigma, size=spec.batch))
        lens = np.clip(lens, lo, hi).astype(np.int64)
    else:
        raise ValueError(kind)
    return lens.astype(np.int32)


def make_layout(spec: Spec, rng: np.random.Generator) -> Layout:
    P = spec.block_size
    lens = sample_lens(spec, rng)
    B = spec.batch
    nblk = (lens.astype(np.int64) + P - 1) // P
    shared = np.zeros(B, bool)
    if spec.shared_prefix_seqs:
        cand = np.nonzero(lens >= spec.shared_min_len)[0]
        pick = rng.permutation(cand)[: spec.shared_prefix_seqs]
        shared[pick] = True
    nshared = spec.shared_prefix_blocks if shared.any() else 0
    if spec.ring_blocks:
        # a ring holds at most ring_blocks blocks per sequence
        assert not nshared, "ring layouts share no prefix blocks"
        nblk = np.minimum(nblk, spec.ring_blocks)
    # logical blocks that need a private physical block
    private = int(nblk.sum() - nshared * (shared.sum() - 1)) if nshared else int(nblk.sum())
    num_blocks = spec.pool_blocks or max(1, int(math.ceil(private * spec.pool_factor)))
    assert num_blocks >= private
    perm = rng.permutation(num_blocks).astype(np.int32)
    maxb = spec.ring_blocks or max(1, int(nblk.max()))
    bt = np.full((B, maxb), -1, np.int32)
    owner = np.zeros(num_blocks, bool)
    nxt = 0
    shared_ids = None
    for b in range(B):
        start = 0
        if shared[b] and shared_ids is not None:
            bt[b, :nshared] = shared_ids
            start = nshared
        for i in range(start, int(nblk[b])):
            bt[b, i] = perm[nxt]
            owner[perm[nxt]] = True
            nxt += 1
        if shared[b] and shared_ids is None:
            shared_ids = bt[b, :nshared].copy()
    return Layout(lens, bt, num_blocks, owner, shared)


def _normal_bf16(rng: np.random.Generator, shape, spec: Spec, sigma=None) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if sigma is not None:
        x *= sigma
    if spec.outlier_frac > 0:
        m = rng.random(size=shape, dtype=np.float32) < spec.outlier_frac
        x[m] *= np.float32(spec.outlier_mult)
    return f32_to_bf16_bits(x)


def history_positions(spec: Spec, layout: Layout) -> Tuple[np.ndarray, np.ndarray]:
    """(seq, position) pairs of the history tokens to write before the step:
    every position < len-1 a decode at position len-1 may read (positions in
    [len-1-w, len-2] on sliding layers, all of them on global layers), minus
    positions inside shared prefix blocks of any but the first sharing seq."""
    P = spec.block_size
    nshared = spec.shared_prefix_blocks * P
    seqs, poss = [], []
    first_shared = None
    for b in range(spec.batch):
        L = int(layout.seq_lens[b])
        lo = max(0, L - 1 - spec.window) if spec.window > 0 else 0
        ranges = [(lo, L - 1)]
        if layout.shared_seqs[b]:
            if first_shared is None:
                # the first sharing sequence writes the whole shared prefix once,
                # whether or not its own window reaches it
                first_shared = b
                ranges = [(0, nshared), (max(lo, nshared), L - 1)]
            else:
                ranges = [(max(lo, nshared), L - 1)]
        for s, e in ranges:
            if e > s:
                seqs.append(np.full(e - s, b, np.int64))
                poss.append(np.arange(s, e, dtype=np.int64))
    if not seqs:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    return np.concatenate(seqs), np.concatenate(poss)


def slot_of(layout: Layout, P: int, seq: np.ndarray, pos: np.ndarray) -> np.ndarray:
    return layout.block_table[seq, pos // P].astype(np.int64) * P + pos % P


def make_workload(spec: Spec, layout: Optional[Layout] = None, seed_offset: int = 0) -> Workload:
    """Build one layer's inputs.  Pass ``layout`` to share lengths and block
    tables between the layers of one step (each layer draws its own values)."""
    rng = np.random.default_rng(spec.seed)
    if layout is None:
        layout = make_layout(spec, rng)
    vrng = np.random.default_rng(spec.seed * 1000 + 17 + seed_offset)
    B, Hq, Hkv, D, P = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    sigma = None
    k_hs = v_hs = None
    if spec.kv == "int8_head":
        # caller-chosen static scales: head h holds N(0, sigma_h^2) values and is
        # given the scale 4 sigma_h / 127, so values beyond 4 sigma saturate.
        sig = (0.5 + 0.25 * np.arange(Hkv, dtype=np.float32)).astype(np.float32)
        sigma = sig[None, :, None]
        k_hs = (np.float32(4.0) * sig / np.float32(127.0)).astype(np.float32)
        v_hs = (np.float32(3.0) * sig / np.float32(127.0)).astype(np.float32)
    q = _normal_bf16(vrng, (B, Hq, D), replace(spec, outlier_frac=0.0))
    seq, pos = history_positions(spec, layout)
    # paged layouts carry their slot ids; for a ring the caller maps
    # (sequence, position) to a slot with its own address map
    hist_slots = None if spec.ring_blocks else slot_of(layout, P, seq, pos)
    hist_k = _normal_bf16(vrng, (len(seq), Hkv, D), spec, sigma)
    hist_v = None if spec.alias else _normal_bf16(vrng, (len(seq), Hkv, D), spec, sigma)
    last = layout.seq_lens.astype(np.int64) - 1
    bidx = np.arange(B, dtype=np.int64)
    new_slots = (None if spec.ring_blocks else
                 np.where(last >= 0, slot_of(layout, P, bidx, np.maximum(last, 0)), -1))
    new_k = _normal_bf16(vrng, (B, Hkv, D), spec, sigma)
    new_v = None if spec.alias else _normal_bf16(vrng, (B, Hkv, D), spec, sigma)
    return Workload(spec, layout, q, hist_k, hist_v, hist_slots, new_k, new_v, new_slots,
                    k_hs, v_hs, seq.astype(np.int32), pos)


def make_step(spec_s: Spec = C5_SLIDING, spec_g: Spec = C5_GLOBAL,
              pattern=C5_LAYERS, share_history: bool = False) -> List[Workload]:
    """A continuous-batching step: one layout shared by all layers, one
    workload per layer (sliding or global spec by the pattern).  Each layer
    draws its own query and new token.  With ``share_history`` the layers of
    one kind reuse the first such layer's history values (the same arrays,
    appended into each layer's own pool), which keeps full-size six-layer
    steps affordable on the host."""
    rng = np.random.default_rng(spec_s.seed)
    layout = make_layout(spec_s, rng)
    out = []
    first = {}
    for i, kind in enumerate(pattern):
        spec = spec_s if kind == "S" else spec_g
        if not share_history or kind not in first:
            w = make_workload(spec, layout, seed_offset=i)
            first.setdefault(kind, w)
        else:
            w0 = first[kind]
            vrng = np.random.default_rng(spec.seed * 1000 + 17 + i)
            B, Hq, Hkv, D = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
            sigma = None
            if spec.kv == "int8_head":
                sigma = (0.5 + 0.25 * np.arange(Hkv, dtype=np.float32))[None, :, None]
            q = _normal_bf16(vrng, (B, Hq, D), replace(spec, outlier_frac=0.0))
            nk = _normal_bf16(vrng, (B, Hkv, D), spec, sigma)
            nv = None if spec.alias else _normal_bf16(vrng, (B, Hkv, D), spec, sigma)
            w = replace(w0, q=q, new_k=nk, new_v=nv)
        out.append(w)
    return out


def empty_pool_arrays(spec: Spec, layout: Layout):
    """Pool arrays filled with poison: (k, v, k_scale, v_scale) numpy arrays.
    Every slot that a correct decode reads is overwritten by the appends."""
    shape = (layout.num_blocks, spec.block_size, spec.num_kv_heads, spec.head_dim)
    if spec.kv == "bf16":
        k = np.full(shape, BF16_NAN, np.uint16)
    else:
        k = np.full(shape, INT8_POISON, np.int8)
    v = None if spec.alias else k.copy()
    ks = vs = None
    if spec.kv == "int8_token":
        ks = np.full(layout.num_blocks * spec.block_size, F32_NAN, np.float32)
        vs = None if spec.alias else ks.copy()
    return k, v, ks, vs


def shrink(spec: Spec, **kw) -> Spec:
    """A smaller variant of a workload for oracle-speed parity tests."""
    return replace(spec, **kw)


@dataclass
class ChunkWorkload:
    """A chunk of n_b new tokens per sequence (chunked prefill, or the
    gamma + 1 tokens a speculative step verifies): the chunk is the last n_b
    tokens of each sequence (seq_lens include it); queries are rows
    q_start[b] .. q_start[b+1]-1 of q; the chunk's K/V are appended before
    attending, after the history the chunk's queries may read."""
    spec: Spec
    layout: Layout
    q: np.ndarray              # [total, H_q, D] uint16
    q_start: np.ndarray        # [B + 1] int32
    hist_k: np.ndarray         # [T, H_kv, D] uint16
    hist_v: Optional[np.ndarray]
    hist_slots: np.ndarray     # [T] int64
    new_k: np.ndarray          # [total, H_kv, D] uint16, the chunk's tokens in order
    new_v: Optional[np.ndarray]
    new_slots: Optional[np.ndarray]  # [total] int64 (paged layouts; None for rings)
    k_head_scale: Optional[np.ndarray] = None
    v_head_scale: Optional[np.ndarray] = None
    hist_seq: Optional[np.ndarray] = None
    hist_pos: Optional[np.ndarray] = None
    new_seq: Optional[np.ndarray] = None
    new_pos: Optional[np.ndarray] = None

    @property
    def seq_lens(self):
        return self.layout.seq_lens

    @property
    def block_table(self):
        return self.layout.block_table


def make_chunk_workload(spec: Spec, q_lens) -> ChunkWorkload:
    """``q_lens``: chunk length per sequence (an int for all, or a sequence of
    B ints), clipped to each sequence's length.  For a ring layout the slots
    are left to each side's own address map (positions are given)."""
    rng = np.random.default_rng(spec.seed)
    layout = make_layout(spec, rng)
    vrng = np.random.default_rng(spec.seed * 1000 + 29)
    B, Hq, Hkv, D, P = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    lens = layout.seq_lens.astype(np.int64)
    n = np.broadcast_to(np.asarray(q_lens, np.int64), (B,))
    n = np.minimum(n, lens).astype(np.int64)
    q_start = np.zeros(B + 1, np.int32)
    q_start[1:] = np.cumsum(n)
    total = int(q_start[-1])
    sigma = None
    k_hs = v_hs = None
    if spec.kv == "int8_head":
        sig = (0.5 + 0.25 * np.arange(Hkv, dtype=np.float32)).astype(np.float32)
        sigma = sig[None, :, None]
        k_hs = (np.float32(4.0) * sig / np.float32(127.0)).astype(np.float32)
        v_hs = (np.float32(3.0) * sig / np.float32(127.0)).astype(np.float32)
    q = _normal_bf16(vrng, (total, Hq, D), replace(spec, outlier_frac=0.0))
    # history: the positions before each chunk that its first query may read
    seqs, poss = [], []
    for b in range(B):
        first = int(lens[b] - n[b])
        lo = max(0, first - spec.window) if spec.window > 0 else 0
        if first > lo:
            seqs.append(np.full(first - lo, b, np.int64))
            poss.append(np.arange(lo, first, dtype=np.int64))
    hseq = np.concatenate(seqs) if seqs else np.zeros(0, np.int64)
    hpos = np.concatenate(poss) if poss else np.zeros(0, np.int64)
    hist_slots = None if spec.ring_blocks else slot_of(layout, P, hseq, hpos)
    hist_k = _normal_bf16(vrng, (len(hseq), Hkv, D), spec, sigma)
    hist_v = None if spec.alias else _normal_bf16(vrng, (len(hseq), Hkv, D), spec, sigma)
    nseq = np.repeat(np.arange(B, dtype=np.int64), n)
    npos = np.concatenate([np.arange(lens[b] - n[b], lens[b], dtype=np.int64) for b in range(B)]) \
        if total else np.zeros(0, np.int64)
    new_slots = None if spec.ring_blocks else slot_of(layout, P, nseq, npos)
    new_k = _normal_bf16(vrng, (total, Hkv, D), spec, sigma)
    new_v = None if spec.alias else _normal_bf16(vrng, (total, Hkv, D), spec, sigma)
    return ChunkWorkload(spec, layout, q, q_start, hist_k, hist_v, hist_slots, new_k, new_v,
                         new_slots, k_hs, v_hs, hseq.astype(np.int32), hpos,
                         nseq.astype(np.int32), npos)
