"""Pins of the oracle's ring-KV layout ("实验五：Gemma4 端到端推理优化", Ring KV
Cache: the KV of absolute position t lives in slot t mod W of a fixed ring,
overwriting keys that have left the window, and the method does not change
the attention range, so with correct indexing there is no accuracy loss).

The oracle's paged gather is pinned elsewhere (dense attention, block
permutation invariance, ...); here the ring gather is pinned to it: the same
keys through a ring and through a paged table give identical fp64 results,
at every offset of the window's ends inside a block, and when every position
of a sequence is written into the ring in order (so that old keys are really
overwritten).  A ring one block short of ceil((w + 1) / P) (fewer slots
than the w + 1 keys of an inclusive window) loses a key of some window,
which the same comparison catches."""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest

import oracle
from paged_kv_decode_03_gb300 import synth

P = 16


def _pools(w, ring_blocks):
    k, v, ks, vs = synth.empty_pool_arrays(w.spec, w.layout)
    mode = {"bf16": oracle.SCALE_NONE, "int8_token": oracle.SCALE_PER_TOKEN,
            "int8_head": oracle.SCALE_PER_HEAD}[w.spec.kv]
    if w.spec.kv == "int8_head":
        ks, vs = w.k_head_scale.copy(), (None if w.spec.alias else w.v_head_scale.copy())
    return oracle.OraclePool(k=k, v=v, k_scale=ks, v_scale=vs, scale_mode=mode,
                             ring_blocks=ring_blocks)


def _fill(w, pool):
    """History then the step's token, at the slots the pool's layout gives."""
    hs = oracle.slot_mapping(pool, w.block_table, w.hist_seq, w.hist_pos)
    assert np.all(hs >= 0)
    oracle.append(w.hist_k, w.hist_v, hs, pool)
    B = len(w.seq_lens)
    ns = oracle.slot_mapping(pool, w.block_table, np.arange(B, dtype=np.int32),
                             w.seq_lens.astype(np.int64) - 1)
    oracle.append(w.new_k, w.new_v, ns, pool)
    return pool


def _decode(w, pool):
    s = w.spec
    return oracle.decode(w.q, pool, w.block_table, w.seq_lens, s.num_q_heads, s.window,
                         np.float32(s.softmax_scale))


def _pair(spec, ring_blocks):
    """The same workload (lengths, values) in a ring layout and a paged one."""
    wr = synth.make_workload(replace(spec, ring_blocks=ring_blocks))
    wp = synth.make_workload(replace(spec, ring_blocks=0))
    assert np.array_equal(wr.seq_lens, wp.seq_lens)
    assert np.array_equal(wr.hist_k, wp.hist_k) and np.array_equal(wr.q, wp.q)
    return wr, wp


@pytest.mark.parametrize("kv", ["bf16", "int8_head"])
@pytest.mark.parametrize("window", [15, 16, 17, 40])
def test_ring_equals_paged_at_every_window_offset(kv, window):
    """Lengths put pos % P and (pos - w) % P through every value: the ring and
    the paged table give bit-identical results (no accuracy loss)."""
    lens = tuple(range(1, 3 * P + 2)) + tuple(range(5 * P, 7 * P + 1))
    spec = synth.Spec(f"ring_w{window}", batch=len(lens), num_q_heads=4, num_kv_heads=2,
                      head_dim=64, lens=("fixed", lens), window=window, kv=kv, seed=11)
    wr, wp = _pair(spec, synth.ring_blocks_for(window))
    got = _decode(wr, _fill(wr, _pools(wr, wr.spec.ring_blocks)))
    want = _decode(wp, _fill(wp, _pools(wp, 0)))
    assert np.array_equal(got, want)


def test_ring_memory_is_bounded_by_the_window():
    """O(min(S, W)) blocks per sequence: a sequence never owns more than the
    ring's blocks, however long it is."""
    spec = replace(synth.C2_RING, batch=16, lens=("fixed", tuple([1, 17, 1000, 1025, 1040,
                                                                  1041, 5000, 8192] * 2)))
    w = synth.make_workload(spec)
    used = (w.block_table >= 0).sum(axis=1)
    assert used.max() == synth.ring_blocks_for(1024) == w.block_table.shape[1]
    assert np.all(used == np.minimum(-(-w.seq_lens // P), spec.ring_blocks))


def _sequential_ring(window, ring_blocks, lens, seed=3):
    """Every position 0..len-1 of each sequence written into the ring in
    order (a real ring: later positions overwrite earlier ones), against a
    paged pool holding every position.  Returns both decodes."""
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, D = len(lens), 4, 2, 32
    lens = np.array(lens, np.int32)
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, Hq, D), dtype=np.float32))
    seq = np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int64) for L in lens])
    k = synth.f32_to_bf16_bits(rng.standard_normal((len(pos), Hkv, D), dtype=np.float32))
    v = synth.f32_to_bf16_bits(rng.standard_normal((len(pos), Hkv, D), dtype=np.float32))
    nblk = -(-lens // P)
    # paged: a private block per logical block
    bt_p = np.full((B, int(nblk.max())), -1, np.int32)
    nxt = 0
    for b in range(B):
        bt_p[b, :nblk[b]] = np.arange(nxt, nxt + nblk[b])
        nxt += nblk[b]
    paged = oracle.OraclePool(k=np.full((nxt, P, Hkv, D), synth.BF16_NAN, np.uint16),
                              v=np.full((nxt, P, Hkv, D), synth.BF16_NAN, np.uint16))
    oracle.append(k, v, oracle.slot_mapping(paged, bt_p, seq, pos), paged)
    # ring: ring_blocks blocks per sequence, positions written in order
    bt_r = (np.arange(B * ring_blocks, dtype=np.int32).reshape(B, ring_blocks))
    ring = oracle.OraclePool(k=np.full((B * ring_blocks, P, Hkv, D), synth.BF16_NAN, np.uint16),
                             v=np.full((B * ring_blocks, P, Hkv, D), synth.BF16_NAN, np.uint16),
                             ring_blocks=ring_blocks)
    oracle.append(k, v, oracle.slot_mapping(ring, bt_r, seq, pos), ring)
    scale = np.float32(1 / np.sqrt(D))
    return (oracle.decode(q, ring, bt_r, lens, Hq, window, scale),
            oracle.decode(q, paged, bt_p, lens, Hq, window, scale))


@pytest.mark.parametrize("window", [15, 16, 17, 33])
def test_sequential_ring_writes_lose_no_window_key(window):
    lens = list(range(1, 6 * P)) + [200, 333]
    got, want = _sequential_ring(window, synth.ring_blocks_for(window), lens)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("window", [16, 17, 33])
def test_a_ring_one_block_short_overwrites_a_window_key(window):
    """One block fewer than ceil((w + 1) / P) holds fewer slots than the window
    has keys: some window's oldest key has been overwritten by a newer
    position, and the result differs."""
    lens = list(range(1, 6 * P))
    got, want = _sequential_ring(window, synth.ring_blocks_for(window) - 1, lens)
    assert not np.array_equal(got, want)


def test_ring_slots_cycle_with_period_w():
    """Slots of positions t .. t+W-1 are the W distinct slots of the ring, and
    position t + W reuses the slot of t (slot t mod W)."""
    R = 5
    W = R * P
    bt = np.array([[7, 3, 11, 0, 5]], np.int32)
    pool = oracle.OraclePool(k=np.zeros((12, P, 1, 8), np.uint16), ring_blocks=R)
    pos = np.arange(4 * W, dtype=np.int64)
    s = oracle.slot_mapping(pool, bt, np.zeros(len(pos), np.int32), pos)
    for t0 in (0, 1, 15, 16, 17, W - 1, 2 * W + 3):
        window = s[t0:t0 + W]
        assert len(np.unique(window)) == W
        assert set(window.tolist()) == {int(b) * P + o for b in bt[0] for o in range(P)}
    assert np.array_equal(s[W:], s[:-W])
    assert np.array_equal(oracle.slot_mapping(pool, bt, np.zeros(1, np.int32),
                                              np.array([-1], np.int64)), [-1])
