"""Pins of the oracle's attention for a chunk of new tokens per sequence
(q_len > 1: chunked prefill, "实验五：Gemma4 端到端推理优化" Flash Attention and
continuous-batching sections; the gamma + 1 tokens a speculative step
verifies, tiniestgpt notes section 7).

The chunk is the last n tokens of each sequence, causal among themselves.
Pinned to the already-pinned decode and to a library attention routine: a
chunk of one token is the decode; every query of a chunk equals the decode
of the sequence cut after that query's position (the cache beyond it is
masked); on identity paging the chunk equals torch's scaled-dot-product
attention with an explicit causal (and band) mask in fp64."""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest

import oracle
from paged_kv_decode_03_gb300 import synth

torch = pytest.importorskip("torch")


def _pool(w):
    k, v, ks, vs = synth.empty_pool_arrays(w.spec, w.layout)
    mode = {"bf16": oracle.SCALE_NONE, "int8_token": oracle.SCALE_PER_TOKEN,
            "int8_head": oracle.SCALE_PER_HEAD}[w.spec.kv]
    if w.spec.kv == "int8_head":
        ks, vs = w.k_head_scale.copy(), (None if w.spec.alias else w.v_head_scale.copy())
    pool = oracle.OraclePool(k=k, v=v, k_scale=ks, v_scale=vs, scale_mode=mode)
    if len(w.hist_slots):
        oracle.append(w.hist_k, w.hist_v, w.hist_slots, pool)
    oracle.append(w.new_k, w.new_v, w.new_slots, pool)
    return pool


def _spec(window, kv="bf16", hq=4, hkv=2, lens=(1, 2, 16, 17, 33, 100, 257)):
    return synth.Spec(f"chunk_w{window}_{kv}", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=32, lens=("fixed", lens), window=window, kv=kv, seed=31)


def _prefill(w, pool):
    s = w.spec
    return oracle.prefill(w.q, pool, w.block_table, w.seq_lens, w.q_start, s.num_q_heads,
                          s.window, np.float32(s.softmax_scale))


@pytest.mark.parametrize("window", [0, 5, 16])
def test_chunk_of_one_is_the_decode(window):
    w = synth.make_chunk_workload(_spec(window), 1)
    pool = _pool(w)
    got = _prefill(w, pool)
    want = oracle.decode(w.q, pool, w.block_table, w.seq_lens, w.spec.num_q_heads, w.spec.window,
                         np.float32(w.spec.softmax_scale))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kv", ["bf16", "int8_token", "int8_head"])
@pytest.mark.parametrize("window,n", [(0, 4), (0, 17), (7, 17), (16, 5), (40, 64)])
def test_each_query_is_the_decode_of_its_prefix(kv, window, n):
    """Query i of sequence b (position len - n + i) gives what a decode of
    the same cache with length len - n + i + 1 gives for that query."""
    w = synth.make_chunk_workload(_spec(window, kv), n)
    pool = _pool(w)
    got = _prefill(w, pool)
    s = w.spec
    for b in range(len(w.seq_lens)):
        q0, q1 = int(w.q_start[b]), int(w.q_start[b + 1])
        for i in range(q1 - q0):
            lens = w.seq_lens.copy()
            lens[b] = w.seq_lens[b] - (q1 - q0) + i + 1
            qb = np.repeat(w.q[q0 + i][None], len(lens), axis=0)
            rows = np.array([[b, h] for h in range(s.num_q_heads)], np.int32)
            want = oracle.decode(qb, pool, w.block_table, lens, s.num_q_heads, s.window,
                                 np.float32(s.softmax_scale), rows=rows)
            assert np.array_equal(got[q0 + i], want), (b, i)


@pytest.mark.parametrize("window", [0, 9])
def test_chunk_equals_causal_sdpa_on_identity_paging(window):
    """One sequence whose logical block j is physical block j: the chunk's
    output is softmax(Q K^T * scale + M) V with M the causal band of the
    pages' mask, computed by torch in fp64 (GQA by repeating K/V heads)."""
    L, n, hq, hkv, D = 70, 23, 4, 2, 32
    spec = synth.Spec("sdpa_chunk", batch=1, num_q_heads=hq, num_kv_heads=hkv, head_dim=D,
                      lens=("fixed", (L,)), window=window, seed=41, pool_factor=1.0)
    w = synth.make_chunk_workload(spec, n)
    nb = -(-L // 16)
    w = replace(w, layout=replace(w.layout, block_table=np.arange(nb, dtype=np.int32)[None]))
    pos_all = np.arange(L)
    first = L - n
    lo = max(0, first - window) if window else 0
    hist_pos = np.arange(lo, first)
    w = replace(w, hist_slots=hist_pos.astype(np.int64), new_slots=np.arange(first, L, dtype=np.int64))
    pool = _pool(w)
    got = _prefill(w, pool)
    # dense K/V in logical order (positions below lo are never written: poison,
    # masked out below)
    K = oracle.bf16_bits_to_f64(pool.k.reshape(-1, hkv, D)[:L])
    V = oracle.bf16_bits_to_f64(pool.v.reshape(-1, hkv, D)[:L])
    Q = oracle.bf16_bits_to_f64(w.q)                              # [n, hq, D]
    G = hq // hkv
    Kt = torch.from_numpy(np.repeat(K, G, axis=1)).permute(1, 0, 2)   # [hq, L, D]
    Vt = torch.from_numpy(np.repeat(V, G, axis=1)).permute(1, 0, 2)
    Kt = torch.nan_to_num(Kt)
    Vt = torch.nan_to_num(Vt)
    Qt = torch.from_numpy(Q).permute(1, 0, 2)                     # [hq, n, D]
    qpos = np.arange(first, L)[:, None]
    allowed = (pos_all[None, :] <= qpos) & ((pos_all[None, :] >= qpos - window) if window else True)
    allowed &= pos_all[None, :] >= lo
    mask = torch.from_numpy(allowed)
    ref = torch.nn.functional.scaled_dot_product_attention(
        Qt, Kt, Vt, attn_mask=mask, scale=float(np.float32(spec.softmax_scale)))
    np.testing.assert_allclose(got, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)
