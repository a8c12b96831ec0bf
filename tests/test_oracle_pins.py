"""Pins for the CPU oracle: each test checks the oracle against something
other than itself -- hand-derived golden vectors, closed forms, invariants
that the pages' definitions imply, or a library attention routine on special
cases that reduce to it.  CPU only."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_03_gb300 import synth
from tests import _util

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def bits(x):
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


# --------------------------------------------------------------- quantiser
@pytest.mark.parametrize("case", _util.read_quantizer_golden(), ids=lambda c: str(c[2][:2]))
def test_quantizer_golden(case):
    """Hand-derived vectors (CS336 lecture 10, int8 quantisation section)."""
    mode, scale, x, q = case
    xb = bits(x)
    assert np.array_equal(synth.bf16_bits_to_f32(xb), x, equal_nan=True), \
        "fixture inputs must be bf16-exact"
    if mode == "per_token":
        s = oracle.per_token_scale(xb)
        assert s.view(np.uint32) == scale.view(np.uint32), (s, scale)
    else:
        s = scale
    got = oracle.quantize(xb, float(s))
    assert np.array_equal(got, q), (got, q)


def _tiny_pool(kind="bf16", nb=4, P=16, hkv=2, D=8, alias=False):
    shape = (nb, P, hkv, D)
    if kind == "bf16":
        k = np.full(shape, synth.BF16_NAN, np.uint16)
    else:
        k = np.full(shape, synth.INT8_POISON, np.int8)
    v = None if alias else k.copy()
    ks = vs = None
    mode = oracle.SCALE_NONE
    if kind == "int8_token":
        ks = np.full(nb * P, np.nan, np.float32)
        vs = None if alias else ks.copy()
        mode = oracle.SCALE_PER_TOKEN
    elif kind == "int8_head":
        ks = np.full(hkv, 0.5, np.float32)
        vs = None if alias else np.full(hkv, 0.25, np.float32)
        mode = oracle.SCALE_PER_HEAD
    return oracle.OraclePool(k=k, v=v, k_scale=ks, v_scale=vs, scale_mode=mode)


def test_append_bf16_is_a_bit_copy_and_skips_padding():
    rng = np.random.default_rng(0)
    pool = _tiny_pool()
    k = bits(rng.standard_normal((3, 2, 8)))
    v = bits(rng.standard_normal((3, 2, 8)))
    slots = np.array([5, -1, 16 * 3 + 15], np.int64)
    oracle.append(k, v, slots, pool)
    assert np.array_equal(pool.k[0, 5], k[0]) and np.array_equal(pool.v[0, 5], v[0])
    assert np.array_equal(pool.k[3, 15], k[2]) and np.array_equal(pool.v[3, 15], v[2])
    # padding token and every other slot untouched
    untouched = np.ones((4, 16), bool)
    untouched[0, 5] = untouched[3, 15] = False
    assert np.all(pool.k[untouched] == synth.BF16_NAN)
    assert np.all(pool.v[untouched] == synth.BF16_NAN)


def test_append_alias_writes_k_only():
    pool = _tiny_pool(alias=True)
    k = bits(np.ones((1, 2, 8)))
    oracle.append(k, None, np.array([0], np.int64), pool)
    assert pool.v is None and np.array_equal(pool.k[0, 0], k[0])


def test_append_int8_per_token_scale_lands_at_slot():
    pool = _tiny_pool("int8_token")
    # token row amax = 63.5 over all heads -> scale 0.5 (closed form)
    x = np.zeros((1, 2, 8), np.float32)
    x[0, 1, 3] = -63.5
    x[0, 0, 0] = 1.25
    slots = np.array([16 * 2 + 7], np.int64)
    oracle.append(bits(x), bits(2 * x), slots, pool)
    assert pool.k_scale[39] == np.float32(0.5) and pool.v_scale[39] == np.float32(1.0)
    assert pool.k[2, 7, 1, 3] == -127 and pool.k[2, 7, 0, 0] == 2  # 2.5 -> 2 (half-even)
    assert pool.v[2, 7, 1, 3] == -127 and pool.v[2, 7, 0, 0] == 2  # 2.5/1 -> 2
    assert np.isnan(pool.k_scale[38]) and np.isnan(pool.k_scale[40])


def test_append_int8_per_head_uses_static_scale_and_saturates():
    pool = _tiny_pool("int8_head")  # k scale 0.5, v scale 0.25 per head
    x = np.zeros((1, 2, 8), np.float32)
    x[0, 0, 0], x[0, 1, 0], x[0, 1, 1] = 100.0, -0.75, 0.25
    oracle.append(bits(x), bits(x), np.array([0], np.int64), pool)
    assert pool.k[0, 0, 0, 0] == 127 and pool.k[0, 0, 1, 0] == -2 and pool.k[0, 0, 1, 1] == 0
    assert pool.v[0, 0, 0, 0] == 127 and pool.v[0, 0, 1, 0] == -3 and pool.v[0, 0, 1, 1] == 1


# --------------------------------------------------------------- attention
def _identity_workload(lens, hq, hkv, D, window=0, P=16, seed=0, alias=False):
    """Pool whose block table is the identity: sequence b owns blocks
    [b*nb, (b+1)*nb) in order, so its keys are a plain reshape of the pool."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    nb = max(1, max((l + P - 1) // P for l in lens))
    shape = (B * nb, P, hkv, D)
    k = bits(rng.standard_normal(shape))
    v = k if alias else bits(rng.standard_normal(shape))
    bt = np.arange(B * nb, dtype=np.int32).reshape(B, nb)
    q = bits(rng.standard_normal((B, hq, D)))
    pool = oracle.OraclePool(k=k, v=None if alias else v)
    return q, pool, bt, np.array(lens, np.int32), k, v, nb


def _sdpa_reference(q, k, v, lens, hq, window, scale, nb, P=16):
    """torch scaled_dot_product_attention (float64, CPU) on the dense keys of
    an identity-paged pool, with the band/causal mask as a boolean mask."""
    B = len(lens)
    hkv = k.shape[2]
    G = hq // hkv
    out = np.zeros((B, hq, k.shape[3]))
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        kd = synth.bf16_bits_to_f32(k[b * nb:(b + 1) * nb].reshape(nb * P, hkv, -1)[:L])
        vd = synth.bf16_bits_to_f32(v[b * nb:(b + 1) * nb].reshape(nb * P, hkv, -1)[:L])
        kt = torch.from_numpy(kd.astype(np.float64)).permute(1, 0, 2)  # [hkv, L, D]
        vt = torch.from_numpy(vd.astype(np.float64)).permute(1, 0, 2)
        kt = kt.repeat_interleave(G, dim=0)
        vt = vt.repeat_interleave(G, dim=0)
        qt = torch.from_numpy(synth.bf16_bits_to_f32(q[b]).astype(np.float64))[:, None, :]
        j = torch.arange(L)
        allowed = j <= L - 1
        if window > 0:
            allowed &= j >= L - 1 - window
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=allowed[None, None, :], scale=scale)
        out[b] = o[:, 0, :].numpy()
    return out


@pytest.mark.parametrize("window", [0, 5, 16, 40])
@pytest.mark.parametrize("hq,hkv", [(4, 2), (3, 3), (8, 1)])
def test_decode_matches_library_attention_on_identity_paging(window, hq, hkv):
    lens = [1, 7, 16, 17, 33, 64]
    q, pool, bt, sl, k, v, nb = _identity_workload(lens, hq, hkv, 32, window)
    scale = np.float32(1 / math.sqrt(32))
    got = oracle.decode(q, pool, bt, sl, hq, window, scale)
    ref = _sdpa_reference(q, k, v, sl, hq, window, float(scale), nb)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_single_key_returns_its_value_exactly():
    q, pool, bt, sl, k, v, nb = _identity_workload([1, 1], 4, 2, 16)
    got = oracle.decode(q, pool, bt, sl, 4, 0, 0.3)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(got[b, h], synth.bf16_bits_to_f32(v[b * nb, 0, h // 2]))


def test_gqa_maps_consecutive_query_heads_to_one_kv_head():
    """Lab5-Gemma4, GQA section: query heads share a KV head by repetition;
    with one key the output of head h is V of kv head h // G."""
    q, pool, bt, sl, k, v, nb = _identity_workload([1], 6, 3, 8)
    got = oracle.decode(q, pool, bt, sl, 6, 0, 1.0)
    vv = synth.bf16_bits_to_f32(v[0, 0])
    for h in range(6):
        assert np.array_equal(got[0, h], vv[h // 2])


def test_constant_value_rows_return_that_value():
    q, pool, bt, sl, k, v, nb = _identity_workload([5, 40, 33], 4, 2, 16, seed=3)
    c = bits(np.linspace(-2, 2, 16))
    pool.v[...] = c
    got = oracle.decode(q, pool, bt, sl, 4, 0, 0.25)
    np.testing.assert_allclose(got, np.broadcast_to(synth.bf16_bits_to_f32(c), got.shape),
                               rtol=0, atol=1e-14)


def test_zero_scale_gives_mean_of_window_values():
    lens, w = [30, 50], 9
    q, pool, bt, sl, k, v, nb = _identity_workload(lens, 2, 2, 8, window=w, seed=4)
    got = oracle.decode(q, pool, bt, sl, 2, w, 0.0)
    for b, L in enumerate(lens):
        vd = synth.bf16_bits_to_f32(v[b * nb:(b + 1) * nb].reshape(-1, 2, 8)[:L]).astype(np.float64)
        np.testing.assert_allclose(got[b], vd[L - 1 - w:L].mean(0), rtol=1e-13)


def test_window_endpoints_are_inclusive():
    """Lab5-Gemma4, sliding-window section: position i sees [i-w, i] -- w+1
    keys.  A key with an overwhelming score at i-w dominates the output; the
    same key at i-w-1 has no effect at all."""
    L, w, D = 40, 10, 8
    base = _identity_workload([L], 1, 1, D, seed=5)
    q, pool, bt, sl, k, v, nb = base
    q[...] = bits(np.eye(1, D))
    for j in range(L):
        pool.k[j // 16, j % 16, 0] = bits(np.zeros(D))
    ref = oracle.decode(q, pool, bt, sl, 1, w, 1.0)
    # inside: j = L-1-w
    j = L - 1 - w
    pool.k[j // 16, j % 16, 0] = bits(np.eye(1, D)[0] * 200.0)
    got = oracle.decode(q, pool, bt, sl, 1, w, 1.0)
    np.testing.assert_allclose(got[0, 0], synth.bf16_bits_to_f32(pool.v[j // 16, j % 16, 0]),
                               rtol=1e-12)
    # outside: move it to j-1
    pool.k[j // 16, j % 16, 0] = bits(np.zeros(D))
    pool.k[(j - 1) // 16, (j - 1) % 16, 0] = bits(np.eye(1, D)[0] * 200.0)
    got2 = oracle.decode(q, pool, bt, sl, 1, w, 1.0)
    np.testing.assert_array_equal(got2, ref)


def test_two_key_closed_form_golden():
    g = _util.read_two_key_golden()
    pool = oracle.OraclePool(k=np.zeros((1, 16, 1, 4), np.uint16),
                             v=np.zeros((1, 16, 1, 4), np.uint16))
    pool.k[0, 0, 0], pool.k[0, 1, 0] = bits(g["k0"]), bits(g["k1"])
    pool.v[0, 0, 0], pool.v[0, 1, 0] = bits(g["v0"]), bits(g["v1"])
    got = oracle.decode(bits(g["q"]).reshape(1, 1, 4), pool, np.zeros((1, 1), np.int32),
                        np.array([2], np.int32), 1, 0, float(g["softmax_scale"][0]))
    np.testing.assert_allclose(got[0, 0], g["y"], rtol=0, atol=1e-12)


def test_large_scores_do_not_overflow():
    q, pool, bt, sl, k, v, nb = _identity_workload([20], 1, 1, 8, seed=6)
    q[...] = bits(np.full((1, 1, 8), 100.0))
    j = 13
    pool.k[0, :, 0] = bits(np.zeros((16, 8)))
    pool.k[j // 16, j % 16, 0] = bits(np.full(8, 100.0))  # score 8e4 * scale
    got = oracle.decode(q, pool, bt, sl, 1, 0, 1.0)
    assert np.all(np.isfinite(got))
    np.testing.assert_array_equal(got[0, 0], synth.bf16_bits_to_f32(pool.v[0, j, 0]))


def test_window_at_least_length_equals_global():
    w = synth.make_workload(synth.shrink(synth.C2, batch=6, lens=("uniform", 1, 90), window=0,
                                         num_q_heads=4, num_kv_heads=2, head_dim=32))
    pool = _util.oracle_pool(w)
    g = oracle.decode(w.q, pool, w.block_table, w.seq_lens, 4, 0, 0.2)
    for win in (90, 200):
        s = oracle.decode(w.q, pool, w.block_table, w.seq_lens, 4, win, 0.2)
        np.testing.assert_array_equal(s, g)


def test_block_permutation_invariance():
    """Lab5-Gemma4, Paged Attention: paging changes where blocks live, not the
    result.  Permute the physical blocks and the table together."""
    w = synth.make_workload(synth.shrink(synth.C2, batch=5, lens=("uniform", 1, 100), window=23,
                                         num_q_heads=4, num_kv_heads=2, head_dim=32))
    pool = _util.oracle_pool(w)
    ref = oracle.decode(w.q, pool, w.block_table, w.seq_lens, 4, 23, 0.2)
    perm = np.random.default_rng(9).permutation(pool.k.shape[0])
    inv = np.argsort(perm)
    pool2 = oracle.OraclePool(k=np.ascontiguousarray(pool.k[perm]),
                              v=np.ascontiguousarray(pool.v[perm]))
    bt2 = np.where(w.block_table >= 0, inv[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    got = oracle.decode(w.q, pool2, bt2, w.seq_lens, 4, 23, 0.2)
    np.testing.assert_array_equal(got, ref)


def test_gqa_equals_explicit_kv_repetition():
    w = synth.make_workload(synth.shrink(synth.C2, batch=4, lens=("uniform", 1, 70), window=30,
                                         num_q_heads=8, num_kv_heads=2, head_dim=16))
    pool = _util.oracle_pool(w)
    ref = oracle.decode(w.q, pool, w.block_table, w.seq_lens, 8, 30, 0.3)
    rep = oracle.OraclePool(k=np.ascontiguousarray(np.repeat(pool.k, 4, axis=2)),
                            v=np.ascontiguousarray(np.repeat(pool.v, 4, axis=2)))
    got = oracle.decode(w.q, rep, w.block_table, w.seq_lens, 8, 30, 0.3)
    np.testing.assert_array_equal(got, ref)


def test_kv_alias_equals_separate_copy():
    w = synth.make_workload(synth.shrink(synth.C3, batch=3, lens=("uniform", 1, 80),
                                         num_q_heads=4, head_dim=16))
    pool = _util.oracle_pool(w)
    assert pool.v is None
    ref = oracle.decode(w.q, pool, w.block_table, w.seq_lens, 4, 0, 0.25)
    two = oracle.OraclePool(k=pool.k, v=pool.k.copy())
    got = oracle.decode(w.q, two, w.block_table, w.seq_lens, 4, 0, 0.25)
    np.testing.assert_array_equal(got, ref)


def test_shared_prefix_blocks_equal_private_copies():
    spec = synth.shrink(synth.C5_GLOBAL, batch=12, num_q_heads=4, head_dim=16,
                        lens=("uniform", 140, 200), shared_prefix_seqs=5)
    w = synth.make_workload(spec)
    pool = _util.oracle_pool(w)
    ref = oracle.decode(w.q, pool, w.block_table, w.seq_lens, 4, 0, 0.25)
    # give every sharing sequence private copies of the shared blocks
    bt = w.block_table.copy()
    k, v = list(pool.k), list(pool.v)
    shared = np.nonzero(w.layout.shared_seqs)[0]
    for b in shared[1:]:
        for i in range(spec.shared_prefix_blocks):
            k.append(pool.k[bt[b, i]].copy())
            v.append(pool.v[bt[b, i]].copy())
            bt[b, i] = len(k) - 1
    priv = oracle.OraclePool(k=np.ascontiguousarray(np.stack(k)), v=np.ascontiguousarray(np.stack(v)))
    got = oracle.decode(w.q, priv, bt, w.seq_lens, 4, 0, 0.25)
    np.testing.assert_array_equal(got, ref)


def test_int8_dequantises_after_gather_per_token():
    """tiniestgpt notes, section 5: int8 values times their token's scale.
    With scale 0 on the scores every allowed key weighs the same, so the
    output is the mean of the dequantised values."""
    codes = np.array([[1, -2, 3, 0], [5, 5, -5, 7], [-127, 0, 2, 1]], np.int8)
    scales = np.array([0.5, 0.25, 2.0], np.float32)
    bt = np.array([[1, 0]], np.int32)  # logical block 0 lives in physical block 1
    pool = _tiny_pool("int8_token", nb=2, hkv=1, D=4)
    phys = [(1, 0), (1, 1), (1, 2)]   # keys 0..2 -> block 1, offsets 0..2
    for i, (blk, off) in enumerate(phys):
        pool.k[blk, off, 0] = codes[i]
        pool.v[blk, off, 0] = codes[i]
        pool.k_scale[blk * 16 + off] = scales[i]
        pool.v_scale[blk * 16 + off] = scales[i]
    got = oracle.decode(bits(np.ones((1, 1, 4))), pool, bt, np.array([3], np.int32), 1, 0, 0.0)
    want = (codes.astype(np.float64) * scales[:, None]).mean(0)
    np.testing.assert_allclose(got[0, 0], want, rtol=1e-15)


def test_int8_dequantises_per_head():
    pool = _tiny_pool("int8_head", nb=1, hkv=2, D=4)  # k 0.5, v 0.25
    pool.v_scale[:] = np.array([0.25, 4.0], np.float32)
    codes = np.arange(2 * 2 * 4, dtype=np.int8).reshape(2, 2, 4) - 8
    pool.k[0, :2] = codes
    pool.v[0, :2] = codes
    got = oracle.decode(bits(np.ones((1, 4, 4))), pool, np.zeros((1, 1), np.int32),
                        np.array([2], np.int32), 4, 0, 0.0)
    for h in range(4):
        g = h // 2
        want = codes[:, g].astype(np.float64).mean(0) * pool.v_scale[g]
        np.testing.assert_allclose(got[0, h], want, rtol=1e-15)


def test_empty_sequence_gives_zeros():
    q, pool, bt, sl, k, v, nb = _identity_workload([0, 3], 2, 1, 8)
    got = oracle.decode(q, pool, bt, sl, 2, 0, 0.5)
    assert np.all(got[0] == 0) and np.all(np.isfinite(got[1]))


# ------------------------------------------------------- split-KV partials
def test_partial_over_whole_range_is_the_decode_and_logsumexp():
    q, pool, bt, sl, k, v, nb = _identity_workload([9, 40], 2, 1, 8, seed=11)
    full = oracle.decode(q, pool, bt, sl, 2, 0, 0.5)
    lse, o = oracle.partial(q, pool, bt, sl, 2, 0, 0.5, np.zeros(2), sl.astype(np.int64))
    np.testing.assert_array_equal(o, full)
    for b in range(2):
        L = sl[b]
        kd = synth.bf16_bits_to_f32(k[b * nb:(b + 1) * nb].reshape(-1, 1, 8)[:L, 0]).astype(np.float64)
        for h in range(2):
            qq = synth.bf16_bits_to_f32(q[b, h]).astype(np.float64)
            s = torch.from_numpy(0.5 * kd @ qq)
            assert lse[b, h] == pytest.approx(float(torch.logsumexp(s, 0)), rel=1e-13)


def test_single_key_partial_lse_is_the_score():
    q, pool, bt, sl, k, v, nb = _identity_workload([5], 1, 1, 8, seed=12)
    lse, o = oracle.partial(q, pool, bt, sl, 1, 0, 0.5, np.array([2]), np.array([3]))
    s = 0.5 * float(synth.bf16_bits_to_f32(q[0, 0]).astype(np.float64)
                    @ synth.bf16_bits_to_f32(k[0, 2, 0]).astype(np.float64))
    assert lse[0, 0] == pytest.approx(s, rel=1e-14)
    np.testing.assert_array_equal(o[0, 0], synth.bf16_bits_to_f32(v[0, 2, 0]))


@pytest.mark.parametrize("nsplit", [2, 3, 7])
def test_split_partials_combine_to_the_full_decode(nsplit):
    """Merging (lse, o) states of disjoint key ranges gives the single-pass
    result (associativity of the online-softmax update)."""
    q, pool, bt, sl, k, v, nb = _identity_workload([70, 41], 4, 2, 16, window=50, seed=13)
    full = oracle.decode(q, pool, bt, sl, 4, 50, 0.3)
    cuts = [np.linspace(0, L, nsplit + 1).astype(np.int64) for L in sl]
    parts = [oracle.partial(q, pool, bt, sl, 4, 50, 0.3,
                            np.array([c[i] for c in cuts]), np.array([c[i + 1] for c in cuts]))
             for i in range(nsplit)]
    for b in range(2):
        for h in range(4):
            y, _ = oracle.lse_combine(np.array([p[0][b, h] for p in parts]),
                                      np.stack([p[1][b, h] for p in parts]))
            np.testing.assert_allclose(y, full[b, h], rtol=1e-12, atol=1e-14)


def test_combine_ignores_empty_partials():
    o = np.array([[1.0, 2.0], [5.0, 6.0]])
    y, L = oracle.lse_combine(np.array([0.7, -np.inf]), o)
    np.testing.assert_array_equal(y, o[0])
    assert L == 0.7
    y, L = oracle.lse_combine(np.array([-np.inf, -np.inf]), o)
    assert np.all(y == 0) and L == -np.inf
    # equal weights: log(2) apart -> weights 2/3, 1/3
    y, L = oracle.lse_combine(np.array([math.log(2.0), 0.0]), o)
    np.testing.assert_allclose(y, (2 * o[0] + o[1]) / 3, rtol=1e-15)
    assert L == pytest.approx(math.log(3.0), rel=1e-15)


def test_oracle_threads_do_not_change_results():
    w = synth.make_workload(synth.shrink(synth.C2, batch=8, lens=("uniform", 1, 120), window=40,
                                         num_q_heads=4, num_kv_heads=2, head_dim=32))
    pool = _util.oracle_pool(w)
    a = _util.oracle_decode(w, pool, num_threads=1)
    b = _util.oracle_decode(w, pool, num_threads=4)
    np.testing.assert_array_equal(a, b)


# --------------------------------------------------------------- byte model
def test_kv_cache_bytes_worked_example():
    """CS336 lecture 10, KV-cache size section: n_kv=64, d_h=128, bf16 gives
    32 KiB per token per layer; S=100,000 tokens and L=80 layers give about
    244 GiB (262 GB)."""
    from paged_kv_decode_03_gb300 import bytes_model as bm
    assert bm.kv_cache_bytes(1, 1, 64, 128, 2) == 32 * 1024
    total = bm.kv_cache_bytes(80, 100_000, 64, 128, 2)
    assert round(total / 2**30) == 244 and round(total / 1e9) == 262


def test_decode_bytes_counts_window_keys_once():
    from paged_kv_decode_03_gb300 import bytes_model as bm
    spec = synth.shrink(synth.C2, batch=3, lens=("fixed", (1, 1025, 5000)))
    w = synth.make_workload(spec)
    d = bm.decode_bytes(spec, w.seq_lens, w.block_table)
    assert d["keys"] == 1 + 1025 + 1025
    assert d["kv"] == d["unique_keys"] * 8 * 256 * 2 * 2
    # shared prefix blocks are read once
    g = synth.shrink(synth.C5_GLOBAL, batch=10, lens=("uniform", 140, 200), shared_prefix_seqs=4)
    wg = synth.make_workload(g)
    dg = bm.decode_bytes(g, wg.seq_lens, wg.block_table)
    assert dg["keys"] - dg["unique_keys"] == 3 * 8 * 16


def test_bytes_per_key_of_the_workloads():
    """Per-key algorithmic bytes: K and V rows of every kv head (one tensor
    when K == V), plus the int8 per-token scales; per-head scales count once
    per launch."""
    from paged_kv_decode_03_gb300 import bytes_model as bm
    assert bm.bytes_per_key(8, 256, "bf16", False) == 8192        # Gemma4 sliding layer
    assert bm.bytes_per_key(1, 256, "bf16", True) == 512          # Gemma4 global, K == V
    assert bm.bytes_per_key(40, 128, "int8_token", False) == 10240 + 8  # Llama-2-13B-like
    assert bm.bytes_per_key(8, 256, "int8_head", False) == 4096
    spec = synth.shrink(synth.C5_SLIDING, batch=2, lens=("fixed", (20, 40)),
                        shared_prefix_seqs=0)
    w = synth.make_workload(spec)
    d = bm.decode_bytes(spec, w.seq_lens, w.block_table)
    assert d["kv"] == d["unique_keys"] * 4096 + 2 * spec.num_kv_heads * 4
    assert d["q"] == 2 * spec.num_q_heads * spec.head_dim * 2
