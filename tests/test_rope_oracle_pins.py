"""Pins of the oracle's rotary position embedding (RoPE fused with the append).

The pages name p-RoPE on Gemma4's global layers (Lab5-Gemma4, model overview)
without a formula; the oracle follows RoFormer (Su et al., section 3.2 and the
element-wise form of section 3.4.2) with p-RoPE's truncation of the lowest
frequencies (Barbero et al., "Round and Round We Go!").  Nothing here compares
the oracle with itself: the pins are decimal values of cos and sin, hand-worked
rotations that fix the sign and the pairing, invariants of rotations (norms,
composition, dependence on relative position only), the fp64 rotation as an
error bound on the rounded one, and torch's fp32 -> bf16 conversion.
"""
import math

import numpy as np
import pytest
import torch

import oracle

# cos and sin of 1, 2, 3 and 0.02 radians (tables of the circular functions)
COS1, SIN1 = 0.54030230586813971740, 0.84147098480789650665
COS2, SIN2 = -0.41614683654714238700, 0.90929742682568169540
COS3, SIN3 = -0.98999249660044545727, 0.14112000805986722210
COS002, SIN002 = 0.99980000666657777841, 0.01999866669333307937


def roformer_theta(head_dim: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/D), i < D/2 (RoFormer section 3.2)."""
    return base ** (-2.0 * np.arange(head_dim // 2) / head_dim)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    return oracle.bf16_bits_to_f64(bits)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    # exact midpoints between neighbouring bf16 numbers (ties) and their
    # neighbours, large and tiny magnitudes, signed zeros, infinities
    base = (rng.integers(0, 1 << 15, 2000, dtype=np.uint32) << 16) | 0x8000
    ties = base.view(np.float32)
    extra = np.array([0.0, -0.0, np.inf, -np.inf, 3.3e38, -3.39e38, 1e-40, -1e-42,
                      1.00390625, 1.01171875, -1.00390625], np.float32)
    x = np.concatenate([x, ties[np.isfinite(ties)], extra])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(got, want)


def test_table_closed_forms():
    table, amb = oracle.rope_table(np.array([1.0, 0.01]), 4)
    want = np.array([[1.0, 0.0], [COS1, SIN1], [COS2, SIN2], [COS3, SIN3]], np.float32)
    np.testing.assert_array_equal(table[:, 0, :], want)
    np.testing.assert_array_equal(table[2, 1, :], np.array([COS002, SIN002], np.float32))
    assert not amb.any()


def test_table_on_the_unit_circle():
    theta = roformer_theta(256, 1e6)
    table, _ = oracle.rope_table(theta, 3000)
    r = table[..., 0].astype(np.float64) ** 2 + table[..., 1].astype(np.float64) ** 2
    assert np.abs(r - 1.0).max() <= 2.0 ** -22
    np.testing.assert_array_equal(table[0], np.tile(np.array([1.0, 0.0], np.float32), (128, 1)))


def test_midpoint_flag():
    # cos of acos(v) for v halfway between two fp32 numbers below 1 is flagged;
    # one a quarter of an fp32 step away from the midpoint is not
    mid = 1.0 - 1.5 * 2.0 ** -24
    _, amb = oracle.rope_table(np.array([math.acos(mid), math.acos(0.75 + 2.0 ** -26)]), 2)
    assert amb[1, 0] and not amb[1, 1] and not amb[0].any()


@pytest.mark.parametrize("layout", [oracle.ROPE_HALVES, oracle.ROPE_INTERLEAVED])
def test_exact_rotation_hand_examples(layout):
    theta = np.array([1.0, 0.01])
    e = np.eye(4)
    y = [oracle.rope_exact(e[d], 2.0, theta, 2, layout) for d in range(4)]
    if layout == oracle.ROPE_HALVES:  # pairs (0, 2) and (1, 3)
        want = [[COS2, 0, SIN2, 0], [0, COS002, 0, SIN002],
                [-SIN2, 0, COS2, 0], [0, -SIN002, 0, COS002]]
    else:  # pairs (0, 1) and (2, 3)
        want = [[COS2, SIN2, 0, 0], [-SIN2, COS2, 0, 0],
                [0, 0, COS002, SIN002], [0, 0, -SIN002, COS002]]
    np.testing.assert_allclose(np.array(y), np.array(want), rtol=0, atol=1e-15)


@pytest.mark.parametrize("layout", [oracle.ROPE_HALVES, oracle.ROPE_INTERLEAVED])
def test_exact_rotation_invariants(layout):
    rng = np.random.default_rng(5)
    D = 64
    theta = roformer_theta(D, 10000.0)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    for pairs in (0, 8, 32):
        # each pair keeps its length; dims past the rotated pairs are untouched
        y = oracle.rope_exact(q, 123.0, theta, pairs, layout)
        if layout == oracle.ROPE_HALVES:
            ia, ib = np.arange(D // 2), np.arange(D // 2) + D // 2
        else:
            ia, ib = np.arange(0, D, 2), np.arange(1, D, 2)
        np.testing.assert_allclose(y[ia] ** 2 + y[ib] ** 2, q[ia] ** 2 + q[ib] ** 2, rtol=1e-13)
        np.testing.assert_array_equal(y[ia[pairs:]], q[ia[pairs:]])
        np.testing.assert_array_equal(y[ib[pairs:]], q[ib[pairs:]])
        # position 0 is the identity; turning by m1 then m2 is turning by m1 + m2
        np.testing.assert_array_equal(oracle.rope_exact(q, 0.0, theta, pairs, layout), q)
        two = oracle.rope_exact(oracle.rope_exact(q, 17.0, theta, pairs, layout), 40.0, theta,
                                pairs, layout)
        np.testing.assert_allclose(two, oracle.rope_exact(q, 57.0, theta, pairs, layout),
                                   rtol=0, atol=1e-12)
        # q.k after rotation depends only on the distance of the positions
        def score(m, n):
            return float(oracle.rope_exact(q, m, theta, pairs, layout) @
                         oracle.rope_exact(k, n, theta, pairs, layout))
        s0 = score(100.0, 37.0)
        for shift in (1.0, 250.0, 4096.0):
            assert abs(score(100.0 + shift, 37.0 + shift) - s0) <= 1e-10 * (1 + abs(s0))
        if pairs:
            assert abs(score(100.0, 38.0) - s0) > 1e-6


@pytest.mark.parametrize("base,pairs", [(10000.0, 64), (1e6, 16), (10000.0, 5)])
@pytest.mark.parametrize("layout", [oracle.ROPE_HALVES, oracle.ROPE_INTERLEAVED])
def test_rounded_rotation_within_half_a_bf16_step_of_exact(base, pairs, layout):
    """The stored rotation (fp32 table, fp32 fused multiply-adds, bf16 round to
    nearest) lies within half a bf16 step of the exact rotation, widened by the
    fp32 error bound; truncation, a dropped term or a sign error does not."""
    rng = np.random.default_rng(int(base) % 97 + pairs)
    T, H, D = 24, 3, 128
    theta = roformer_theta(D, base)[:pairs]
    npos = 70000
    pos = rng.integers(0, npos, T)
    pos[:3] = [0, 1, npos - 1]
    x = torch.randn(T, H, D).mul(2.0).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    table, _ = oracle.rope_table(theta, npos)
    y, rc = oracle.rope(x, pos, table, layout)
    assert rc == 0
    xv, yv = bf16_value(x), bf16_value(y)
    if layout == oracle.ROPE_HALVES:
        partner = np.concatenate([np.arange(D // 2) + D // 2, np.arange(D // 2)])
    else:
        partner = np.arange(D) ^ 1
    for t in range(T):
        for h in range(H):
            e = oracle.rope_exact(xv[t, h], float(pos[t]), theta, pairs, layout)
            eps = 3.5 * 2.0 ** -24 * (np.abs(xv[t, h]) + np.abs(xv[t, h][partner]))
            mag = np.abs(e) + eps
            step = np.exp2(np.floor(np.log2(np.maximum(mag, 2.0 ** -126))) - 7)
            assert np.all(np.abs(yv[t, h] - e) <= 0.5 * step + eps), (t, h)


def test_rope_padding_and_positions_past_the_table():
    rng = np.random.default_rng(3)
    x = rng.integers(0, 1 << 14, (4, 2, 8)).astype(np.uint16)
    table, _ = oracle.rope_table(roformer_theta(8, 10000.0), 10)
    y, rc = oracle.rope(x, np.array([-1, 3, 10, 9]), table)
    assert rc == oracle.E_POS
    np.testing.assert_array_equal(y[0], x[0])
    np.testing.assert_array_equal(y[2], x[2])
    assert not np.array_equal(y[1], x[1]) and not np.array_equal(y[3], x[3])


def test_append_rope_without_rotated_pairs_is_the_append():
    """With no rotated pairs the fused operation is the (pinned) append; a
    padding position appends nothing."""
    rng = np.random.default_rng(8)
    T, Hkv, D, nb = 6, 2, 16, 4
    k = rng.integers(0, 1 << 14, (T, Hkv, D)).astype(np.uint16)
    v = rng.integers(0, 1 << 14, (T, Hkv, D)).astype(np.uint16)
    slots = np.array([3, 17, 40, 5, 63, 20], np.int64)
    pos = np.array([0, 5, 9, -1, 2, 7], np.int64)
    table, _ = oracle.rope_table(np.zeros(0), 10)
    p1 = oracle.OraclePool(k=np.zeros((nb, 16, Hkv, D), np.int8), v=np.zeros((nb, 16, Hkv, D), np.int8),
                           k_scale=np.zeros(nb * 16, np.float32), v_scale=np.zeros(nb * 16, np.float32),
                           scale_mode=oracle.SCALE_PER_TOKEN)
    p2 = oracle.OraclePool(k=p1.k.copy(), v=p1.v.copy(), k_scale=p1.k_scale.copy(),
                           v_scale=p1.v_scale.copy(), scale_mode=oracle.SCALE_PER_TOKEN)
    q_out, rc = oracle.append_rope(k, k, v, pos, slots, p1, table)
    assert rc == 0
    np.testing.assert_array_equal(q_out, k)
    oracle.append(k, v, np.where(pos >= 0, slots, -1), p2)
    for a, b in ((p1.k, p2.k), (p1.v, p2.v), (p1.k_scale, p2.k_scale), (p1.v_scale, p2.v_scale)):
        np.testing.assert_array_equal(a, b)
    assert not p1.k.reshape(-1, Hkv, D)[5].any()
