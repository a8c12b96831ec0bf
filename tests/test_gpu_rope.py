"""RoPE fused with the append (paged_rope_cos_sin_table, paged_kv_append_rope)
against the oracle: the (cos, sin) table entry by entry, the rotated q and
every pool byte (bf16 rows, int8 codes, per-token scales) bit for bit, and a
decode over a pool filled through the fused append on the Gemma4 global
layer's shape (p-RoPE, K and V one tensor) and an int8 sliding layer.

The rotation follows RoFormer (Su et al., section 3.2) with p-RoPE's
truncation (Barbero et al.); the theta tables are the caller's, here
RoFormer's base^(-2i/D).  A table entry whose fp64 cosine or sine lies within
a few fp64 ulps of an fp32 rounding midpoint may round either way on two
faithful math libraries; the oracle flags such entries and tokens at those
positions are compared by value instead of by bits (none are expected).
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import paged_kv_decode_03_gb300 as pkv  # noqa: E402
from paged_kv_decode_03_gb300 import synth  # noqa: E402
from tests import _util  # noqa: E402

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
BAD_POSITION = 32  # PKV_DEV_BAD_POSITION


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    pkv.device_status(clear=True)


from tests import _gpu  # noqa: E402


def roformer_theta(head_dim: int, base: float, pairs: int) -> np.ndarray:
    """The first ``pairs`` of theta_i = base^(-2i/D) (RoFormer section 3.2)."""
    return (base ** (-2.0 * np.arange(head_dim // 2) / head_dim))[:pairs].astype(np.float64)


def tables(theta: np.ndarray, npos: int):
    """(device table, oracle table, oracle ambiguity flags)."""
    td = pkv.paged_rope_cos_sin_table(torch.from_numpy(theta).cuda(), npos)
    to, amb = oracle.rope_table(theta, npos)
    return td, to, amb


@pytest.mark.parametrize("head_dim,base,pairs,npos", [
    (256, 1e6, 32, 70000), (256, 1e4, 128, 9000), (128, 1e4, 64, 20000), (64, 5e5, 7, 3000)])
def test_rope_table_matches_oracle(head_dim, base, pairs, npos):
    theta = roformer_theta(head_dim, base, pairs)
    td, to, amb = tables(theta, npos)
    got = td.cpu().numpy()
    assert amb.mean() < 1e-5
    same = got.view(np.uint32) == to.view(np.uint32)
    assert same.all(axis=2)[~amb].all()
    # flagged entries: either neighbour of the midpoint
    diff = np.abs(got.view(np.int32).astype(np.int64) - to.view(np.int32).astype(np.int64))
    assert (diff[amb] <= 1).all()


def _pool(kv: str, alias: bool, nb: int, hkv: int, D: int, rng):
    shape = (nb, 16, hkv, D)
    if kv == "bf16":
        k = np.full(shape, synth.BF16_NAN, np.uint16)
        return dict(k=k, v=None if alias else k.copy(), ks=None, vs=None, mode=oracle.SCALE_NONE)
    k = np.full(shape, synth.INT8_POISON, np.int8)
    v = None if alias else k.copy()
    if kv == "int8_token":
        ks = np.full(nb * 16, synth.F32_NAN, np.float32)
        return dict(k=k, v=v, ks=ks, vs=None if alias else ks.copy(), mode=oracle.SCALE_PER_TOKEN)
    ks = (np.float32(4.0) * (0.5 + 0.25 * np.arange(hkv, dtype=np.float32)) / np.float32(127.0))
    return dict(k=k, v=v, ks=ks.astype(np.float32), vs=None if alias else (ks * 0.75).astype(np.float32),
                mode=oracle.SCALE_PER_HEAD)


def _dev_pool(a) -> pkv.PagedKVPool:
    conv = _gpu.to_dev_bits if a["k"].dtype == np.uint16 else _gpu.to_dev
    mode = {oracle.SCALE_NONE: pkv.SCALE_NONE, oracle.SCALE_PER_TOKEN: pkv.SCALE_PER_TOKEN,
            oracle.SCALE_PER_HEAD: pkv.SCALE_PER_HEAD}[a["mode"]]
    return pkv.PagedKVPool(k=conv(a["k"]), v=None if a["v"] is None else conv(a["v"]),
                           k_scale=None if a["ks"] is None else _gpu.to_dev(a["ks"]),
                           v_scale=None if a["vs"] is None else _gpu.to_dev(a["vs"]),
                           scale_mode=mode)


def _ora_pool(a) -> oracle.OraclePool:
    c = lambda x: None if x is None else x.copy()  # noqa: E731
    return oracle.OraclePool(k=c(a["k"]), v=c(a["v"]), k_scale=c(a["ks"]), v_scale=c(a["vs"]),
                             scale_mode=a["mode"])


def _bf16(rng, shape, sigma=1.0):
    return synth.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma))


def _compare(gp, op, q_out_d, q_out_o, pos, slots, amb, npos):
    """q rows and pool rows bit for bit, except tokens at flagged positions."""
    flagged = np.array([0 <= p < npos and bool(amb[p].any()) for p in pos])
    assert flagged.mean() < 0.05
    if q_out_o is not None:
        got = q_out_d.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got[~flagged], q_out_o[~flagged]), "rotated q differs"
    k, v, ks, vs = _gpu.pool_to_host(gp)
    skip = np.zeros(op.k.shape[0] * 16, bool)
    skip[slots[flagged & (slots >= 0)]] = True

    def rows(a):
        return a.reshape(skip.shape[0], -1)[~skip]
    assert np.array_equal(rows(k), rows(op.k)), "K pool differs"
    if op.v is not None:
        assert np.array_equal(rows(v), rows(op.v)), "V pool differs"
    if op.scale_mode == oracle.SCALE_PER_TOKEN:
        assert np.array_equal(ks[~skip].view(np.uint32), op.k_scale[~skip].view(np.uint32))
        if op.v_scale is not None:
            assert np.array_equal(vs[~skip].view(np.uint32), op.v_scale[~skip].view(np.uint32))


CASES = [  # kv, alias, head_dim, H_q, H_kv, layout, rotated pairs
    ("bf16", False, 128, 8, 2, pkv.ROPE_HALVES, 64),
    ("bf16", True, 256, 16, 1, pkv.ROPE_HALVES, 32),
    ("bf16", False, 64, 4, 4, pkv.ROPE_HALVES, 0),
    ("bf16", False, 256, 8, 1, pkv.ROPE_INTERLEAVED, 128),
    ("int8_token", False, 128, 4, 4, pkv.ROPE_INTERLEAVED, 64),
    ("int8_token", True, 64, 8, 2, pkv.ROPE_INTERLEAVED, 5),
    ("int8_token", False, 256, 16, 8, pkv.ROPE_HALVES, 13),
    ("int8_head", False, 256, 16, 8, pkv.ROPE_HALVES, 128),
    ("int8_head", True, 128, 8, 2, pkv.ROPE_HALVES, 16),
]


@pytest.mark.parametrize("kv,alias,D,hq,hkv,layout,pairs", CASES)
def test_append_rope_matches_oracle(kv, alias, D, hq, hkv, layout, pairs):
    rng = np.random.default_rng(D * 7 + hq * 3 + pairs + (11 if alias else 0))
    T, nb, npos = 45, 8, 40000
    sigma = (0.5 + 0.25 * np.arange(hkv, dtype=np.float32))[None, :, None] if kv == "int8_head" else 1.0
    q = _bf16(rng, (T, hq, D))
    k = _bf16(rng, (T, hkv, D), sigma)
    v = None if alias else _bf16(rng, (T, hkv, D), sigma)
    slots = rng.choice(nb * 16, T, replace=False).astype(np.int64)
    slots[[3, 17]] = -1
    pos = rng.integers(0, npos, T).astype(np.int64)
    pos[[0, 1, 2, 9]] = [0, 1, npos - 1, -1]
    theta = roformer_theta(D, 10000.0, pairs)
    td, to, amb = tables(theta, npos)
    a = _pool(kv, alias, nb, hkv, D, rng)
    gp, op = _dev_pool(a), _ora_pool(a)
    q_d = _gpu.to_dev_bits(q)
    q_out = torch.empty_like(q_d)
    pkv.paged_kv_append_rope(q_d, q_out, _gpu.to_dev_bits(k), None if v is None else _gpu.to_dev_bits(v),
                             _gpu.to_dev(pos), _gpu.to_dev(slots), gp, td, layout)
    q_out_o, rc = oracle.append_rope(q, k, v, pos, slots, op, to, layout)
    assert rc == 0
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) == 0
    _compare(gp, op, q_out, q_out_o, pos, slots, amb, npos)
    # the padding token's q row passes unchanged
    assert np.array_equal(q_out[9].view(torch.int16).cpu().numpy().view(np.uint16), q[9])


def test_append_rope_in_place_and_without_q():
    rng = np.random.default_rng(3)
    T, hq, hkv, D, npos, pairs = 20, 8, 2, 128, 1000, 64
    q = _bf16(rng, (T, hq, D))
    k = _bf16(rng, (T, hkv, D))
    slots = rng.choice(64, T, replace=False).astype(np.int64)
    pos = rng.integers(0, npos, T).astype(np.int64)
    theta = roformer_theta(D, 10000.0, pairs)
    td, to, amb = tables(theta, npos)
    a = _pool("bf16", True, 4, hkv, D, rng)
    gp, op = _dev_pool(a), _ora_pool(a)
    q_d = _gpu.to_dev_bits(q)
    pkv.paged_kv_append_rope(q_d, q_d, _gpu.to_dev_bits(k), None, _gpu.to_dev(pos),
                             _gpu.to_dev(slots), gp, td)
    q_out_o, _ = oracle.append_rope(q, k, None, pos, slots, op, to)
    torch.cuda.synchronize()
    _compare(gp, op, q_d, q_out_o, pos, slots, amb, npos)
    # k only: the same pool bytes
    gp2, op2 = _dev_pool(a), _ora_pool(a)
    pkv.paged_kv_append_rope(None, None, _gpu.to_dev_bits(k), None, _gpu.to_dev(pos),
                             _gpu.to_dev(slots), gp2, td)
    oracle.append_rope(None, k, None, pos, slots, op2, to)
    torch.cuda.synchronize()
    _compare(gp2, op2, None, None, pos, slots, amb, npos)


def test_append_rope_position_past_the_table():
    rng = np.random.default_rng(4)
    T, hq, hkv, D, npos, pairs = 6, 4, 2, 64, 100, 32
    q = _bf16(rng, (T, hq, D))
    k = _bf16(rng, (T, hkv, D))
    v = _bf16(rng, (T, hkv, D))
    slots = np.arange(T, dtype=np.int64) * 3
    pos = np.array([5, 100, 99, 1000, 0, 42], np.int64)
    theta = roformer_theta(D, 10000.0, pairs)
    td, to, amb = tables(theta, npos)
    a = _pool("int8_token", False, 2, hkv, D, rng)
    gp, op = _dev_pool(a), _ora_pool(a)
    q_d = _gpu.to_dev_bits(q)
    q_out = torch.empty_like(q_d)
    pkv.device_status(clear=True)
    pkv.paged_kv_append_rope(q_d, q_out, _gpu.to_dev_bits(k), _gpu.to_dev_bits(v), _gpu.to_dev(pos),
                             _gpu.to_dev(slots), gp, td)
    q_out_o, rc = oracle.append_rope(q, k, v, pos, slots, op, to)
    assert rc == oracle.E_POS
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) & BAD_POSITION
    _compare(gp, op, q_out, q_out_o, pos, slots, amb, npos)
    got = q_out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got[[1, 3]], q[[1, 3]])


def _rope_workload(w, theta, npos, layout):
    """Fill a pool with the workload's history and step tokens through the
    fused append (history positions hist_pos, step tokens seq_lens - 1), on
    the device and in the oracle; returns (device pool, oracle pool, device
    q_out, oracle q_out, flagged positions)."""
    td, to, amb = tables(theta, npos)
    gp = _gpu.device_pool(w)
    spec = w.spec
    k0, v0, ks0, vs0 = synth.empty_pool_arrays(spec, w.layout)
    mode = {"bf16": oracle.SCALE_NONE, "int8_token": oracle.SCALE_PER_TOKEN,
            "int8_head": oracle.SCALE_PER_HEAD}[spec.kv]
    if spec.kv == "int8_head":
        ks0 = w.k_head_scale.copy()
        vs0 = None if spec.alias else w.v_head_scale.copy()
    op = oracle.OraclePool(k=k0, v=v0, k_scale=ks0, v_scale=vs0, scale_mode=mode,
                           ring_blocks=spec.ring_blocks)
    hist_slots, new_slots = _util.oracle_slots(w, op)
    B = len(w.seq_lens)
    new_pos = w.seq_lens.astype(np.int64) - 1
    chunk = 1 << 16
    for s in range(0, len(w.hist_pos), chunk):
        e = min(len(w.hist_pos), s + chunk)
        pkv.paged_kv_append_rope(None, None, _gpu.to_dev_bits(w.hist_k[s:e]),
                                 None if w.hist_v is None else _gpu.to_dev_bits(w.hist_v[s:e]),
                                 _gpu.to_dev(w.hist_pos[s:e].astype(np.int64)),
                                 _gpu.to_dev(hist_slots[s:e]), gp, td, layout)
    oracle.append_rope(None, w.hist_k, w.hist_v, w.hist_pos.astype(np.int64), hist_slots, op, to,
                       layout)
    q_d = _gpu.to_dev_bits(w.q)
    q_out = torch.empty_like(q_d)
    pkv.paged_kv_append_rope(q_d, q_out, _gpu.to_dev_bits(w.new_k),
                             None if w.new_v is None else _gpu.to_dev_bits(w.new_v),
                             _gpu.to_dev(new_pos), _gpu.to_dev(new_slots), gp, td, layout)
    q_out_o, rc = oracle.append_rope(w.q, w.new_k, w.new_v, new_pos, new_slots, op, to, layout)
    assert rc == 0
    assert B == q_out_o.shape[0]
    return gp, op, q_out, q_out_o, amb


@pytest.mark.parametrize("which", ["c5g_full", "c5s_small"])
def test_decode_after_fused_rope_append(which):
    """Decode over a pool written by the fused append, with the rotated q:
    the Gemma4 global layer at full size (p-RoPE on a quarter of the pairs,
    K and V one tensor) and the int8 per-head sliding layer (full RoPE)."""
    if which == "c5g_full":
        spec, base, pairs = synth.C5_GLOBAL, 1e6, synth.C5_GLOBAL.head_dim // 8
    else:
        spec, base, pairs = synth.shrink(synth.C5_SLIDING, batch=24), 1e4, synth.C5_SLIDING.head_dim // 2
    w = synth.make_workload(spec)
    npos = int(w.seq_lens.max()) + 1
    theta = roformer_theta(spec.head_dim, base, pairs)
    gp, op, q_out, q_out_o, amb = _rope_workload(w, theta, npos, pkv.ROPE_HALVES)
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) == 0
    assert not amb.any()
    got_q = q_out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got_q, q_out_o)
    k, v, ks, vs = _gpu.pool_to_host(gp)
    assert np.array_equal(k, op.k)
    if op.v is not None:
        assert np.array_equal(v, op.v)
    out = torch.empty(q_out.shape, dtype=torch.bfloat16, device="cuda")
    pkv.paged_decode_attention(q_out, gp, _gpu.to_dev(w.block_table), _gpu.to_dev(w.seq_lens),
                               spec.window, np.float32(spec.softmax_scale), out,
                               int(w.seq_lens.max()))
    rng = np.random.default_rng(1)
    B, Hq = w.q.shape[:2]
    rows = np.array(sorted({(int(rng.integers(B)), int(rng.integers(Hq))) for _ in range(40)}),
                    np.int32)
    ref = oracle.decode(q_out_o, op, w.block_table, w.seq_lens, spec.num_q_heads, spec.window,
                        np.float32(spec.softmax_scale), rows=rows)
    got = _gpu.out_to_f64(out)[rows[:, 0], rows[:, 1]]
    assert _gpu.max_abs_err(got, ref) <= BF16_TOL
