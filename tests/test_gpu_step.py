"""The six-layer continuous-batching step through paged_decode_step: five
int8 per-head sliding layers and one bf16 global layer over one ragged
layout with shared prefix blocks (CS336 lecture 10, local/global mix;
tiniestgpt notes, prefix caching), each layer appending one token per
sequence and then decoding.  The whole step is captured once as a CUDA
graph over static buffers and replayed (tiniestgpt notes, section 8).
Every layer's pool must equal the oracle's append bit for bit and every
layer's output must match the oracle's decode (all rows on the small step,
sampled rows at full size)."""
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


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    pkv.device_status(clear=True)
    yield
    torch.cuda.synchronize()


from tests import _gpu  # noqa: E402


def _rope_tables(layers, npos):
    """Per layer (device table, oracle table, flags): RoFormer's theta =
    base^(-2i/D); every pair with base 10^4 on sliding layers, p-RoPE on the
    first quarter of the pairs with base 10^6 on the global layer."""
    out = []
    for w in layers:
        D = w.spec.head_dim
        base, pairs = (1e4, D // 2) if w.spec.window else (1e6, D // 8)
        theta = (base ** (-2.0 * np.arange(D // 2) / D))[:pairs].astype(np.float64)
        td = pkv.paged_rope_cos_sin_table(torch.from_numpy(theta).cuda(), npos)
        to, amb = oracle.rope_table(theta, npos)
        out.append((td, to, amb))
    return out


def _captured_step(layers, rope=None):
    """Device pools with each layer's history, static step buffers, and the
    whole step (every layer's append + decode) captured in one graph.  With
    ``rope`` (per layer: device table, ...) each layer rotates q into its own
    q_rotated buffer and its new k before storing it."""
    w0 = layers[0]
    pools = []
    hist_dev = {}
    for w in layers:
        gp = _gpu.device_pool(w)
        key = id(w.hist_k)
        if key not in hist_dev:  # layers sharing history values upload them once
            hist_dev[key] = [(_gpu.to_dev_bits(w.hist_k[s:s + (1 << 16)]),
                              None if w.hist_v is None else _gpu.to_dev_bits(w.hist_v[s:s + (1 << 16)]),
                              _gpu.to_dev(w.hist_slots[s:s + (1 << 16)]))
                             for s in range(0, len(w.hist_slots), 1 << 16)]
        for k, v, sl in hist_dev[key]:
            pkv.paged_kv_append(k, v, sl, gp)
        pools.append(gp)
    del hist_dev
    slots = _gpu.to_dev(w0.new_slots)
    bt = _gpu.to_dev(w0.block_table)
    lens = _gpu.to_dev(w0.seq_lens)
    max_len = int(w0.seq_lens.max())
    dl = []
    for i, (w, gp) in enumerate(zip(layers, pools)):
        q = _gpu.to_dev_bits(w.q)
        extra = {}
        if rope is not None:
            extra = dict(rope_table=rope[i][0], rope_layout=pkv.ROPE_HALVES,
                         q_rotated=torch.empty_like(q))
        dl.append(pkv.DecodeLayer(pool=gp, q=q, k_new=_gpu.to_dev_bits(w.new_k),
                                  v_new=None if w.new_v is None else _gpu.to_dev_bits(w.new_v),
                                  out=torch.full(q.shape, float("nan"), dtype=torch.bfloat16,
                                                 device="cuda"),
                                  window=w.spec.window, softmax_scale=w.spec.softmax_scale,
                                  **extra))
    ws = torch.empty(max(256, pkv.paged_decode_step_workspace_bytes(dl, max_len)),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            pkv.paged_decode_step(dl, slots, bt, lens, max_len, workspace=ws)
    torch.cuda.current_stream().wait_stream(cap)
    assert pkv.last_launch_count() >= 2 * len(layers)
    return pools, dl, graph


def _oracle_layer_pools(layers, rope=None):
    """Oracle pools after each layer's append of history + new token, one at
    a time (a generator of (pool, rotated q or None)); layers that share
    history arrays share one history append.  With ``rope`` the new token is
    appended by the oracle's RoPE + append at position seq_len - 1."""
    base = {}
    seen = []
    for w in layers:
        key = id(w.hist_k)
        if key not in base:
            base[key] = _util.oracle_pool(w, append_new=False)
        b = base[key]
        op = oracle.OraclePool(k=b.k.copy(), v=None if b.v is None else b.v.copy(),
                               k_scale=None if b.k_scale is None else b.k_scale.copy(),
                               v_scale=None if b.v_scale is None else b.v_scale.copy(),
                               scale_mode=b.scale_mode)
        if rope is None:
            oracle.append(w.new_k, w.new_v, w.new_slots, op)
            yield op, None
        else:
            q_rot, rc = oracle.append_rope(w.q, w.new_k, w.new_v, w.seq_lens.astype(np.int64) - 1,
                                           w.new_slots, op, rope[len(seen)][1])
            assert rc == 0
            yield op, q_rot
        seen.append(w)


def _check_pool(gp, op, name):
    k, v, ks, vs = _gpu.pool_to_host(gp)
    assert np.array_equal(k, op.k), f"{name}: K pool differs from the oracle's append"
    if op.v is not None:
        assert np.array_equal(v, op.v), f"{name}: V pool differs from the oracle's append"
    if op.scale_mode == oracle.SCALE_PER_TOKEN:
        assert np.array_equal(ks.view(np.uint32), op.k_scale.view(np.uint32))


def _run(layers, rows=None, replays=2, with_rope=False):
    rope = _rope_tables(layers, int(layers[0].seq_lens.max())) if with_rope else None
    if rope is not None:
        assert not any(r[2].any() for r in rope)  # no entry near an fp32 rounding midpoint
    pools, dl, graph = _captured_step(layers, rope)
    for _ in range(replays):  # the replays append the same tokens to the same slots
        graph.replay()
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) == 0
    for i, (w, gp, (op, q_rot), d) in enumerate(zip(layers, pools,
                                                    _oracle_layer_pools(layers, rope), dl)):
        name = f"layer {i} ({w.spec.name})"
        _check_pool(gp, op, name)
        q_ref = w.q
        if q_rot is not None:
            got_q = d.q_rotated.view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got_q, q_rot), f"{name}: rotated q differs"
            q_ref = q_rot
        got = _gpu.out_to_f64(d.out)
        assert np.all(np.isfinite(got)), name
        s = w.spec
        ref = oracle.decode(q_ref, op, w.block_table, w.seq_lens, s.num_q_heads, s.window,
                            np.float32(s.softmax_scale), rows=rows)
        if rows is None:
            err = _gpu.max_abs_err(got, ref)
        else:
            err = _gpu.max_abs_err(got[rows[:, 0], rows[:, 1]], ref)
        assert err <= BF16_TOL, (name, err)


def test_six_layer_step_small_captured():
    s = synth.shrink(synth.C5_SLIDING, batch=24, lens=("lognormal", 300.0, 1.0, 1, 4000),
                     shared_prefix_seqs=6)
    g = synth.shrink(synth.C5_GLOBAL, batch=24, lens=("lognormal", 300.0, 1.0, 1, 4000),
                     shared_prefix_seqs=6)
    _run(synth.make_step(s, g))


def test_six_layer_step_small_captured_with_rope():
    """The same step with RoPE fused into every layer's append (the sliding
    layers turn every pair, the global layer a quarter of them)."""
    s = synth.shrink(synth.C5_SLIDING, batch=24, lens=("lognormal", 300.0, 1.0, 1, 4000),
                     shared_prefix_seqs=6)
    g = synth.shrink(synth.C5_GLOBAL, batch=24, lens=("lognormal", 300.0, 1.0, 1, 4000),
                     shared_prefix_seqs=6)
    _run(synth.make_step(s, g), with_rope=True)


@pytest.mark.parametrize("with_rope", [False, True])
def test_six_layer_step_full_captured(with_rope):
    """The full continuous-batching workload: batch 256, lognormal lengths
    up to 65536, 8 prefix blocks shared by 64 sequences.  The five sliding
    layers share history values (each has its own pool); queries and new
    tokens differ per layer.  Also with RoPE fused into every append."""
    layers = synth.make_step(share_history=True)
    w = layers[0]
    rng = np.random.default_rng(5)
    B, Hq = w.q.shape[:2]
    rows = {(int(rng.integers(B)), int(rng.integers(Hq))) for _ in range(40)}
    shared = np.nonzero(w.layout.shared_seqs)[0]
    for b in (int(np.argmax(w.seq_lens)), int(np.argmin(w.seq_lens)), int(shared[0]),
              int(shared[-1])):
        rows.add((b, 0))
        rows.add((b, Hq - 1))
    _run(layers, rows=np.array(sorted(rows), np.int32), replays=2, with_rope=with_rope)
