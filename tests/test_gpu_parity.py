"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.  Append/quantise must be bit-exact; attention must match
within max |err| <= 2e-2 on bf16 outputs and a normwise per-row relative
error <= 1e-4 on fp32 outputs."""
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
F32_REL_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    pkv.device_status(clear=True)
    yield
    torch.cuda.synchronize()


from tests import _gpu  # noqa: E402


def _check_pool_bits(gpu_pool, ora_pool):
    k, v, ks, vs = _gpu.pool_to_host(gpu_pool)
    assert np.array_equal(k, ora_pool.k), "K pool differs from the oracle's append"
    if ora_pool.v is not None:
        assert np.array_equal(v, ora_pool.v), "V pool differs from the oracle's append"
    if ora_pool.scale_mode == oracle.SCALE_PER_TOKEN:
        assert np.array_equal(ks.view(np.uint32), ora_pool.k_scale.view(np.uint32))
        if ora_pool.v_scale is not None:
            assert np.array_equal(vs.view(np.uint32), ora_pool.v_scale.view(np.uint32))


def _run_case(spec, splits=(0, pkv.SPLIT_AUTO), out_modes=(False, True), check_pool=True):
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    op = _util.oracle_pool(w)
    torch.cuda.synchronize()
    if check_pool:
        _check_pool_bits(gp, op)
    ref = _util.oracle_decode(w, op)
    step = _gpu.DeviceStep(w)
    for st in splits:
        for f32 in out_modes:
            got = _gpu.out_to_f64(step.decode(gp, split_tokens=st, out_f32=f32))
            torch.cuda.synchronize()
            if f32:
                err = _gpu.max_row_rel_err(got, ref)
                assert err <= F32_REL_TOL, (spec.name, st, "f32", err)
            else:
                err = _gpu.max_abs_err(got, ref)
                assert err <= BF16_TOL, (spec.name, st, "bf16", err)
    assert pkv.device_status(clear=True) == 0
    return w, gp, op, ref


def test_c1_tiny_global():
    _run_case(synth.C1, splits=(0, 16, 32, pkv.SPLIT_AUTO))


def test_c2_sliding_small():
    spec = synth.shrink(synth.C2, batch=8, lens=("uniform", 1, 3000))
    _run_case(spec, splits=(0, 256, 1024, pkv.SPLIT_AUTO))


def test_c3_global_kv_shared_small():
    spec = synth.shrink(synth.C3, batch=4, lens=("uniform", 1, 5000))
    _run_case(spec, splits=(0, 1024, pkv.SPLIT_AUTO))


def test_c4_int8_per_token_small():
    spec = synth.shrink(synth.C4, batch=4, lens=("const", 300))
    _run_case(spec, splits=(0, 64, pkv.SPLIT_AUTO))


def test_c5_step_small():
    """Six layers (5 sliding int8 per-head + 1 global bf16) over one ragged
    layout with shared prefix blocks: append one token per sequence, then
    decode, layer by layer."""
    s = synth.shrink(synth.C5_SLIDING, batch=24, lens=("lognormal", 300.0, 1.0, 1, 4000),
                     shared_prefix_seqs=6)
    g = synth.shrink(synth.C5_GLOBAL, batch=24, lens=("lognormal", 300.0, 1.0, 1, 4000),
                     shared_prefix_seqs=6)
    layers = synth.make_step(s, g)
    for w in layers:
        gp = _gpu.device_pool(w)
        _gpu.append_all(w, gp)
        op = _util.oracle_pool(w)
        torch.cuda.synchronize()
        _check_pool_bits(gp, op)
        ref = _util.oracle_decode(w, op)
        got = _gpu.out_to_f64(_gpu.DeviceStep(w).decode(gp))
        assert _gpu.max_abs_err(got, ref) <= BF16_TOL
    assert pkv.device_status(clear=True) == 0


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("kv", ["bf16", "int8_token", "int8_head"])
@pytest.mark.parametrize("hq,hkv", [(2, 2), (6, 2), (8, 2), (16, 1)])
def test_edge_shapes(D, kv, hq, hkv):
    """Ragged lengths at block edges (0, 1, 15, 16, 17, 33, ...), GQA group
    sizes 1, 3, 4, 16, every head_dim, every KV format."""
    spec = synth.Spec(f"edge_{D}_{kv}_{hq}_{hkv}", batch=9, num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=D, lens=("fixed", (0, 1, 15, 16, 17, 33, 64, 100, 257)), kv=kv,
                      seed=77 + D + hq)
    _run_case(spec, splits=(0, 16, 48, pkv.SPLIT_AUTO))


@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 5000])
def test_window_edges(window):
    spec = synth.Spec(f"win_{window}", batch=7, num_q_heads=4, num_kv_heads=2, head_dim=128,
                      lens=("fixed", (1, 2, 16, 17, 18, 130, 700)), window=window, seed=91)
    _run_case(spec, splits=(0, 32, pkv.SPLIT_AUTO))


def test_int8_kv_alias_per_token():
    spec = synth.Spec("alias_int8", batch=5, num_q_heads=8, num_kv_heads=1, head_dim=256,
                      lens=("fixed", (1, 40, 200, 333, 17)), kv="int8_token", alias=True, seed=5)
    _run_case(spec, splits=(0, 64))


@pytest.mark.parametrize("kv", ["int8_token", "int8_head"])
def test_append_non_finite_inputs_bit_exact(kv):
    """NaN and +-inf in the appended rows: codes and scales bit-exact with the
    oracle (a NaN has no code and is stored as 0; an inf makes the token's
    per-token scale inf, so its codes are 0, or saturates under a per-head
    scale)."""
    import dataclasses
    spec = synth.Spec(f"nonfinite_{kv}", batch=6, num_q_heads=4, num_kv_heads=2, head_dim=64,
                      lens=("fixed", (1, 5, 16, 17, 30, 40)), kv=kv, seed=13)
    w = synth.make_workload(spec)
    nk, nv = w.new_k.copy(), w.new_v.copy()
    nk[0, 0, 3] = 0x7F80   # +inf
    nk[1, 1, 0] = 0x7FC0   # NaN
    nv[2, 0, 5] = 0xFF80   # -inf
    nv[3, 1, 7] = 0x7FC0   # NaN
    nk[4, 0, :] = 0x7FC0   # one head all NaN
    w = dataclasses.replace(w, new_k=nk, new_v=nv)
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    op = _util.oracle_pool(w)
    torch.cuda.synchronize()
    _check_pool_bits(gp, op)
    assert pkv.device_status(clear=True) == 0


def test_split_partial_matches_oracle_partials():
    """paged_decode_split_partial writes, per split, the log-sum-exp and the
    normalised output of that split's keys."""
    spec = synth.shrink(synth.C2, batch=6, num_q_heads=4, num_kv_heads=2, head_dim=128,
                        lens=("fixed", (5, 300, 1100, 1500, 2000, 64)), window=1024)
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    op = _util.oracle_pool(w)
    step = _gpu.DeviceStep(w)
    split = 256
    ns = pkv.paged_decode_num_splits(step.max_seq_len, spec.window, split)
    B, Hq, D = w.q.shape
    lse = torch.full((B, ns, Hq), float("nan"), device="cuda")      # split-major
    po = torch.full((B, ns, Hq, D), float("nan"), device="cuda")
    out = torch.zeros((B, Hq, D), dtype=torch.float32, device="cuda")
    pkv.paged_decode_split_partial(step.q, gp, step.block_table, step.seq_lens, spec.window,
                                   np.float32(spec.softmax_scale), split, lse, po, out,
                                   step.max_seq_len)
    torch.cuda.synchronize()
    lse_h, po_h, out_h = lse.cpu().numpy(), po.cpu().numpy(), out.cpu().numpy()
    full = _util.oracle_decode(w, op)
    for b in range(B):
        L = int(w.seq_lens[b])
        pos = L - 1
        lo = max(0, pos - spec.window)
        nblk = pos // 16 - lo // 16 + 1
        nsb = -(-nblk // (split // 16))
        if nsb == 1:
            assert _gpu.max_row_rel_err(out_h[b].astype(np.float64), full[b]) <= F32_REL_TOL
            continue
        for s in range(nsb):
            kb = (lo // 16 + s * (split // 16)) * 16
            ke = kb + split
            ol, oo = oracle.partial(w.q, op, w.block_table, w.seq_lens, Hq, spec.window,
                                    np.float32(spec.softmax_scale),
                                    np.full(B, kb), np.full(B, ke))
            np.testing.assert_allclose(lse_h[b, s], ol[b], rtol=0, atol=2e-5)
            assert _gpu.max_row_rel_err(po_h[b, s].astype(np.float64), oo[b]) <= F32_REL_TOL
    # the combine step on these partials gives the full decode
    out2 = out.clone()
    pkv.paged_decode_lse_combine(lse, po, step.seq_lens, spec.window, split, out2)
    torch.cuda.synchronize()
    assert _gpu.max_row_rel_err(out2.cpu().numpy().astype(np.float64), full) <= F32_REL_TOL


@pytest.mark.parametrize("hq,hkv,D,alias", [(16, 1, 256, True), (16, 2, 128, False)])
def test_tc_split_partial_matches_oracle_partials(hq, hkv, D, alias):
    """On the tensor-core kernel the split partials come from the stream-K
    walk: splits cut between SMs are merged by the CTA holding their last part
    before they are written.  Each split's log-sum-exp and normalised output
    must match the oracle's partial of the same keys."""
    spec = synth.Spec(f"tc_split_{hq}_{hkv}_{D}", batch=7, num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=D, lens=("fixed", (0, 5, 300, 2100, 4500, 64, 9000)), alias=alias,
                      seed=21 + D)
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    op = _util.oracle_pool(w)
    step = _gpu.DeviceStep(w)
    split = 512
    ns = pkv.paged_decode_num_splits(step.max_seq_len, spec.window, split)
    B, Hq, _ = w.q.shape
    lse = torch.full((B, ns, Hq), float("nan"), device="cuda")      # split-major
    po = torch.full((B, ns, Hq, D), float("nan"), device="cuda")
    out = torch.zeros((B, Hq, D), dtype=torch.float32, device="cuda")
    pkv.paged_decode_split_partial(step.q, gp, step.block_table, step.seq_lens, spec.window,
                                   np.float32(spec.softmax_scale), split, lse, po, out,
                                   step.max_seq_len)
    torch.cuda.synchronize()
    lse_h, po_h, out_h = lse.cpu().numpy(), po.cpu().numpy(), out.cpu().numpy()
    full = _util.oracle_decode(w, op)
    for b in range(B):
        L = int(w.seq_lens[b])
        nblk = (L - 1) // 16 + 1 if L > 0 else 0
        nsb = max(1, -(-nblk // (split // 16)))
        if nsb == 1:
            assert _gpu.max_row_rel_err(out_h[b].astype(np.float64), full[b]) <= F32_REL_TOL
            continue
        for s_ in range(nsb):
            kb = s_ * split
            ol, oo = oracle.partial(w.q, op, w.block_table, w.seq_lens, Hq, spec.window,
                                    np.float32(spec.softmax_scale),
                                    np.full(B, kb), np.full(B, kb + split))
            np.testing.assert_allclose(lse_h[b, s_], ol[b], rtol=0, atol=2e-5)
            assert _gpu.max_row_rel_err(po_h[b, s_].astype(np.float64), oo[b]) <= F32_REL_TOL
    out2 = out.clone()
    pkv.paged_decode_lse_combine(lse, po, step.seq_lens, spec.window, split, out2)
    torch.cuda.synchronize()
    assert _gpu.max_row_rel_err(out2.cpu().numpy().astype(np.float64), full) <= F32_REL_TOL
    assert pkv.device_status(clear=True) == 0


@pytest.mark.parametrize("lens", [
    (0, 1, 20000, 0, 3, 129, 128),        # one range cut by many SM boundaries, empty rows
    (1, 17, 130),                          # fewer tiles than SMs: one tile per CTA
    (0, 0, 0),                             # nothing to read at all
    tuple(range(1, 4000, 97)),             # many short ranges, some cut
])
def test_tc_stream_k_partition(lens):
    """The stream-K walk of the tensor-core kernel: any mix of lengths splits
    into equal tile shares per SM; ranges cut between SMs are merged by the
    CTA holding their last part."""
    spec = synth.Spec(f"tc_sk_{len(lens)}_{max(lens)}", batch=len(lens), num_q_heads=16,
                      num_kv_heads=1, head_dim=256, lens=("fixed", lens), alias=True,
                      seed=5 + len(lens))
    _run_case(spec, splits=(0,))


def test_tc_stream_k_gqa8_window():
    spec = synth.Spec("tc_sk_gqa8", batch=11, num_q_heads=32, num_kv_heads=4, head_dim=128,
                      lens=("fixed", (3000, 1, 0, 700, 1025, 1026, 2048, 16, 5000, 333, 64)),
                      window=1024, seed=44)
    _run_case(spec, splits=(0,))


def test_tc_graph_capture():
    """The tensor-core path (plan and persistent cooperative decode kernels)
    captures into a CUDA graph and replays."""
    spec = synth.shrink(synth.C3, batch=5, lens=("uniform", 1, 6000))
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp, new=False)
    op = _util.oracle_pool(w)
    step = _gpu.DeviceStep(w)
    k_new, slots = _gpu.to_dev_bits(w.new_k), _gpu.to_dev(w.new_slots)
    B, Hq, D = w.q.shape
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(1, pkv.paged_decode_workspace_bytes(B, Hq, spec.num_kv_heads, D,
                                                             step.max_seq_len, spec.window)),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkv.paged_kv_append(k_new, None, slots, gp)
        pkv.paged_decode_attention(step.q, gp, step.block_table, step.seq_lens, spec.window,
                                   spec.softmax_scale, out, step.max_seq_len, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.paged_kv_append(k_new, None, slots, gp)
        pkv.paged_decode_attention(step.q, gp, step.block_table, step.seq_lens, spec.window,
                                   spec.softmax_scale, out, step.max_seq_len, workspace=ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    oracle.append(w.new_k, None, w.new_slots, op)
    ref = _util.oracle_decode(w, op)
    assert _gpu.max_abs_err(_gpu.out_to_f64(out), ref) <= BF16_TOL
    assert pkv.device_status(clear=True) == 0


def test_lse_combine_on_given_partials():
    """The combine alone, on partial states computed by the oracle."""
    rng = np.random.default_rng(3)
    B, Hq, ns, D = 3, 2, 4, 64
    lens = np.array([16 * 4 * 3, 16 * 4 * 4, 16 * 4 + 1], np.int32)  # 3, 4 and 2 splits of 64
    lse = rng.normal(size=(B, Hq, ns)).astype(np.float32) * 3
    po = rng.normal(size=(B, Hq, ns, D)).astype(np.float32)
    lse[0, :, 3] = np.nan  # beyond sequence 0's splits: must be ignored
    out = torch.zeros((B, Hq, D), dtype=torch.float32, device="cuda")
    # the library's partials are split-major: [B][splits][H_q](, D)
    lse_d = _gpu.to_dev(np.ascontiguousarray(lse.transpose(0, 2, 1)))
    po_d = _gpu.to_dev(np.ascontiguousarray(po.transpose(0, 2, 1, 3)))
    pkv.paged_decode_lse_combine(lse_d, po_d, _gpu.to_dev(lens), 0, 64, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for b, nsb in enumerate((3, 4, 2)):
        for h in range(Hq):
            y, _ = oracle.lse_combine(lse[b, h, :nsb].astype(np.float64),
                                      po[b, h, :nsb].astype(np.float64))
            np.testing.assert_allclose(got[b, h], y, rtol=2e-5, atol=2e-6)


@pytest.mark.parametrize("D,max_splits,f32,offset", [
    (256, 40, False, 0),    # 16-byte columns, two split subsets per column
    (256, 31, True, 0),
    (100, 300, False, 1),   # scalar columns (head_dim % 4 != 0), misaligned out
    (64, 300, True, 1),     # misaligned fp32 out: scalar stores
    (512, 9, False, 0),     # as many columns as threads
    (1024, 5, True, 0),     # more columns than threads: two passes
])
def test_lse_combine_shapes(D, max_splits, f32, offset):
    """The combine on oracle partials over its column and split layouts:
    more splits than threads, rows with fewer or more 16-byte columns than
    threads, head_dim not a multiple of four, and an output that is not
    16-byte aligned (element offset)."""
    rng = np.random.default_rng(D + max_splits)
    B, Hq, split_tokens = 5, 3, 16
    nsb = np.array([max_splits, 1, 2, max_splits - 1, 7], np.int64)
    nsb = np.minimum(nsb, max_splits)
    lens = (nsb * split_tokens).astype(np.int32)
    lse = rng.normal(size=(B, Hq, max_splits)).astype(np.float32) * 4
    po = rng.normal(size=(B, Hq, max_splits, D)).astype(np.float32)
    dt = torch.float32 if f32 else torch.bfloat16
    base = torch.zeros(B * Hq * D + offset, dtype=dt, device="cuda")
    out = base[offset:].view(B, Hq, D)
    lse_d = _gpu.to_dev(np.ascontiguousarray(lse.transpose(0, 2, 1)))
    po_d = _gpu.to_dev(np.ascontiguousarray(po.transpose(0, 2, 1, 3)))
    pkv.paged_decode_lse_combine(lse_d, po_d, _gpu.to_dev(lens), 0, split_tokens, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    for b in range(B):
        for h in range(Hq):
            if nsb[b] <= 1:
                assert np.all(got[b, h] == 0)  # single-split rows are left untouched
                continue
            y, _ = oracle.lse_combine(lse[b, h, :nsb[b]].astype(np.float64),
                                      po[b, h, :nsb[b]].astype(np.float64))
            if f32:
                np.testing.assert_allclose(got[b, h], y, rtol=2e-5, atol=2e-6)
            else:
                np.testing.assert_allclose(got[b, h], y, rtol=1 / 128, atol=1e-3)
    assert base[:offset].float().abs().sum().item() == 0  # nothing written before out


def test_bad_block_id_is_reported_not_faulted():
    spec = synth.Spec("badblk", batch=3, num_q_heads=4, num_kv_heads=2, head_dim=64,
                      lens=("fixed", (40, 40, 40)), seed=8)
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    op = _util.oracle_pool(w)
    ref = _util.oracle_decode(w, op)
    step = _gpu.DeviceStep(w)
    pkv.device_status(clear=True)
    bt = w.block_table.copy()
    bt[1, 1] = w.layout.num_blocks + 1000
    step.block_table = _gpu.to_dev(bt)
    got = _gpu.out_to_f64(step.decode(gp, split_tokens=0))
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) & 1  # PKV_DEV_BAD_BLOCK
    # the other sequences are unaffected
    assert _gpu.max_abs_err(got[[0, 2]], ref[[0, 2]]) <= BF16_TOL


@pytest.mark.parametrize("alias", [True, False])
def test_bad_block_id_tensor_core_path(alias):
    """A block id outside the pool on the tensor-core path: reported, never
    dereferenced (its box reads as zeros), the sequence's own output finite
    but unspecified, the other sequences exact; single pass and splits."""
    spec = synth.Spec("badblk_tc", batch=3, num_q_heads=16, num_kv_heads=1, head_dim=128,
                      lens=("fixed", (700, 700, 700)), alias=alias, seed=18)
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    assert pkv.uses_tensor_cores(gp, spec.num_q_heads)
    _gpu.append_all(w, gp)
    op = _util.oracle_pool(w)
    ref = _util.oracle_decode(w, op)
    step = _gpu.DeviceStep(w)
    bt = w.block_table.copy()
    bt[1, 20] = w.layout.num_blocks + 1000
    step.block_table = _gpu.to_dev(bt)
    # single pass
    pkv.device_status(clear=True)
    got = _gpu.out_to_f64(step.decode(gp, split_tokens=0))
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) & 1  # PKV_DEV_BAD_BLOCK
    assert np.isfinite(got[1]).all()
    assert _gpu.max_abs_err(got[[0, 2]], ref[[0, 2]]) <= BF16_TOL
    # split partials and the combine
    split = 256
    ns = pkv.paged_decode_num_splits(step.max_seq_len, spec.window, split)
    B, Hq, D = w.q.shape
    lse = torch.empty((B, ns, Hq), device="cuda")
    po = torch.empty((B, ns, Hq, D), device="cuda")
    out = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    pkv.device_status(clear=True)
    pkv.paged_decode_split_partial(step.q, gp, step.block_table, step.seq_lens, spec.window,
                                   np.float32(spec.softmax_scale), split, lse, po, out,
                                   step.max_seq_len)
    pkv.paged_decode_lse_combine(lse, po, step.seq_lens, spec.window, split, out)
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) & 1
    got = _gpu.out_to_f64(out)
    assert np.isfinite(got[1]).all()
    assert _gpu.max_abs_err(got[[0, 2]], ref[[0, 2]]) <= BF16_TOL


def test_bad_slot_is_reported_not_faulted():
    spec = synth.Spec("badslot", batch=2, num_q_heads=2, num_kv_heads=2, head_dim=64,
                      lens=("fixed", (5, 5)), seed=9)
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    before = gp.k.clone()
    pkv.device_status(clear=True)
    slots = np.array([w.layout.num_blocks * 16 + 3, -1], np.int64)
    pkv.paged_kv_append(_gpu.to_dev_bits(w.new_k), _gpu.to_dev_bits(w.new_v), _gpu.to_dev(slots), gp)
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) & 4  # PKV_DEV_BAD_SLOT
    assert torch.equal(gp.k.view(torch.int16), before.view(torch.int16))


def test_length_beyond_host_bound_is_reported():
    spec = synth.Spec("bound", batch=2, num_q_heads=2, num_kv_heads=1, head_dim=64,
                      lens=("fixed", (100, 20)), seed=10)
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    step = _gpu.DeviceStep(w)
    step.max_seq_len = 50  # lies: sequence 0 has 100 keys
    pkv.device_status(clear=True)
    step.decode(gp, split_tokens=16)
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) & 16  # PKV_DEV_LEN_BOUND


def test_graph_capture_replays_the_step():
    """The calls read no device data on the host, so a decode step captures
    into a CUDA graph and replays with new inputs in the same buffers."""
    spec = synth.shrink(synth.C2, batch=4, lens=("uniform", 100, 2000))
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp, new=False)
    op = _util.oracle_pool(w)
    step = _gpu.DeviceStep(w)
    k_new, v_new, slots = (_gpu.to_dev_bits(w.new_k), _gpu.to_dev_bits(w.new_v),
                           _gpu.to_dev(w.new_slots))
    B, Hq, D = w.q.shape
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(1, pkv.paged_decode_workspace_bytes(B, Hq, spec.num_kv_heads, D,
                                                             step.max_seq_len, spec.window)),
                     dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        # warm-up outside capture
        pkv.paged_kv_append(k_new, v_new, slots, gp)
        pkv.paged_decode_attention(step.q, gp, step.block_table, step.seq_lens, spec.window,
                                   spec.softmax_scale, out, step.max_seq_len, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.paged_kv_append(k_new, v_new, slots, gp)
        pkv.paged_decode_attention(step.q, gp, step.block_table, step.seq_lens, spec.window,
                                   spec.softmax_scale, out, step.max_seq_len, workspace=ws)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    oracle.append(w.new_k, w.new_v, w.new_slots, op)
    ref = _util.oracle_decode(w, op)
    assert _gpu.max_abs_err(_gpu.out_to_f64(out), ref) <= BF16_TOL


@pytest.mark.parametrize("case", ["c2", "c3", "edge"])
def test_cuda_core_kernel_on_bf16_shapes(case, monkeypatch):
    """bf16 pools with head_dim 128/256 normally run on the tensor-core
    kernel; PKV_DISABLE_TC=1 selects the CUDA-core kernel, which must match
    the oracle on the same shapes."""
    monkeypatch.setenv("PKV_DISABLE_TC", "1")
    if case == "c2":
        spec = synth.shrink(synth.C2, batch=6, lens=("uniform", 1, 2500))
    elif case == "c3":
        spec = synth.shrink(synth.C3, batch=3, lens=("uniform", 1, 4000))
    else:
        spec = synth.Spec("edge_cc", batch=9, num_q_heads=6, num_kv_heads=2, head_dim=128,
                          lens=("fixed", (0, 1, 15, 16, 17, 33, 64, 100, 257)), window=40, seed=3)
    _run_case(spec, splits=(0, 32, pkv.SPLIT_AUTO))


@pytest.mark.parametrize("case", ["c2", "edge128", "edge256"])
def test_tensor_core_kernel_on_small_groups(case, monkeypatch):
    """GQA groups below 8 normally run on the CUDA-core kernel;
    PKV_FORCE_TC=1 runs them on the tensor-core kernel, which must match the
    oracle too (padded query heads, masked edges, splits)."""
    monkeypatch.setenv("PKV_FORCE_TC", "1")
    if case == "c2":
        spec = synth.shrink(synth.C2, batch=6, lens=("uniform", 1, 2500))
    else:
        D = 128 if case == "edge128" else 256
        spec = synth.Spec(f"edge_tc_{D}", batch=9, num_q_heads=6, num_kv_heads=2, head_dim=D,
                          lens=("fixed", (0, 1, 15, 16, 17, 33, 64, 100, 257)), window=40, seed=4)
    _run_case(spec, splits=(0, 32, 128, pkv.SPLIT_AUTO))


def test_tensor_core_and_cuda_core_kernels_agree():
    """Both kernels on one workload, fp32 output: they reduce in different
    orders, so they agree to the oracle tolerance, not bit for bit."""
    import os
    spec = synth.shrink(synth.C3, batch=4, lens=("uniform", 100, 3000))
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    step = _gpu.DeviceStep(w)
    a = _gpu.out_to_f64(step.decode(gp, split_tokens=0, out_f32=True))  # tensor cores (G=16)
    os.environ["PKV_DISABLE_TC"] = "1"
    try:
        c = _gpu.out_to_f64(step.decode(gp, split_tokens=0, out_f32=True))
    finally:
        del os.environ["PKV_DISABLE_TC"]
    torch.cuda.synchronize()
    assert _gpu.max_row_rel_err(a, c) <= 2 * F32_REL_TOL


@pytest.mark.parametrize("spin", [False, True])
def test_bounded_wait_runs_out_and_reports(spin):
    """The failure path of every pipeline wait: a wait on an mbarrier phase
    that nothing completes gives up after its limit (1 ms here), sets
    PKV_DEV_TIMEOUT and returns; the context stays usable (a decode right
    after it matches the oracle)."""
    assert pkv.device_status(clear=True) == 0
    out = torch.zeros(64, dtype=torch.int32, device="cuda")
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    pkv.check_bounded_wait(1_000_000, spin, out)
    t1.record()
    torch.cuda.synchronize()
    assert int(out.sum()) == 64, "every thread's wait must give up"
    assert pkv.device_status(clear=True) & 8  # PKV_DEV_TIMEOUT
    assert t0.elapsed_time(t1) < 1000.0  # bounded: returned well within a second
    _run_case(synth.C1, splits=(0,), out_modes=(False,))
