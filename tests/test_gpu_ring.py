"""Ring-KV layout of sliding layers on the GPU ("实验五：Gemma4 端到端推理优化",
Ring KV Cache: position t in slot t mod W of a fixed ring per sequence)
against the oracle's ring gather, which is pinned to its paged gather.

The library's slot mapping must give the oracle's slots bit for bit, the
appends through it must leave the oracle's pool, and the decode must match
the oracle: on small cases that put the window's ends at every offset of a
block and wrap the ring, on both decode kernels, and at the full Gemma4
sliding-layer and continuous-batching sliding-layer sizes."""
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
P = 16


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    pkv.device_status(clear=True)
    yield
    torch.cuda.synchronize()


from tests import _gpu  # noqa: E402


def _check_slots_and_pool(w, gp, op):
    """The library's slot mapping equals the oracle's, for the history and
    the step's tokens; the pools agree bit for bit."""
    hist_o, new_o = _util.oracle_slots(w, op)
    hist_g = _gpu.library_slots(w, gp, w.hist_seq, w.hist_pos).cpu().numpy()
    new_g = _gpu.new_token_slots(w, gp).cpu().numpy()
    assert np.array_equal(hist_g, hist_o)
    assert np.array_equal(new_g, new_o)
    k, v, ks, vs = _gpu.pool_to_host(gp)
    assert np.array_equal(k, op.k), "K pool differs from the oracle's append"
    if op.v is not None:
        assert np.array_equal(v, op.v), "V pool differs from the oracle's append"
    if op.scale_mode == oracle.SCALE_PER_TOKEN:
        assert np.array_equal(ks.view(np.uint32), op.k_scale.view(np.uint32))


def _ring_case(spec, splits=(0, pkv.SPLIT_AUTO), out_modes=(False, True), rows=None,
               expect_tc=None, w=None):
    w = w if w is not None else synth.make_workload(spec)
    assert w.hist_slots is None and w.spec.ring_blocks > 0
    gp = _gpu.device_pool(w)
    if expect_tc is not None:
        assert pkv.uses_tensor_cores(gp, spec.num_q_heads) == expect_tc
    _gpu.append_all(w, gp)
    op = _util.oracle_pool(w)
    torch.cuda.synchronize()
    _check_slots_and_pool(w, gp, op)
    ref = _util.oracle_decode(w, op, rows=rows)
    step = _gpu.DeviceStep(w)
    for st in splits:
        for f32 in out_modes:
            got = _gpu.out_to_f64(step.decode(gp, split_tokens=st, out_f32=f32))
            torch.cuda.synchronize()
            if rows is not None:
                got = got[rows[:, 0], rows[:, 1]]
            if f32:
                assert _gpu.max_row_rel_err(got, ref) <= F32_REL_TOL, (spec.name, st)
            else:
                assert _gpu.max_abs_err(got, ref) <= BF16_TOL, (spec.name, st)
    assert pkv.device_status(clear=True) == 0


_LENS = tuple(range(1, 3 * P + 2)) + (95, 96, 97, 200, 333, 1000)


@pytest.mark.parametrize("kv", ["bf16", "int8_token", "int8_head"])
@pytest.mark.parametrize("window", [15, 16, 17, 40])
def test_ring_every_window_offset(kv, window):
    """CUDA-core kernel (2 query heads per KV head): the window's ends at
    every offset of a block, lengths up to ~25 trips round the ring."""
    spec = synth.Spec(f"ring_{kv}_{window}", batch=len(_LENS), num_q_heads=4, num_kv_heads=2,
                      head_dim=128, lens=("fixed", _LENS), window=window, kv=kv, seed=21,
                      ring_blocks=synth.ring_blocks_for(window))
    _ring_case(spec, splits=(0, 16, 32, pkv.SPLIT_AUTO), expect_tc=False)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("window", [16, 100])
def test_ring_tensor_core_kernel(D, window):
    """Tensor-core kernel (16 query heads per KV head, bf16), K == V and
    separate K/V."""
    for alias in (True, False):
        spec = synth.Spec(f"ring_tc_{D}_{window}_{alias}", batch=len(_LENS), num_q_heads=16,
                          num_kv_heads=1, head_dim=D, lens=("fixed", _LENS), window=window,
                          alias=alias, seed=22, ring_blocks=synth.ring_blocks_for(window))
        _ring_case(spec, expect_tc=True)


def test_ring_larger_than_needed():
    """Any W >= w + 1 is a valid ring (here two blocks more)."""
    spec = synth.Spec("ring_loose", batch=len(_LENS), num_q_heads=8, num_kv_heads=2,
                      head_dim=64, lens=("fixed", _LENS), window=24, seed=23,
                      ring_blocks=synth.ring_blocks_for(24) + 2)
    _ring_case(spec)


def _sample_rows(w, n=40, seed=0):
    rng = np.random.default_rng(seed)
    B, Hq = w.q.shape[:2]
    rows = {(int(rng.integers(B)), int(rng.integers(Hq))) for _ in range(n)}
    for b in (int(np.argmax(w.seq_lens)), int(np.argmin(w.seq_lens))):
        rows.add((b, 0))
        rows.add((b, Hq - 1))
    return np.array(sorted(rows), np.int32)


def test_ring_c2_gemma4_sliding_full():
    """Gemma4 sliding layer (batch 64, lengths U[512, 8192], w = 1024) in the
    ring layout: 65 blocks per sequence at most."""
    w = synth.make_workload(synth.C2_RING)
    _ring_case(synth.C2_RING, splits=(pkv.SPLIT_AUTO,), out_modes=(False,), rows=_sample_rows(w),
               w=w)


def test_ring_c5_sliding_full():
    """Continuous-batching sliding layer (batch 256, lognormal lengths up to
    65536, int8 per-head scales) in the ring layout."""
    w = synth.make_workload(synth.C5_SLIDING_RING)
    _ring_case(synth.C5_SLIDING_RING, splits=(pkv.SPLIT_AUTO,), out_modes=(False,),
               rows=_sample_rows(w), w=w)
