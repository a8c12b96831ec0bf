"""Parity at the full workload sizes, in the launch configuration the
benchmark times (automatic split length, bf16 output) and with fp32 outputs:
append/quantise is compared bit for bit over the whole pool; attention on a
sample of output rows that the oracle computes one by one (plus the longest
and shortest sequences)."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import paged_kv_decode_03_gb300 as pkv  # noqa: E402
from paged_kv_decode_03_gb300 import synth  # noqa: E402
from tests import _util  # noqa: E402

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
F32_REL_TOL = 1e-4  # normwise per (b, h) row, fp32 outputs


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load_library()
    pkv.device_status(clear=True)


from tests import _gpu  # noqa: E402


def _sample_rows(w, n=48, seed=0):
    rng = np.random.default_rng(seed)
    B, Hq = w.q.shape[:2]
    rows = {(int(rng.integers(B)), int(rng.integers(Hq))) for _ in range(n)}
    for b in (int(np.argmax(w.seq_lens)), int(np.argmin(w.seq_lens))):
        rows.add((b, 0))
        rows.add((b, Hq - 1))
    return np.array(sorted(rows), np.int32)


def _full_case(spec, check_pool_bits=True):
    w = synth.make_workload(spec)
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    op = _util.oracle_pool(w)
    torch.cuda.synchronize()
    if check_pool_bits:
        k, v, ks, vs = _gpu.pool_to_host(gp)
        assert np.array_equal(k, op.k)
        if op.v is not None:
            assert np.array_equal(v, op.v)
        if ks is not None and spec.kv == "int8_token":
            assert np.array_equal(ks.view(np.uint32), op.k_scale.view(np.uint32))
            assert np.array_equal(vs.view(np.uint32), op.v_scale.view(np.uint32))
    step = _gpu.DeviceStep(w)
    got = _gpu.out_to_f64(step.decode(gp, split_tokens=spec.split_tokens or pkv.SPLIT_AUTO))
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) == 0
    rows = _sample_rows(w)
    ref = _util.oracle_decode(w, op, rows=rows)
    err = _gpu.max_abs_err(got[rows[:, 0], rows[:, 1]], ref)
    assert err <= BF16_TOL, (spec.name, err)
    assert np.all(np.isfinite(got))
    # fp32 outputs (the parity mode) at full size, on the same sampled rows
    got32 = _gpu.out_to_f64(step.decode(gp, split_tokens=spec.split_tokens or pkv.SPLIT_AUTO,
                                        out_f32=True))
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) == 0
    rel = _gpu.max_row_rel_err(got32[rows[:, 0], rows[:, 1]], ref)
    assert rel <= F32_REL_TOL, (spec.name, rel)


def test_c2_gemma4_sliding_full():
    _full_case(synth.C2)


def test_c3_gemma4_global_full():
    _full_case(synth.C3)


def test_c4_llama2_int8_full():
    _full_case(synth.C4)


def test_c5_step_full_global_layer():
    layers = synth.make_step()
    _full_case_layer = layers[-1]
    w = _full_case_layer
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    op = _util.oracle_pool(w)
    got = _gpu.out_to_f64(_gpu.DeviceStep(w).decode(gp))
    torch.cuda.synchronize()
    rows = _sample_rows(w)
    ref = _util.oracle_decode(w, op, rows=rows)
    assert _gpu.max_abs_err(got[rows[:, 0], rows[:, 1]], ref) <= BF16_TOL


def test_c5_step_full_sliding_layer():
    layers = synth.make_step(pattern=("S",))
    w = layers[0]
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    op = _util.oracle_pool(w)
    torch.cuda.synchronize()
    k, v, _, _ = _gpu.pool_to_host(gp)
    assert np.array_equal(k, op.k) and np.array_equal(v, op.v)
    got = _gpu.out_to_f64(_gpu.DeviceStep(w).decode(gp))
    torch.cuda.synchronize()
    rows = _sample_rows(w)
    ref = _util.oracle_decode(w, op, rows=rows)
    assert _gpu.max_abs_err(got[rows[:, 0], rows[:, 1]], ref) <= BF16_TOL
