"""paged_decode_attention_noalloc: the decode entry point for callers that
cannot allocate device memory (a plugin given only its inputs and outputs,
an engine that reserved all of HBM for its KV pool, a loop in which an
allocation would synchronise the device).  Its split partials live in a fixed
per-device array inside the library instead of a caller workspace.

Collected last on purpose: a run that stops at the first failure has then
already run every other test."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import paged_kv_decode_03_gb300 as pkv  # noqa: E402
from paged_kv_decode_03_gb300 import binding, synth  # noqa: E402

BF16_TOL = 2e-2  # the attention tolerance the parity tests use on bf16 outputs
FAKE = 0x7F0000000000


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    """Host-side check only: nothing is launched."""
    lib = pkv.load_library()
    pool = binding.PkvPoolC(FAKE, FAKE + (1 << 30), None, None, 1 << 20, 16, 1, 256,
                            pkv.PKV_BF16, pkv.SCALE_NONE)
    # 4096 sequences x 16 heads x 64 splits x 257 floats is far beyond 32 MiB
    rc = lib.paged_decode_attention_noalloc(FAKE, ctypes.byref(pool), FAKE, 4096, FAKE, 4096, 16,
                                            65536, 0, 0.0625, 1024, FAKE, 0, None)
    assert rc == -4  # PKV_E_WORKSPACE
    assert b"static scratch" in lib.pkv_last_error()


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests import _gpu
    pkv.load_library()
    specs = [
        (synth.shrink(synth.C2, batch=8, lens=("uniform", 600, 4000)), 256),
        (synth.shrink(synth.C3, batch=6, lens=("uniform", 3000, 9000)), 1024),
    ]
    for spec, split in specs:  # two calls in a row; the second reuses the array
        w = synth.make_workload(spec)
        gp = _gpu.device_pool(w)
        _gpu.append_all(w, gp)
        step = _gpu.DeviceStep(w)
        ref = _gpu.out_to_f64(step.decode(gp, split_tokens=split))
        out = torch.full(step.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        pkv.paged_decode_attention_noalloc(step.q, gp, step.block_table, step.seq_lens,
                                           spec.window, np.float32(spec.softmax_scale), out,
                                           step.max_seq_len, split_tokens=split)
        torch.cuda.synchronize()
        got = _gpu.out_to_f64(out)
        assert np.all(np.isfinite(got))
        assert _gpu.max_abs_err(got, ref) <= BF16_TOL, (spec.name, _gpu.max_abs_err(got, ref))
    assert pkv.device_status(clear=True) == 0
