"""paged_decode_attention_noalloc: the decode entry point for callers that
cannot allocate device memory (a plugin given only its inputs and outputs,
an engine that reserved all of HBM for its KV pool, a loop in which an
allocation would synchronise the device).  Its split partials live in a fixed
per-device array inside the library instead of a caller workspace.

Run last (tests/conftest.py orders the collection): a run that stops at the
first failure has then already run every other test."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import paged_kv_decode_03_gb300 as pkv  # noqa: E402
from paged_kv_decode_03_gb300 import binding, synth  # noqa: E402

BF16_TOL = 2e-2  # the attention tolerance the parity tests use on bf16 outputs
FAKE = 0x7F0000000000
STATIC_BYTES = 32 << 20  # PKV_STATIC_SCRATCH_BYTES


def _fake_pool(num_kv_heads, head_dim, dtype=pkv.PKV_BF16):
    return binding.PkvPoolC(FAKE, FAKE + (1 << 30), None, None, 1 << 20, 16, num_kv_heads,
                            head_dim, dtype, pkv.SCALE_NONE)


def _noalloc_rc(lib, pool, batch, hq, max_len, split):
    maxb = (max_len + 15) // 16
    return lib.paged_decode_attention_noalloc(FAKE, ctypes.byref(pool), FAKE, maxb, FAKE, batch,
                                              hq, max_len, 0, 0.0625, split, FAKE, 0, None)


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    """Host-side check only: nothing is launched.  A CUDA-core split whose
    partials (4096 sequences x 16 heads x 64 splits x 257 floats) are far
    beyond 32 MiB is refused before any device call."""
    lib = pkv.load_library()
    pool = _fake_pool(4, 256)  # 4 query heads per KV head: the CUDA-core kernel
    rc = _noalloc_rc(lib, pool, 4096, 16, 65536, 1024)
    assert rc == -4  # PKV_E_WORKSPACE
    assert b"static scratch" in lib.pkv_last_error()


def test_noalloc_sizes_the_tensor_core_path_by_its_own_scratch():
    """The tensor-core kernel (16 query heads per KV head, bf16) balances the
    key ranges itself and ignores the split length, so a short split on the
    Gemma4 global shape (64 MiB of partials if it were honoured) is not
    refused for lack of static scratch: the host check passes, and the call
    gets as far as looking the array up on the device (which fails here,
    without a GPU, or succeeds on one)."""
    lib = pkv.load_library()
    pool = _fake_pool(1, 256)
    assert lib.paged_decode_workspace_bytes(32, 16, 1, 256, 16, 32768, 0, 256) > STATIC_BYTES
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the call would launch on fake pointers")
    rc = _noalloc_rc(lib, pool, 32, 16, 32768, 256)
    assert rc != -4, lib.pkv_last_error()


def _near_limit_batch(lib, hq, hkv, D, max_len, split):
    """Largest batch whose CUDA-core split workspace fits the static array."""
    b = 1
    while lib.paged_decode_workspace_bytes(b + 1, hq, hkv, D, 16, max_len, 0, split) <= STATIC_BYTES:
        b += 1
    return b


def test_noalloc_boundary_batch_is_host_checked():
    """One sequence more than the largest batch that fits is refused on the
    host (PKV_E_WORKSPACE), whatever the device."""
    lib = pkv.load_library()
    hq, hkv, D, L, split = 8, 2, 256, 4080, 16
    b = _near_limit_batch(lib, hq, hkv, D, L, split)
    need = lib.paged_decode_workspace_bytes(b, hq, hkv, D, 16, L, 0, split)
    assert STATIC_BYTES - need < lib.paged_decode_workspace_bytes(1, hq, hkv, D, 16, L, 0, split)
    rc = _noalloc_rc(lib, _fake_pool(hkv, D), b + 1, hq, L, split)
    assert rc == -4, lib.pkv_last_error()


def _oracle_rows(w, rows):
    from tests import _util
    op = _util.oracle_pool(w)
    return _util.oracle_decode(w, op, rows=np.asarray(rows, np.int32)), op


@pytest.mark.gpu
def test_noalloc_matches_the_oracle_and_the_workspace_entry_point_twice():
    """Two calls in a row (the second reuses the array) on a sliding layer
    (CUDA-core kernel, 256-token splits) and a global K == V layer
    (tensor-core kernel): each output against the oracle and against
    paged_decode_attention with a caller workspace."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests import _gpu, _util
    pkv.load_library()
    specs = [
        (synth.shrink(synth.C2, batch=8, lens=("uniform", 600, 4000)), 256),
        (synth.shrink(synth.C3, batch=6, lens=("uniform", 3000, 9000)), 1024),
    ]
    for spec, split in specs:
        w = synth.make_workload(spec)
        gp = _gpu.device_pool(w)
        _gpu.append_all(w, gp)
        step = _gpu.DeviceStep(w)
        ws_out = _gpu.out_to_f64(step.decode(gp, split_tokens=split))
        ref = _util.oracle_decode(w, _util.oracle_pool(w))
        out = torch.full(step.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        pkv.paged_decode_attention_noalloc(step.q, gp, step.block_table, step.seq_lens,
                                           spec.window, np.float32(spec.softmax_scale), out,
                                           step.max_seq_len, split_tokens=split)
        torch.cuda.synchronize()
        got = _gpu.out_to_f64(out)
        assert np.all(np.isfinite(got))
        assert _gpu.max_abs_err(got, ref) <= BF16_TOL, (spec.name, _gpu.max_abs_err(got, ref))
        assert _gpu.max_abs_err(got, ws_out) <= BF16_TOL, spec.name
    assert pkv.device_status(clear=True) == 0


@pytest.mark.gpu
def test_noalloc_split_partials_up_to_the_end_of_the_array():
    """A CUDA-core split (8 query heads on 2 KV heads, 16-token splits) whose
    workspace is the largest batch that fits in the static array, so the
    partial outputs reach its last bytes: the output matches the workspace
    entry point on every row and the oracle on sampled rows, twice."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests import _gpu
    lib = pkv.load_library()
    hq, hkv, D, L, split = 8, 2, 256, 4080, 16
    b = _near_limit_batch(lib, hq, hkv, D, L, split)
    lens = np.random.default_rng(3).integers(L - 600, L + 1, b)
    lens[-1] = L  # the last sequence uses the last split: the array's last bytes
    spec = synth.Spec("noalloc_near_limit", batch=b, num_q_heads=hq, num_kv_heads=hkv,
                      head_dim=D, lens=("fixed", tuple(int(x) for x in lens)), seed=4242)
    w = synth.make_workload(spec)
    assert int(w.seq_lens.max()) == L
    assert lib.paged_decode_workspace_bytes(b, hq, hkv, D, 16, L, 0, split) <= STATIC_BYTES
    gp = _gpu.device_pool(w)
    _gpu.append_all(w, gp)
    step = _gpu.DeviceStep(w)
    ws_out = _gpu.out_to_f64(step.decode(gp, split_tokens=split))
    rng = np.random.default_rng(7)
    rows = sorted({(int(bb), int(h)) for bb, h in zip(rng.integers(0, b, 24),
                                                     rng.integers(0, hq, 24))}
                  | {(b - 1, hq - 1), (b - 1, 0)})
    ref, _ = _oracle_rows(w, rows)
    for _ in range(2):
        out = torch.full(step.q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        pkv.paged_decode_attention_noalloc(step.q, gp, step.block_table, step.seq_lens, 0,
                                           np.float32(spec.softmax_scale), out, L,
                                           split_tokens=split)
        torch.cuda.synchronize()
        got = _gpu.out_to_f64(out)
        assert np.all(np.isfinite(got))
        assert _gpu.max_abs_err(got, ws_out) <= BF16_TOL
        sampled = np.stack([got[bb, h] for bb, h in rows])
        assert _gpu.max_abs_err(sampled, ref) <= BF16_TOL
    assert pkv.device_status(clear=True) == 0
