"""Chunk attention on the GPU (q_len > 1: chunked prefill and speculative
verification; "实验五：Gemma4 端到端推理优化" Flash Attention section, tiniestgpt
notes section 7) against the oracle's chunk attention, which is pinned to
the decode and to dense causal attention.

Chunks of 1, 4, 17 and 128 tokens (the last token tile partial), global and
windowed layers, every GQA group the kernel takes, K == V and separate K/V,
head dims 64 to 256, paged and ring layouts, bf16 and fp32 outputs, and a
Gemma4 sliding layer at full batch with 128-token chunks.  A chunk of one
token must also agree with the decode kernels."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import paged_kv_decode_03_gb300 as pkv  # noqa: E402
from paged_kv_decode_03_gb300 import synth  # noqa: E402

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


def _oracle_pool(w):
    k, v, ks, vs = synth.empty_pool_arrays(w.spec, w.layout)
    pool = oracle.OraclePool(k=k, v=v, ring_blocks=w.spec.ring_blocks)
    hs = (w.hist_slots if w.hist_slots is not None
          else oracle.slot_mapping(pool, w.block_table, w.hist_seq, w.hist_pos))
    ns = (w.new_slots if w.new_slots is not None
          else oracle.slot_mapping(pool, w.block_table, w.new_seq, w.new_pos))
    if len(hs):
        oracle.append(w.hist_k, w.hist_v, hs, pool)
    oracle.append(w.new_k, w.new_v, ns, pool)
    return pool


def _device_pool(w):
    k, v, _, _ = synth.empty_pool_arrays(w.spec, w.layout)
    gp = pkv.PagedKVPool(k=_gpu.to_dev_bits(k), v=None if v is None else _gpu.to_dev_bits(v),
                         ring_blocks=w.spec.ring_blocks)
    bt = _gpu.to_dev(w.block_table)

    def slots(pre, seq, pos):
        if pre is not None:
            return _gpu.to_dev(pre)
        out = torch.empty(len(pos), dtype=torch.int64, device="cuda")
        pkv.paged_kv_slot_mapping(gp, bt, _gpu.to_dev(pos), out, seq_ids=_gpu.to_dev(seq))
        return out

    if len(w.hist_pos):
        pkv.paged_kv_append(_gpu.to_dev_bits(w.hist_k),
                            None if w.hist_v is None else _gpu.to_dev_bits(w.hist_v),
                            slots(w.hist_slots, w.hist_seq, w.hist_pos), gp)
    pkv.paged_kv_append(_gpu.to_dev_bits(w.new_k), None if w.new_v is None else _gpu.to_dev_bits(w.new_v),
                        slots(w.new_slots, w.new_seq, w.new_pos), gp)
    return gp


def _run(spec, q_lens, out_f32=False, rows=None):
    w = synth.make_chunk_workload(spec, q_lens)
    gp = _device_pool(w)
    op = _oracle_pool(w)
    torch.cuda.synchronize()
    q = _gpu.to_dev_bits(w.q)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32 if out_f32 else torch.bfloat16,
                     device="cuda")
    n = np.diff(w.q_start)
    pkv.paged_prefill_attention(q, _gpu.to_dev(w.q_start), gp, _gpu.to_dev(w.block_table),
                                _gpu.to_dev(w.seq_lens), spec.window,
                                np.float32(spec.softmax_scale), out, int(w.seq_lens.max()),
                                int(n.max()))
    torch.cuda.synchronize()
    assert pkv.device_status(clear=True) == 0
    got = _gpu.out_to_f64(out)
    assert np.all(np.isfinite(got))
    ref = oracle.prefill(w.q, op, w.block_table, w.seq_lens, w.q_start, spec.num_q_heads,
                         spec.window, np.float32(spec.softmax_scale))
    if rows is not None:
        got, ref = got[rows], ref[rows]
    if out_f32:
        err = _gpu.max_row_rel_err(got, ref)
        assert err <= F32_REL_TOL, (spec.name, q_lens, err)
    else:
        err = _gpu.max_abs_err(got, ref)
        assert err <= BF16_TOL, (spec.name, q_lens, err)
    return w, gp, got


_LENS = (1, 5, 16, 17, 40, 128, 129, 300, 700)


@pytest.mark.parametrize("q_len", [1, 4, 17, 128])
@pytest.mark.parametrize("window", [0, 16, 100])
@pytest.mark.parametrize("hq,hkv,D", [(4, 4, 128), (16, 8, 256), (16, 1, 256)])
def test_chunks(q_len, window, hq, hkv, D):
    spec = synth.Spec(f"chunk_{hq}_{hkv}_{D}_w{window}", batch=len(_LENS), num_q_heads=hq,
                      num_kv_heads=hkv, head_dim=D, lens=("fixed", _LENS), window=window,
                      seed=51 + q_len)
    _run(spec, q_len)


@pytest.mark.parametrize("alias", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_chunks_kv_shared_and_fp32(alias, D):
    spec = synth.Spec(f"chunk_alias{alias}_{D}", batch=len(_LENS), num_q_heads=8, num_kv_heads=2,
                      head_dim=D, lens=("fixed", _LENS), window=33, alias=alias, seed=61)
    _run(spec, 17, out_f32=True)
    _run(spec, (1, 2, 3, 4, 5, 6, 7, 8, 9))  # a different chunk length per sequence


def test_chunks_ring_layout():
    """A sliding layer's ring (W >= w + chunk) serves a chunk too."""
    w, n = 40, 17
    spec = synth.Spec("chunk_ring", batch=len(_LENS), num_q_heads=16, num_kv_heads=8,
                      head_dim=256, lens=("fixed", _LENS), window=w, seed=62,
                      ring_blocks=-(-(w + n) // 16))
    _run(spec, n)


def test_chunk_of_one_agrees_with_the_decode_kernels():
    spec = synth.Spec("chunk_one", batch=len(_LENS), num_q_heads=16, num_kv_heads=8,
                      head_dim=256, lens=("fixed", _LENS), window=64, seed=63)
    w, gp, got = _run(spec, 1)
    dec = torch.empty((len(_LENS), 16, 256), dtype=torch.bfloat16, device="cuda")
    pkv.paged_decode_attention(_gpu.to_dev_bits(w.q), gp, _gpu.to_dev(w.block_table),
                               _gpu.to_dev(w.seq_lens), spec.window, np.float32(spec.softmax_scale),
                               dec, int(w.seq_lens.max()))
    torch.cuda.synchronize()
    assert _gpu.max_abs_err(got, _gpu.out_to_f64(dec)) <= BF16_TOL


def test_chunked_prefill_gemma4_sliding_shape():
    """Gemma4 sliding layer shape (lengths U[512, 8192], 16 query heads on 8
    kv heads, head_dim 256, window 1024), 16 sequences, 128-token chunks."""
    spec = synth.shrink(synth.C2, batch=16)
    _run(spec, 128)
