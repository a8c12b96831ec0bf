"""The C ABI without a GPU: the library loads, exports every function that
include/pagedkv.h declares, and rejects invalid arguments on the host before
launching anything.  No call here reaches a kernel."""
from __future__ import annotations

import ctypes
import subprocess

import numpy as np
import pytest

import paged_kv_decode_03_gb300 as pkv
from paged_kv_decode_03_gb300 import binding

E_NULL, E_SHAPE, E_UNSUPPORTED, E_WORKSPACE, E_ALIGN, E_ARG = -1, -2, -3, -4, -5, -6
FAKE = 0x7F0000000000  # an aligned address the host checks never dereference


@pytest.fixture(scope="module")
def lib():
    return pkv.load_library()


def test_library_exports_every_declared_symbol(lib):
    names = pkv.exported_symbols()
    assert {"paged_kv_append", "paged_decode_attention", "paged_decode_split_partial",
            "paged_decode_lse_combine", "pkv_last_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.library_path()], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported
    # the statically linked CUDA runtime stays private
    assert not any(s.startswith("cuda") for s in exported)


def _pool(**kw):
    d = dict(k=FAKE, v=FAKE + (1 << 30), k_scale=None, v_scale=None, num_blocks=64, block_size=16,
             num_kv_heads=2, head_dim=128, dtype=pkv.PKV_BF16, scale_mode=pkv.SCALE_NONE)
    d.update(kw)
    return binding.PkvPoolC(**d)


def _decode(lib, pool, q=FAKE, bt=FAKE, max_blocks=8, sl=FAKE, batch=2, hq=4, max_len=100,
            window=0, split=0, ws=None, ws_bytes=0, out=FAKE, out_dtype=0):
    return lib.paged_decode_attention(q, ctypes.byref(pool), bt, max_blocks, sl, batch, hq, max_len,
                                      window, 0.1, split, ws, ws_bytes, out, out_dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), E_UNSUPPORTED),
    (dict(block_size=32), E_UNSUPPORTED),
    (dict(k=None), E_NULL),
    (dict(k=FAKE + 8), E_ALIGN),
    (dict(dtype=pkv.PKV_INT8), E_ARG),                       # int8 without a scale mode
    (dict(dtype=pkv.PKV_INT8, scale_mode=pkv.SCALE_PER_TOKEN), E_NULL),  # no tables
    (dict(dtype=pkv.PKV_INT8, scale_mode=pkv.SCALE_PER_TOKEN, k_scale=FAKE + 4,
          v_scale=FAKE), E_ALIGN),
    (dict(scale_mode=pkv.SCALE_PER_HEAD), E_ARG),            # bf16 with scales
    (dict(num_kv_heads=0), E_SHAPE),
])
def test_pool_validation(lib, kw, code):
    assert _decode(lib, _pool(**kw)) == code
    assert lib.pkv_last_error().decode()


@pytest.mark.parametrize("kw,code", [
    (dict(hq=3), E_SHAPE),
    (dict(q=None), E_NULL),
    (dict(out=None), E_NULL),
    (dict(q=FAKE + 2), E_ALIGN),
    (dict(window=-1), E_ARG),
    (dict(max_len=200), E_SHAPE),          # beyond max_blocks * block_size
    (dict(out_dtype=7), E_ARG),
    (dict(split=24), E_ARG),               # not a multiple of block_size
    (dict(split=32), E_WORKSPACE),         # needs scratch, none given
    (dict(split=32, ws=FAKE, ws_bytes=16), E_WORKSPACE),
    (dict(batch=70000), E_UNSUPPORTED),
])
def test_decode_argument_validation(lib, kw, code):
    assert _decode(lib, _pool(), **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(ring=-1, window=32), E_ARG),
    (dict(ring=3, window=0), E_ARG),        # a ring needs a sliding window
    (dict(ring=3, window=48), E_SHAPE),     # 48 slots < the window's 49 keys
    (dict(ring=4, window=48, max_blocks=3), E_SHAPE),  # table rows shorter than the ring
])
def test_ring_layout_validation(lib, kw, code):
    """Ring layouts (position t in slot t mod W, W = ring_blocks * 16) are
    checked on the host: W must hold the inclusive window's w + 1 keys."""
    ring = kw.pop("ring")
    assert _decode(lib, _pool(ring_blocks=ring), **kw) == code
    assert lib.pkv_last_error().decode()


def test_ring_lengths_are_not_bounded_by_the_table(lib):
    """A ring of 4 blocks serves a length far beyond 4 * 16: the host check
    passes (the call then needs a device; here it stops at the tensor map or
    the error word, never at the shape check)."""
    rc = _decode(lib, _pool(ring_blocks=4), max_blocks=4, max_len=5000, window=40)
    assert rc not in (E_SHAPE, E_ARG, E_ALIGN, E_NULL), lib.pkv_last_error()


def test_slot_mapping_validation(lib):
    pool = _pool(ring_blocks=4)
    f = lib.paged_kv_slot_mapping
    assert f(ctypes.byref(pool), None, 4, None, FAKE, 8, FAKE, None) == E_NULL
    assert f(ctypes.byref(pool), FAKE, 4, None, FAKE + 4, 8, FAKE, None) == E_ALIGN
    assert f(ctypes.byref(pool), FAKE, 3, None, FAKE, 8, FAKE, None) == E_SHAPE
    assert f(ctypes.byref(pool), FAKE, 4, None, FAKE, 0, FAKE, None) == 0


def test_append_validation(lib):
    pool = _pool()
    assert lib.paged_kv_append(None, FAKE, FAKE, 4, ctypes.byref(pool), None) == E_NULL
    assert lib.paged_kv_append(FAKE, FAKE, FAKE + 4, 4, ctypes.byref(pool), None) == E_ALIGN
    assert lib.paged_kv_append(FAKE, FAKE, FAKE, -1, ctypes.byref(pool), None) == E_ARG
    # zero tokens: nothing to do, nothing launched
    assert lib.paged_kv_append(FAKE, FAKE, FAKE, 0, ctypes.byref(pool), None) == 0
    # K == V pool: v may be NULL
    alias = _pool(v=None, head_dim=100)
    assert lib.paged_kv_append(FAKE, None, FAKE, 4, ctypes.byref(alias), None) == E_UNSUPPORTED


def test_combine_validation(lib):
    c = lib.paged_decode_lse_combine
    assert c(None, FAKE, FAKE, 2, 4, 128, 16, 0, 64, 4, FAKE, 0, None) == E_NULL
    assert c(FAKE, FAKE, FAKE, 2, 4, 128, 16, 0, 60, 4, FAKE, 0, None) == E_ARG
    assert c(FAKE, FAKE, FAKE, 2, 4, 128, 16, 0, 64, 2000, FAKE, 0, None) == E_SHAPE
    assert c(FAKE, FAKE, FAKE, 2, 4, 128, 32, 0, 64, 4, FAKE, 0, None) == E_UNSUPPORTED


def test_split_geometry(lib):
    ns = lib.paged_decode_num_splits
    # global layer: ceil(len/16) blocks from block 0
    assert ns(16, 32768, 0, 1024) == 32
    assert ns(16, 4097, 0, 1024) == 5
    # sliding window w=1024: 1025 keys touch at most 65 blocks -> 2 splits of 64
    assert ns(16, 8192, 1024, 1024) == 2
    assert ns(16, 8192, 1024, 2048) == 1
    assert ns(16, 500, 1024, 256) == 2
    assert ns(16, 0, 0, 64) == 1
    # window not a multiple of the block: 1001 keys touch at most 64 blocks
    assert ns(16, 10000, 1000, 16) == 64
    st = lib.paged_decode_split_tokens
    assert st(8, 16, 8, 16, 8192, 1024, 0) == 0
    assert st(8, 16, 8, 16, 8192, 1024, 512) == 512
    assert st(8, 16, 8, 16, 8192, 1024, 500) == E_ARG


def test_workspace_bytes(lib):
    wb = lib.paged_decode_workspace_bytes
    pwb = lib.paged_decode_partial_workspace_bytes
    up = lambda x: (x + 255) // 256 * 256
    # CUDA-core shapes (group < 8): split partials, or for a single pass the
    # (sequence, length) order of the batch (256-byte rounded)
    assert wb(32, 16, 8, 256, 16, 32768, 0, 0) == 256
    assert wb(1000, 16, 8, 256, 16, 32768, 0, 0) == up(8 * 1000)
    assert wb(0, 16, 8, 256, 16, 32768, 0, 0) == 0
    assert pwb(32, 16, 8, 256) == 0
    rows = 32 * 16 * 32
    split_bytes = up(rows * 4) + rows * 256 * 4
    assert wb(32, 16, 8, 256, 16, 32768, 0, 1024) == split_bytes
    # tensor-core shapes (group 8..16, head_dim 128/256): the stream-K scratch
    # (plan of up to 256 CTAs, their publish flags, per-sequence prefix, two
    # partial states per CTA)
    grid, npad = 256, 16
    tc = (up(16 * (2 + grid)) + up(4 * 2 * grid) + up(4 * (32 + 1)) + up(4 * grid * 2 * npad)
          + 4 * grid * 2 * npad * 256)
    assert pwb(32, 16, 1, 256) == tc
    assert wb(32, 16, 1, 256, 16, 32768, 0, 0) == tc
    assert wb(32, 16, 1, 256, 16, 32768, 0, 1024) == max(split_bytes, tc)
    assert pwb(32, 16, 1, 64) == 0      # head_dim 64 runs on CUDA cores
    assert pwb(32, 64, 1, 128) == 0     # groups above 16 too


def test_binding_refuses_host_tensors():
    torch = pytest.importorskip("torch")
    k = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16)
    pool = pkv.PagedKVPool(k=k, v=k.clone())
    with pytest.raises(pkv.PagedKVError):
        pool.c_struct()


def test_oracle_is_not_reachable_from_the_product():
    """The product package never imports the oracle (no fallback path)."""
    import pathlib
    root = pathlib.Path(pkv.__file__).parent
    for f in list(root.glob("*.py")) + list((root / "csrc").glob("*")):
        text = f.read_text(errors="ignore")
        assert "import oracle" not in text and "from oracle" not in text, f
        assert "pkv_oracle" not in text and "_liboracle" not in text, f


def test_rope_validation(lib):
    """RoPE fused with the append: arguments rejected on the host."""
    pool = _pool()  # head_dim 128: at most 64 rotated pairs
    f = lib.paged_kv_append_rope

    def call(q=FAKE, q_out=FAKE, hq=4, k=FAKE, v=FAKE, pos=FAKE, slots=FAKE, n=4, table=FAKE,
             npos=100, pairs=16, layout=0):
        return f(q, q_out, hq, k, v, pos, slots, n, table, npos, pairs, layout,
                 ctypes.byref(pool), None)
    assert call(pairs=65) == E_ARG
    assert call(pairs=-1) == E_ARG
    assert call(layout=2) == E_ARG
    assert call(hq=0) == E_ARG
    assert call(n=-1) == E_ARG
    assert call(npos=-1) == E_ARG
    assert call(pos=None) == E_NULL
    assert call(q_out=None) == E_NULL
    assert call(table=None) == E_NULL
    assert call(q=FAKE + 8) == E_ALIGN
    assert call(pos=FAKE + 4) == E_ALIGN
    assert call(table=FAKE + 4) == E_ALIGN
    assert call(n=0) == 0
    t = lib.paged_rope_cos_sin_table
    assert t(FAKE, -1, 10, FAKE, None) == E_ARG
    assert t(None, 4, 10, FAKE, None) == E_NULL
    assert t(FAKE + 4, 4, 10, FAKE, None) == E_ALIGN
    assert t(FAKE, 0, 10, None, None) == 0


def test_step_validation(lib):
    """paged_decode_step checks every layer (and its optional RoPE fields)
    before anything is launched."""
    def layer(**kw):
        d = dict(pool=_pool(), q=FAKE, k_new=FAKE, v_new=FAKE, out=FAKE, window=0,
                 softmax_scale=0.1, rope_table=None, rope_num_positions=0, rope_pairs=0,
                 rope_layout=0, q_rotated=None)
        d.update(kw)
        return binding.PkvLayerC(**d)

    def step(*layers, slots=FAKE):
        arr = (binding.PkvLayerC * len(layers))(*layers)
        return lib.paged_decode_step(arr, len(layers), slots, FAKE, 8, FAKE, 2, 4, 100, 0, None, 0,
                                     0, None)
    assert step(layer(), slots=None) == E_NULL
    assert step(layer(), layer(k_new=None)) == E_NULL
    assert step(layer(), layer(k_new=FAKE + 8)) == E_ALIGN
    rope = dict(rope_table=FAKE, rope_num_positions=100, rope_pairs=16, q_rotated=FAKE)
    assert step(layer(**{**rope, "rope_pairs": 65})) == E_ARG
    assert step(layer(**{**rope, "rope_layout": 3})) == E_ARG
    assert step(layer(**{**rope, "q_rotated": None})) == E_NULL
    assert step(layer(**{**rope, "q_rotated": FAKE + 8})) == E_ALIGN
    assert step(layer(**{**rope, "rope_table": FAKE + 4})) == E_ALIGN
