"""ctypes binding of libpagedkv.so (include/pagedkv.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, and status codes become exceptions.  Every
step of the computation runs in the library's kernels; nothing here computes
attention, and there is no CPU fallback -- if the library is missing or a
tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedkv.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pagedkv.h")

PKV_BF16, PKV_INT8 = 0, 1
SCALE_NONE, SCALE_PER_TOKEN, SCALE_PER_HEAD = 0, 1, 2
OUT_BF16, OUT_F32 = 0, 1
ROPE_HALVES, ROPE_INTERLEAVED = 0, 1
SPLIT_AUTO = -1

_lib = None


class PkvPoolC(ctypes.Structure):
    """Mirror of ``pkv_pool`` in include/pagedkv.h."""
    _fields_ = [
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("scale_mode", ctypes.c_int32),
        ("ring_blocks", ctypes.c_int32),
    ]


class PkvLayerC(ctypes.Structure):
    """Mirror of ``pkv_layer`` in include/pagedkv.h."""
    _fields_ = [
        ("pool", PkvPoolC),
        ("q", ctypes.c_void_p),
        ("k_new", ctypes.c_void_p),
        ("v_new", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("window", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("rope_table", ctypes.c_void_p),
        ("rope_num_positions", ctypes.c_int64),
        ("rope_pairs", ctypes.c_int32),
        ("rope_layout", ctypes.c_int32),
        ("q_rotated", ctypes.c_void_p),
    ]


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load libpagedkv.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    p, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.paged_kv_append.argtypes = [p, p, p, i32, p, p]
    lib.paged_kv_append.restype = ctypes.c_int
    lib.paged_decode_split_tokens.argtypes = [i32] * 7
    lib.paged_decode_split_tokens.restype = i32
    lib.paged_decode_num_splits.argtypes = [i32] * 4
    lib.paged_decode_num_splits.restype = i32
    lib.paged_decode_workspace_bytes.argtypes = [i32] * 8
    lib.paged_decode_workspace_bytes.restype = sz
    lib.paged_decode_attention.argtypes = [p, p, p, i32, p, i32, i32, i32, i32, f32, i32, p, sz,
                                           p, i32, p]
    lib.paged_decode_attention.restype = ctypes.c_int
    lib.paged_decode_partial_workspace_bytes.argtypes = [i32] * 4
    lib.paged_decode_partial_workspace_bytes.restype = sz
    lib.paged_decode_split_partial.argtypes = [p, p, p, i32, p, i32, i32, i32, i32, f32, i32, p,
                                               p, i32, p, sz, p, i32, p]
    lib.paged_decode_split_partial.restype = ctypes.c_int
    lib.paged_decode_lse_combine.argtypes = [p, p, p, i32, i32, i32, i32, i32, i32, i32, p, i32,
                                             p]
    lib.paged_decode_lse_combine.restype = ctypes.c_int
    lib.paged_decode_attention_noalloc.argtypes = [p, p, p, i32, p, i32, i32, i32, i32, f32,
                                                   i32, p, i32, p]
    lib.paged_decode_attention_noalloc.restype = ctypes.c_int
    lib.pkv_check_bounded_wait.argtypes = [ctypes.c_uint64, i32, p, i32, p]
    lib.pkv_check_bounded_wait.restype = ctypes.c_int
    lib.paged_prefill_attention.argtypes = [p, p, i32, i32, p, p, i32, p, i32, i32, i32, i32, f32,
                                            p, i32, p]
    lib.paged_prefill_attention.restype = ctypes.c_int
    i64 = ctypes.c_int64
    lib.paged_rope_cos_sin_table.argtypes = [p, i32, i64, p, p]
    lib.paged_rope_cos_sin_table.restype = ctypes.c_int
    lib.paged_kv_append_rope.argtypes = [p, p, i32, p, p, p, p, i32, p, i64, i32, i32, p, p]
    lib.paged_kv_append_rope.restype = ctypes.c_int
    lib.paged_kv_slot_mapping.argtypes = [p, p, i32, p, p, i32, p, p]
    lib.paged_kv_slot_mapping.restype = ctypes.c_int
    lib.paged_decode_step_workspace_bytes.argtypes = [p, i32, i32, i32, i32, i32]
    lib.paged_decode_step_workspace_bytes.restype = sz
    lib.paged_decode_step.argtypes = [p, i32, p, p, i32, p, i32, i32, i32, i32, p, sz, i32, p]
    lib.paged_decode_step.restype = ctypes.c_int
    lib.paged_decode_uses_tensor_cores.argtypes = [p, i32]
    lib.paged_decode_uses_tensor_cores.restype = i32
    lib.pkv_last_launch_count.argtypes = []
    lib.pkv_last_launch_count.restype = i32
    lib.pkv_last_error.argtypes = []
    lib.pkv_last_error.restype = ctypes.c_char_p
    lib.pkv_device_status.argtypes = [i32]
    lib.pkv_device_status.restype = ctypes.c_int
    _lib = lib
    return lib


def exported_symbols():
    """Names of the functions include/pagedkv.h declares with PKV_API."""
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"PKV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


class PagedKVError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        msg = load_library().pkv_last_error().decode(errors="replace")
        raise PagedKVError(f"{what} failed ({rc}): {msg}")


def _dev_ptr(t, name):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise PagedKVError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise PagedKVError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


@dataclass
class PagedKVPool:
    """One layer's KV pool as torch device tensors.

    k, v: [num_blocks, block_size, num_kv_heads, head_dim], bf16 or int8;
    v None means K and V are one tensor.  int8 pools carry fp32 scale tables
    (per token: [num_blocks * block_size]; per head: [num_kv_heads]).
    ring_blocks: 0 for the paged layout; > 0 for a sliding layer's ring
    layout (each block-table row is the sequence's ring of that many blocks,
    position t in slot t mod (ring_blocks * block_size)).
    """
    k: "object"
    v: Optional[object] = None
    k_scale: Optional[object] = None
    v_scale: Optional[object] = None
    scale_mode: int = SCALE_NONE
    ring_blocks: int = 0

    @property
    def dtype(self) -> int:
        import torch
        return PKV_INT8 if self.k.dtype == torch.int8 else PKV_BF16

    @property
    def num_blocks(self) -> int:
        return int(self.k.shape[0])

    @property
    def block_size(self) -> int:
        return int(self.k.shape[1])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k.shape[2])

    @property
    def head_dim(self) -> int:
        return int(self.k.shape[3])

    def c_struct(self) -> PkvPoolC:
        import torch
        if self.k.dim() != 4:
            raise PagedKVError("pool k must be [num_blocks, block_size, num_kv_heads, head_dim]")
        if self.k.dtype not in (torch.bfloat16, torch.int8):
            raise PagedKVError("pool dtype must be bfloat16 or int8")
        if self.v is not None and (self.v.shape != self.k.shape or self.v.dtype != self.k.dtype):
            raise PagedKVError("pool v must match k")
        for s in (self.k_scale, self.v_scale):
            if s is not None and s.dtype != torch.float32:
                raise PagedKVError("scale tables must be float32")
        return PkvPoolC(_dev_ptr(self.k, "pool.k"), _dev_ptr(self.v, "pool.v"),
                        _dev_ptr(self.k_scale, "pool.k_scale"), _dev_ptr(self.v_scale, "pool.v_scale"),
                        self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim,
                        self.dtype, int(self.scale_mode), int(self.ring_blocks))


def paged_kv_append(k, v, slot_mapping, pool: PagedKVPool, stream=None) -> None:
    """Write the new tokens' K/V ([T, H_kv, D] bf16) into slots ``slot_mapping``
    ([T] int64) of ``pool``, quantising to int8 if the pool is int8."""
    lib = load_library()
    pc = pool.c_struct()
    n = int(slot_mapping.shape[0])
    _check(lib.paged_kv_append(_dev_ptr(k, "k"), _dev_ptr(v, "v"), _dev_ptr(slot_mapping, "slot_mapping"),
                               n, ctypes.byref(pc), _stream(stream)), "paged_kv_append")


def paged_rope_cos_sin_table(theta, num_positions: int, table=None, stream=None):
    """(cos, sin) of every position's angles: ``theta`` [pairs] float64 on the
    device (radians per position); returns ``table`` [num_positions, pairs, 2]
    float32 (allocated if None)."""
    import torch
    pairs = int(theta.shape[0])
    if theta.dtype != torch.float64:
        raise PagedKVError("theta must be float64")
    if table is None:
        table = torch.empty((num_positions, pairs, 2), dtype=torch.float32, device=theta.device)
    if tuple(table.shape) != (num_positions, pairs, 2) or table.dtype != torch.float32:
        raise PagedKVError("table must be [num_positions, pairs, 2] float32")
    _check(load_library().paged_rope_cos_sin_table(_dev_ptr(theta, "theta"), pairs, num_positions,
                                                   _dev_ptr(table, "table"), _stream(stream)),
           "paged_rope_cos_sin_table")
    return table


def paged_kv_append_rope(q, q_out, k, v, positions, slot_mapping, pool: PagedKVPool, table,
                         layout: int = ROPE_HALVES, stream=None) -> None:
    """RoPE fused with the append: q ([T, H_q, D] bf16, or None) rotated into
    ``q_out`` (may be q), k ([T, H_kv, D]) rotated and appended with v at
    ``slot_mapping``, every token at its ``positions`` entry ([T] int64),
    with the (cos, sin) ``table`` of paged_rope_cos_sin_table ([npos, pairs,
    2]; its pairs are the rotated ones)."""
    lib = load_library()
    pc = pool.c_struct()
    n = int(slot_mapping.shape[0])
    hq = int(q.shape[1]) if q is not None else 0
    npos, pairs = int(table.shape[0]), int(table.shape[1])
    _check(lib.paged_kv_append_rope(_dev_ptr(q, "q"), _dev_ptr(q_out, "q_out"), hq,
                                    _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                    _dev_ptr(positions, "positions"),
                                    _dev_ptr(slot_mapping, "slot_mapping"), n,
                                    _dev_ptr(table, "table"), npos, pairs, int(layout),
                                    ctypes.byref(pc), _stream(stream)), "paged_kv_append_rope")


def paged_kv_slot_mapping(pool: PagedKVPool, block_table, positions, slot_mapping,
                          seq_ids=None, stream=None):
    """Slots ([T] int64, written into ``slot_mapping``) of tokens at absolute
    ``positions`` ([T] int64) of sequences ``seq_ids`` ([T] int32; None =
    token i of sequence i) under the pool's layout (paged, or the ring
    t mod W), computed on the device."""
    lib = load_library()
    pc = pool.c_struct()
    _check(lib.paged_kv_slot_mapping(ctypes.byref(pc), _dev_ptr(block_table, "block_table"),
                                     int(block_table.shape[1]), _dev_ptr(seq_ids, "seq_ids"),
                                     _dev_ptr(positions, "positions"), int(positions.shape[0]),
                                     _dev_ptr(slot_mapping, "slot_mapping"), _stream(stream)),
           "paged_kv_slot_mapping")
    return slot_mapping


def paged_decode_split_tokens(batch, num_q_heads, num_kv_heads, max_seq_len, window,
                              split_tokens=SPLIT_AUTO, block_size=16) -> int:
    st = load_library().paged_decode_split_tokens(batch, num_q_heads, num_kv_heads, block_size,
                                                  max_seq_len, window, split_tokens)
    if st < 0:
        _check(st, "paged_decode_split_tokens")
    return st


def paged_decode_num_splits(max_seq_len, window, split_tokens, block_size=16) -> int:
    return int(load_library().paged_decode_num_splits(block_size, max_seq_len, window, split_tokens))


def paged_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_seq_len, window,
                                 split_tokens=SPLIT_AUTO, block_size=16) -> int:
    return int(load_library().paged_decode_workspace_bytes(batch, num_q_heads, num_kv_heads,
                                                           head_dim, block_size, max_seq_len,
                                                           window, split_tokens))


def paged_decode_attention(q, pool: PagedKVPool, block_table, seq_lens, window: int,
                           softmax_scale: float, out, max_seq_len: int,
                           split_tokens: int = SPLIT_AUTO, workspace=None, stream=None):
    """Decode attention of q [B, H_q, D] (bf16) over ``pool`` into ``out``
    ([B, H_q, D], bf16 or fp32).  ``max_seq_len`` is the host-side bound on
    seq_lens.  ``workspace``: a uint8 CUDA tensor of at least
    paged_decode_workspace_bytes(...) bytes (allocated through torch if None)."""
    import torch
    lib = load_library()
    pc = pool.c_struct()
    B, Hq, D = (int(x) for x in q.shape)
    need = lib.paged_decode_workspace_bytes(B, Hq, pool.num_kv_heads, D, pool.block_size,
                                            max_seq_len, window, split_tokens)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _dev_ptr(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(lib.paged_decode_attention(_dev_ptr(q, "q"), ctypes.byref(pc), _dev_ptr(block_table, "block_table"),
                                      int(block_table.shape[1]), _dev_ptr(seq_lens, "seq_lens"), B, Hq,
                                      int(max_seq_len), int(window), float(softmax_scale),
                                      int(split_tokens), ws_ptr, ws_bytes, _dev_ptr(out, "out"),
                                      out_dtype, _stream(stream)), "paged_decode_attention")
    return out


def last_launch_count() -> int:
    """Kernels launched by this thread's last call into the library."""
    return int(load_library().pkv_last_launch_count())


def uses_tensor_cores(pool: PagedKVPool, num_q_heads: int) -> bool:
    """Whether decodes over ``pool`` run on the tensor-core kernel."""
    lib = load_library()
    pc = pool.c_struct()
    r = int(lib.paged_decode_uses_tensor_cores(ctypes.byref(pc), int(num_q_heads)))
    _check(min(r, 0), "paged_decode_uses_tensor_cores")
    return r == 1


def paged_decode_partial_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim) -> int:
    return int(load_library().paged_decode_partial_workspace_bytes(batch, num_q_heads,
                                                                   num_kv_heads, head_dim))


def paged_decode_split_partial(q, pool: PagedKVPool, block_table, seq_lens, window: int,
                               softmax_scale: float, split_tokens: int, partial_lse, partial_o,
                               out, max_seq_len: int, workspace=None, stream=None):
    """Split-KV step 1: partial_lse [B, S, H_q] and partial_o [B, S, H_q, D]
    (fp32, split-major) for multi-split sequences; final rows of single-split
    ones in out.
    ``workspace``: a uint8 CUDA tensor of at least
    paged_decode_partial_workspace_bytes(...) bytes (allocated through torch
    if None and needed)."""
    import torch
    lib = load_library()
    pc = pool.c_struct()
    B, Hq, D = (int(x) for x in q.shape)
    ns = int(partial_lse.shape[1])
    need = lib.paged_decode_partial_workspace_bytes(B, Hq, pool.num_kv_heads, D)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = _dev_ptr(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(lib.paged_decode_split_partial(_dev_ptr(q, "q"), ctypes.byref(pc), _dev_ptr(block_table, "block_table"),
                                          int(block_table.shape[1]), _dev_ptr(seq_lens, "seq_lens"), B, Hq,
                                          int(max_seq_len), int(window), float(softmax_scale),
                                          int(split_tokens), _dev_ptr(partial_lse, "partial_lse"),
                                          _dev_ptr(partial_o, "partial_o"), ns, ws_ptr, ws_bytes,
                                          _dev_ptr(out, "out"), out_dtype, _stream(stream)),
           "paged_decode_split_partial")


def paged_decode_lse_combine(partial_lse, partial_o, seq_lens, window: int, split_tokens: int, out,
                             block_size: int = 16, stream=None):
    """Split-KV step 2: merge the partials (split-major, as step 1 writes them)
    of multi-split sequences into out."""
    import torch
    lib = load_library()
    B, ns, Hq = (int(x) for x in partial_lse.shape)
    D = int(partial_o.shape[3])
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(lib.paged_decode_lse_combine(_dev_ptr(partial_lse, "partial_lse"), _dev_ptr(partial_o, "partial_o"),
                                        _dev_ptr(seq_lens, "seq_lens"), B, Hq, D, block_size, int(window),
                                        int(split_tokens), ns, _dev_ptr(out, "out"), out_dtype,
                                        _stream(stream)), "paged_decode_lse_combine")


STATIC_SCRATCH_BYTES = 32 << 20  # PKV_STATIC_SCRATCH_BYTES in include/pagedkv.h


def paged_decode_attention_noalloc(q, pool: PagedKVPool, block_table, seq_lens, window: int,
                                   softmax_scale: float, out, max_seq_len: int,
                                   split_tokens: int = SPLIT_AUTO, stream=None):
    """paged_decode_attention without a workspace, for callers that cannot
    allocate device memory (a plugin handed only its inputs and outputs, an
    engine that reserved all of HBM for its KV pool, a loop where an
    allocation would synchronise the device).  Split partials go to the
    library's fixed per-device scratch array (STATIC_SCRATCH_BYTES); sizes
    that do not fit raise.  Calls share that array: do not let two of them
    overlap on the GPU.  The first call on a device looks the array up; make
    it before any stream capture."""
    import torch
    lib = load_library()
    pc = pool.c_struct()
    B, Hq, D = (int(x) for x in q.shape)
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(lib.paged_decode_attention_noalloc(
        _dev_ptr(q, "q"), ctypes.byref(pc), _dev_ptr(block_table, "block_table"),
        int(block_table.shape[1]), _dev_ptr(seq_lens, "seq_lens"), B, Hq, int(max_seq_len),
        int(window), float(softmax_scale), int(split_tokens), _dev_ptr(out, "out"), out_dtype,
        _stream(stream)), "paged_decode_attention_noalloc")
    return out


def device_status(clear: bool = True) -> int:
    """Device error word (PKV_DEV_* bits); synchronises the device."""
    rc = load_library().pkv_device_status(1 if clear else 0)
    if rc < 0:
        _check(rc, "pkv_device_status")
    return rc


@dataclass
class DecodeLayer:
    """One layer of a decode step: its pool, query [B, H_q, D] bf16, new
    token K/V [B, H_kv, D] bf16 (v_new None when K and V are one tensor),
    output [B, H_q, D] (bf16 or fp32), window (0 = global) and softmax scale.
    Optional RoPE fused with the append: ``rope_table`` from
    paged_rope_cos_sin_table ([npos, pairs, 2]), pairing ``rope_layout``, and
    ``q_rotated`` ([B, H_q, D] bf16, may be q) that receives the rotated q the
    decode reads; the new tokens sit at positions seq_lens - 1."""
    pool: PagedKVPool
    q: "object"
    k_new: "object"
    v_new: Optional[object]
    out: "object"
    window: int
    softmax_scale: float
    rope_table: Optional[object] = None
    rope_layout: int = ROPE_HALVES
    q_rotated: Optional[object] = None

    def c_struct(self) -> PkvLayerC:
        npos = pairs = 0
        if self.rope_table is not None:
            npos, pairs = int(self.rope_table.shape[0]), int(self.rope_table.shape[1])
        return PkvLayerC(self.pool.c_struct(), _dev_ptr(self.q, "q"), _dev_ptr(self.k_new, "k_new"),
                         _dev_ptr(self.v_new, "v_new"), _dev_ptr(self.out, "out"), int(self.window),
                         float(self.softmax_scale), _dev_ptr(self.rope_table, "rope_table"), npos,
                         pairs, int(self.rope_layout), _dev_ptr(self.q_rotated, "q_rotated"))


def _layers_c(layers):
    arr = (PkvLayerC * len(layers))()
    for i, layer in enumerate(layers):
        arr[i] = layer.c_struct()
    return arr


def paged_decode_step_workspace_bytes(layers, max_seq_len: int,
                                      split_tokens: int = SPLIT_AUTO) -> int:
    B, Hq = (int(x) for x in layers[0].q.shape[:2])
    return int(load_library().paged_decode_step_workspace_bytes(
        _layers_c(layers), len(layers), B, Hq, int(max_seq_len), int(split_tokens)))


def paged_decode_step(layers, slot_mapping, block_table, seq_lens, max_seq_len: int,
                      split_tokens: int = SPLIT_AUTO, workspace=None, stream=None) -> None:
    """One decode step of every layer: append each layer's new tokens at
    ``slot_mapping`` ([B] int64), then decode it, over one shared layout
    (``block_table``, ``seq_lens``), in one library call that a CUDA graph
    can capture.  ``workspace``: uint8 CUDA tensor of at least
    paged_decode_step_workspace_bytes(...) bytes (allocated through torch if
    None and needed)."""
    import torch
    lib = load_library()
    arr = _layers_c(layers)
    B, Hq = (int(x) for x in layers[0].q.shape[:2])
    for layer in layers:
        if layer.out.dtype != layers[0].out.dtype:
            raise PagedKVError("all layers' outputs must have one dtype")
    need = lib.paged_decode_step_workspace_bytes(arr, len(layers), B, Hq, int(max_seq_len),
                                                 int(split_tokens))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=layers[0].q.device)
    ws_ptr = _dev_ptr(workspace, "workspace") if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    out_dtype = OUT_F32 if layers[0].out.dtype == torch.float32 else OUT_BF16
    _check(lib.paged_decode_step(arr, len(layers), _dev_ptr(slot_mapping, "slot_mapping"),
                                 _dev_ptr(block_table, "block_table"), int(block_table.shape[1]),
                                 _dev_ptr(seq_lens, "seq_lens"), B, Hq, int(max_seq_len),
                                 int(split_tokens), ws_ptr, ws_bytes, out_dtype, _stream(stream)),
           "paged_decode_step")


def paged_prefill_attention(q, q_start, pool: PagedKVPool, block_table, seq_lens, window: int,
                            softmax_scale: float, out, max_seq_len: int, max_q_len: int,
                            stream=None):
    """Attention of each sequence's chunk of new tokens (q_len > 1): q
    [total, H_q, D] bf16, rows q_start[b] .. q_start[b+1]-1 ([B + 1] int32)
    are sequence b's last tokens (already appended), causal among
    themselves; out [total, H_q, D] bf16 or fp32.  ``max_q_len`` bounds every
    chunk's length on the host."""
    import torch
    lib = load_library()
    pc = pool.c_struct()
    total, Hq, _ = (int(x) for x in q.shape)
    B = int(seq_lens.shape[0])
    out_dtype = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(lib.paged_prefill_attention(_dev_ptr(q, "q"), _dev_ptr(q_start, "q_start"), total,
                                       int(max_q_len), ctypes.byref(pc),
                                       _dev_ptr(block_table, "block_table"), int(block_table.shape[1]),
                                       _dev_ptr(seq_lens, "seq_lens"), B, Hq, int(max_seq_len),
                                       int(window), float(softmax_scale), _dev_ptr(out, "out"),
                                       out_dtype, _stream(stream)), "paged_prefill_attention")
    return out


def check_bounded_wait(limit_ns: int, spin: bool, out, stream=None) -> None:
    """Run the pipelines' bounded wait out on purpose (see
    pkv_check_bounded_wait): ``out`` is an int32 CUDA tensor, one entry per
    waiting thread, set to 1 where the wait gave up."""
    _check(load_library().pkv_check_bounded_wait(int(limit_ns), 1 if spin else 0,
                                                 _dev_ptr(out, "out"), int(out.numel()),
                                                 _stream(stream)), "pkv_check_bounded_wait")
