"""CPU oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
there is no fallback from the CUDA path to this code.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64 attention, fp32
quantiser); this module only marshals numpy arrays into it.  Every function
is pinned by ``tests/test_oracle_pins.py`` against values that the pages or
the mathematics fix (closed forms, invariants, a library attention routine on
special cases, hand-derived quantiser vectors).

Array conventions (numpy, C-contiguous):
  bf16 data is passed as uint16 bit patterns;
  pool k / v: [num_blocks, block_size, num_kv_heads, head_dim], uint16 or int8;
  q: [B, H_q, D] uint16; block_table: [B, max_blocks] int32; seq_lens: [B] int32.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

from . import build as _build

_lib = None


class _COraclePool(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("is_int8", ctypes.c_int32),
        ("scale_mode", ctypes.c_int32),
        ("ring_blocks", ctypes.c_int32),
    ]


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        p, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_per_token_scale.argtypes = [p, i64]
        lib.oracle_per_token_scale.restype = ctypes.c_float
        lib.oracle_quantize.argtypes = [p, i64, ctypes.c_float, p]
        lib.oracle_quantize.restype = None
        lib.oracle_append.argtypes = [p, p, p, i32, p]
        lib.oracle_append.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [p, p, p, i32, p, i32, i32, i32, f64, p, i32, p, i32]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_partial.argtypes = [p, p, p, i32, p, i32, i32, i32, f64, p, p, p, p, i32]
        lib.oracle_partial.restype = ctypes.c_int
        lib.oracle_lse_combine.argtypes = [p, p, i32, i32, p, p]
        lib.oracle_lse_combine.restype = None
        lib.oracle_prefill.argtypes = [p, p, p, i32, p, p, i32, i32, i32, f64, p, i32]
        lib.oracle_prefill.restype = ctypes.c_int
        lib.oracle_slot_mapping.argtypes = [p, p, i32, p, p, i64, p]
        lib.oracle_slot_mapping.restype = None
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_rope_table.argtypes = [p, i32, i64, p, p]
        lib.oracle_rope_table.restype = None
        lib.oracle_rope.argtypes = [p, p, i64, i32, i32, p, p, i64, i32, i32]
        lib.oracle_rope.restype = ctypes.c_int
        lib.oracle_rope_exact.argtypes = [p, p, i32, f64, p, i32, i32]
        lib.oracle_rope_exact.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


SCALE_NONE, SCALE_PER_TOKEN, SCALE_PER_HEAD = 0, 1, 2


@dataclass
class OraclePool:
    """Paged KV pool as numpy arrays (one layer).

    k, v: [num_blocks, block_size, num_kv_heads, head_dim], uint16 (bf16 bits)
    or int8; v None means K and V are one tensor.  Scale tables: per token
    [num_blocks * block_size] fp32, per head [num_kv_heads] fp32.
    """
    k: np.ndarray
    v: Optional[np.ndarray] = None
    k_scale: Optional[np.ndarray] = None
    v_scale: Optional[np.ndarray] = None
    scale_mode: int = SCALE_NONE
    ring_blocks: int = 0  # 0: paged; > 0: each sequence's ring of this many blocks

    @property
    def is_int8(self) -> bool:
        return self.k.dtype == np.int8

    def _c(self) -> _COraclePool:
        nb, p, hkv, d = self.k.shape
        for a in (self.v,):
            if a is not None:
                assert a.shape == self.k.shape and a.dtype == self.k.dtype
        for s in (self.k_scale, self.v_scale):
            if s is not None:
                assert s.dtype == np.float32
        return _COraclePool(_ptr(self.k), _ptr(self.v), _ptr(self.k_scale), _ptr(self.v_scale),
                            nb, p, hkv, d, int(self.is_int8), int(self.scale_mode),
                            int(self.ring_blocks))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns as float64 (bf16 = top half of fp32)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def per_token_scale(x_bits: np.ndarray) -> np.float32:
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    return np.float32(_load().oracle_per_token_scale(_ptr(x_bits), x_bits.size))


def quantize(x_bits: np.ndarray, scale: float) -> np.ndarray:
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q = np.empty(x_bits.shape, np.int8)
    _load().oracle_quantize(_ptr(x_bits), x_bits.size, ctypes.c_float(scale), _ptr(q))
    return q


def slot_mapping(pool: OraclePool, block_table: np.ndarray, seq: np.ndarray,
                 pos: np.ndarray) -> np.ndarray:
    """Slot ids of tokens (sequence seq[i], absolute position pos[i]) under the
    pool's layout: paged, or the ring (position t in slot t mod W of the
    sequence's ring of W = ring_blocks * block_size slots); -1 for a negative
    position or an unallocated table entry."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    seq = np.ascontiguousarray(seq, dtype=np.int32)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    out = np.empty(len(pos), np.int64)
    _load().oracle_slot_mapping(ctypes.byref(pool._c()), _ptr(bt), bt.shape[1], _ptr(seq),
                                _ptr(pos), len(pos), _ptr(out))
    return out


def append(k_bits: np.ndarray, v_bits: Optional[np.ndarray], slot_mapping: np.ndarray,
           pool: OraclePool) -> None:
    """Scatter (and quantise) T new tokens into ``pool`` in place.

    k_bits, v_bits: [T, num_kv_heads, head_dim] uint16; slot_mapping: [T] int64."""
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = None if v_bits is None else np.ascontiguousarray(v_bits, dtype=np.uint16)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = _load().oracle_append(_ptr(k_bits), _ptr(v_bits), _ptr(slots), len(slots),
                               ctypes.byref(pool._c()))
    if rc != 0:
        raise ValueError(f"oracle_append failed ({rc})")


def decode(q_bits: np.ndarray, pool: OraclePool, block_table: np.ndarray, seq_lens: np.ndarray,
           num_q_heads: int, window: int, softmax_scale: float,
           rows: Optional[np.ndarray] = None, num_threads: int = 0) -> np.ndarray:
    """fp64 decode attention.  Returns [B, H_q, D], or [len(rows), D] when
    ``rows`` (an [n, 2] array of (b, h) pairs) selects a sample of rows."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = sl.shape[0]
    D = pool.k.shape[3]
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        out = np.zeros((rows.shape[0], D), np.float64)
        n = rows.shape[0]
    else:
        out = np.zeros((B, num_q_heads, D), np.float64)
        n = B * num_q_heads
    rc = _load().oracle_decode(_ptr(q_bits), ctypes.byref(pool._c()), _ptr(bt), bt.shape[1],
                               _ptr(sl), B, num_q_heads, window, float(softmax_scale),
                               _ptr(rows), n, _ptr(out), num_threads)
    if rc != 0:
        raise ValueError(f"oracle_decode failed ({rc})")
    return out


def prefill(q_bits: np.ndarray, pool: OraclePool, block_table: np.ndarray, seq_lens: np.ndarray,
            q_start: np.ndarray, num_q_heads: int, window: int, softmax_scale: float,
            num_threads: int = 0) -> np.ndarray:
    """fp64 attention of each sequence's chunk of new tokens: q_bits
    [total, H_q, D] (rows q_start[b] .. q_start[b+1]-1 are sequence b's last
    tokens, causal among themselves).  Returns [total, H_q, D]."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qs = np.ascontiguousarray(q_start, dtype=np.int32)
    D = pool.k.shape[3]
    out = np.zeros((q_bits.shape[0], num_q_heads, D), np.float64)
    rc = _load().oracle_prefill(_ptr(q_bits), ctypes.byref(pool._c()), _ptr(bt), bt.shape[1],
                                _ptr(sl), _ptr(qs), len(sl), num_q_heads, window,
                                float(softmax_scale), _ptr(out), num_threads)
    if rc != 0:
        raise ValueError(f"oracle_prefill failed ({rc})")
    return out


def partial(q_bits: np.ndarray, pool: OraclePool, block_table: np.ndarray, seq_lens: np.ndarray,
            num_q_heads: int, window: int, softmax_scale: float, key_begin: np.ndarray,
            key_end: np.ndarray, num_threads: int = 0):
    """Per-row partial state over key ranges [key_begin[b], key_end[b]).
    Returns (lse [B, H_q] natural log, o [B, H_q, D] normalised)."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    kb = np.ascontiguousarray(key_begin, dtype=np.int64)
    ke = np.ascontiguousarray(key_end, dtype=np.int64)
    B = sl.shape[0]
    D = pool.k.shape[3]
    lse = np.zeros((B, num_q_heads), np.float64)
    o = np.zeros((B, num_q_heads, D), np.float64)
    rc = _load().oracle_partial(_ptr(q_bits), ctypes.byref(pool._c()), _ptr(bt), bt.shape[1],
                                _ptr(sl), B, num_q_heads, window, float(softmax_scale),
                                _ptr(kb), _ptr(ke), _ptr(lse), _ptr(o), num_threads)
    if rc != 0:
        raise ValueError(f"oracle_partial failed ({rc})")
    return lse, o


def lse_combine(lse: np.ndarray, o: np.ndarray):
    """Merge partial states of one row: lse [n], o [n, D] -> (y [D], lse_total)."""
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    n, D = o.shape
    out = np.zeros(D, np.float64)
    tot = ctypes.c_double()
    _load().oracle_lse_combine(_ptr(lse), _ptr(o), n, D, _ptr(out), ctypes.byref(tot))
    return out, tot.value


ROPE_HALVES, ROPE_INTERLEAVED = 0, 1
E_POS = -4


def f32_to_bf16(x: float) -> int:
    """bf16 bit pattern of an fp32 value, round to nearest, ties to even."""
    return int(_load().oracle_f32_to_bf16(ctypes.c_float(x)))


def rope_table(theta: np.ndarray, num_positions: int):
    """RoPE cos / sin table: ([num_positions, pairs, 2] fp32, [num_positions,
    pairs] bool).  Entry (m, i) holds fp32(cos(m theta_i)), fp32(sin(m
    theta_i)); the flag marks entries so close to an fp32 rounding midpoint
    that another faithful fp64 cos / sin may round them the other way."""
    theta = np.ascontiguousarray(theta, dtype=np.float64)
    pairs = theta.shape[0]
    table = np.zeros((num_positions, pairs, 2), np.float32)
    amb = np.zeros((num_positions, pairs), np.uint8)
    _load().oracle_rope_table(_ptr(theta), pairs, num_positions, _ptr(table), _ptr(amb))
    return table, amb.astype(bool)


def rope(x_bits: np.ndarray, positions: np.ndarray, table: np.ndarray, layout: int = ROPE_HALVES):
    """Rotate x_bits [T, H, D] (bf16 bits) by the positions [T] with the
    table [npos, pairs, 2]; returns (rotated bits, status).  Rows at a
    negative position, or at one past the table (status E_POS), are copied."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H, D = x_bits.shape
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    table = np.ascontiguousarray(table, dtype=np.float32)
    y = np.empty_like(x_bits)
    rc = _load().oracle_rope(_ptr(x_bits), _ptr(y), T, H, D, _ptr(pos), _ptr(table),
                             table.shape[0], table.shape[1], layout)
    if rc not in (0, E_POS):
        raise ValueError(f"oracle_rope failed ({rc})")
    return y, rc


def rope_exact(x: np.ndarray, position: float, theta: np.ndarray, pairs: int,
               layout: int = ROPE_HALVES) -> np.ndarray:
    """fp64 rotation of one vector x [D] at a position, without rounding."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    theta = np.ascontiguousarray(theta, dtype=np.float64)
    assert theta.shape[0] >= pairs
    y = np.empty_like(x)
    _load().oracle_rope_exact(_ptr(x), _ptr(y), x.shape[0], float(position), _ptr(theta), pairs,
                              layout)
    return y


def append_rope(q_bits: Optional[np.ndarray], k_bits: np.ndarray, v_bits: Optional[np.ndarray],
                positions: np.ndarray, slot_mapping: np.ndarray, pool: OraclePool,
                table: np.ndarray, layout: int = ROPE_HALVES):
    """RoPE fused with the append, as the composition of its two steps: q and
    k rotated by their positions, then the rotated k (and the unrotated v)
    appended.  A token at a negative position, or past the table, appends
    nothing and its q row is copied.  Returns (q_out bits or None, status)."""
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    q_out, rc_q = (None, 0) if q_bits is None else rope(q_bits, pos, table, layout)
    k_rot, rc_k = rope(k_bits, pos, table, layout)
    valid = (pos >= 0) & (pos < table.shape[0])
    slots = np.where(valid, np.asarray(slot_mapping, dtype=np.int64), -1)
    append(k_rot, v_bits, slots, pool)
    return q_out, (rc_q or rc_k)


def max_threads() -> int:
    return int(_load().oracle_max_threads())
