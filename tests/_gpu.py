"""GPU-side helpers for the parity tests: move a synthetic workload to the
device and run the library's entry points on it.  No oracle code here."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_decode_03_gb300 as pkv
from paged_kv_decode_03_gb300 import synth


def to_dev_bits(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 CUDA tensor (same bits)."""
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def device_pool(w: synth.Workload) -> pkv.PagedKVPool:
    """Poisoned device pool for the workload (nothing appended yet)."""
    k, v, ks, vs = synth.empty_pool_arrays(w.spec, w.layout)
    mode = {"bf16": pkv.SCALE_NONE, "int8_token": pkv.SCALE_PER_TOKEN,
            "int8_head": pkv.SCALE_PER_HEAD}[w.spec.kv]
    if w.spec.kv == "int8_head":
        ks = w.k_head_scale.copy()
        vs = None if w.spec.alias else w.v_head_scale.copy()
    conv = to_dev_bits if k.dtype == np.uint16 else to_dev
    return pkv.PagedKVPool(k=conv(k), v=None if v is None else conv(v),
                           k_scale=None if ks is None else to_dev(ks),
                           v_scale=None if vs is None else to_dev(vs), scale_mode=mode,
                           ring_blocks=w.spec.ring_blocks)


def library_slots(w: synth.Workload, pool: pkv.PagedKVPool, seq, pos) -> torch.Tensor:
    """Slots of (sequence, position) pairs from the library's own address map
    (paged_kv_slot_mapping), on the device."""
    slots = torch.empty(len(pos), dtype=torch.int64, device="cuda")
    if len(pos):
        pkv.paged_kv_slot_mapping(pool, to_dev(w.block_table),
                                  to_dev(np.asarray(pos, np.int64)), slots,
                                  seq_ids=to_dev(np.asarray(seq, np.int32)))
    return slots


def new_token_slots(w: synth.Workload, pool: pkv.PagedKVPool) -> torch.Tensor:
    """The step's new-token slots: the workload's (paged) or the library's
    slot mapping at positions seq_lens - 1 (ring layouts)."""
    if w.new_slots is not None:
        return to_dev(w.new_slots)
    B = len(w.seq_lens)
    return library_slots(w, pool, np.arange(B, dtype=np.int32), w.seq_lens.astype(np.int64) - 1)


def append_all(w: synth.Workload, pool: pkv.PagedKVPool, new: bool = True, chunk: int = 1 << 16):
    """History then (optionally) the step's new tokens, through paged_kv_append
    (ring layouts: at the slots the library's slot mapping gives)."""
    T = len(w.hist_pos)
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        slots = (to_dev(w.hist_slots[s:e]) if w.hist_slots is not None
                 else library_slots(w, pool, w.hist_seq[s:e], w.hist_pos[s:e]))
        pkv.paged_kv_append(to_dev_bits(w.hist_k[s:e]),
                            None if w.hist_v is None else to_dev_bits(w.hist_v[s:e]),
                            slots, pool)
    if new:
        pkv.paged_kv_append(to_dev_bits(w.new_k), None if w.new_v is None else to_dev_bits(w.new_v),
                            new_token_slots(w, pool), pool)


def pool_to_host(pool: pkv.PagedKVPool):
    def h(t):
        if t is None:
            return None
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).cpu().numpy().view(np.uint16)
        return t.cpu().numpy()
    return h(pool.k), h(pool.v), h(pool.k_scale), h(pool.v_scale)


class DeviceStep:
    """Static device buffers of one layer's decode (q, block table, lengths)."""

    def __init__(self, w: synth.Workload):
        self.w = w
        self.q = to_dev_bits(w.q)
        self.block_table = to_dev(w.block_table)
        self.seq_lens = to_dev(w.seq_lens)
        self.max_seq_len = int(w.seq_lens.max()) if len(w.seq_lens) else 0

    def decode(self, pool, split_tokens=pkv.SPLIT_AUTO, out_f32=False, workspace=None):
        s = self.w.spec
        out = torch.empty(self.q.shape, dtype=torch.float32 if out_f32 else torch.bfloat16,
                          device="cuda")
        pkv.paged_decode_attention(self.q, pool, self.block_table, self.seq_lens, s.window,
                                   np.float32(s.softmax_scale), out, self.max_seq_len,
                                   split_tokens=split_tokens, workspace=workspace)
        return out


def out_to_f64(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy().astype(np.float64)


def max_abs_err(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(got - ref))) if got.size else 0.0


def max_row_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max over rows of ||got - ref|| / max(||ref||, 1e-6) (normwise per (b, h) row)."""
    d = np.linalg.norm((got - ref).reshape(-1, got.shape[-1]), axis=1)
    r = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=1)
    return float(np.max(d / np.maximum(r, 1e-6))) if d.size else 0.0
