"""Shared test helpers: build oracle pools from synthetic workloads, parse
golden fixtures.  No attention or quantiser arithmetic lives here."""
from __future__ import annotations

import os
import struct

import numpy as np

import oracle
from paged_kv_decode_03_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def hex_to_f32(h: str) -> np.float32:
    return np.float32(struct.unpack("<f", struct.pack("<I", int(h, 16)))[0])


def oracle_pool(w: synth.Workload, append_new: bool = True) -> oracle.OraclePool:
    """Poisoned pool arrays, then the history and (optionally) the step's
    new tokens appended by the oracle's own append."""
    spec = w.spec
    k, v, ks, vs = synth.empty_pool_arrays(spec, w.layout)
    mode = {"bf16": oracle.SCALE_NONE, "int8_token": oracle.SCALE_PER_TOKEN,
            "int8_head": oracle.SCALE_PER_HEAD}[spec.kv]
    if spec.kv == "int8_head":
        ks = w.k_head_scale.copy()
        vs = None if spec.alias else w.v_head_scale.copy()
    pool = oracle.OraclePool(k=k, v=v, k_scale=ks, v_scale=vs, scale_mode=mode,
                             ring_blocks=spec.ring_blocks)
    hist_slots, new_slots = oracle_slots(w, pool)
    if len(hist_slots):
        oracle.append(w.hist_k, w.hist_v, hist_slots, pool)
    if append_new:
        oracle.append(w.new_k, w.new_v, new_slots, pool)
    return pool


def oracle_slots(w: synth.Workload, pool: oracle.OraclePool):
    """History and new-token slots: the workload's own for paged layouts, the
    oracle's address map for rings (positions seq_lens - 1 for the step)."""
    if w.hist_slots is not None:
        return w.hist_slots, w.new_slots
    B = len(w.seq_lens)
    hist = oracle.slot_mapping(pool, w.block_table, w.hist_seq, w.hist_pos)
    new = oracle.slot_mapping(pool, w.block_table, np.arange(B, dtype=np.int32),
                              w.seq_lens.astype(np.int64) - 1)
    return hist, new


def oracle_decode(w: synth.Workload, pool: oracle.OraclePool, rows=None, num_threads=0):
    s = w.spec
    return oracle.decode(w.q, pool, w.block_table, w.seq_lens, s.num_q_heads, s.window,
                         np.float32(s.softmax_scale), rows=rows, num_threads=num_threads)


def read_quantizer_golden():
    cases = []
    with open(os.path.join(GOLDEN, "int8_quantizer.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, rest = line.split("|")
            mode, scale_hex = head.split()
            xs, qs = rest.split(";")
            cases.append((mode, hex_to_f32(scale_hex),
                          np.array([float(t) for t in xs.split()], np.float32),
                          np.array([int(t) for t in qs.split()], np.int8)))
    return cases


def read_two_key_golden():
    d = {}
    with open(os.path.join(GOLDEN, "two_key_softmax.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            d[key] = np.array([float(t) for t in vals], np.float64)
    return d
