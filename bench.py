#!/usr/bin/env python3
"""Benchmark one decode step of a paged-KV attention layer on GB300.

A step is the whole hot path over one batch: append the batch's new K/V
token (one per sequence) into the paged pool, then decode attention for
every sequence (split-KV partial kernel + log-sum-exp combine when the split
length is > 0, a single pass otherwise).  Default workload: the Gemma4-12B
sliding-window layer (batch 64, lengths uniform in [512, 8192], H_q=16,
H_kv=8, head_dim=256, window 1024, bf16 KV, 16-token blocks, pool 1.25x the
needed blocks, shuffled).  Inputs are seeded synthetic data resident in HBM.

value = algorithmic bytes of the step (KV rows in each window read once, Q,
output, appended rows) / device time per step, in GB/s.
Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_decode_03_gb300 import bytes_model, synth  # noqa: E402

METRIC = "decode-attn achieved HBM GB/s (% of ~8 TB/s) and seq·layer decode steps/sec"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c2", choices=sorted(synth.CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller cases for profiling)")
    ap.add_argument("--split-tokens", type=int, default=None,
                    help="override the split length (0 = single pass, -1 = automatic)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload lines (every config, the six-layer step, "
                         "the oracle at all threads and at one thread)")
    ap.add_argument("--per-config-steps", type=int, default=100)
    ap.add_argument("--record-traffic", metavar="RAW_CSV", default=None,
                    help="write profiles/traffic.json's entry for --config from an ncu capture of "
                         "its decode kernel on --batch sequences (the raw page as CSV: ncu -i "
                         "REPORT --page raw --csv), scaled to the full batch by algorithmic bytes")
    ap.add_argument("--chunk-only", type=int, default=0,
                    help="time only the chunk attention (q_len > 1) with chunks of this many "
                         "tokens on --config's shapes (prints that measurement, not a bench line)")
    ap.add_argument("--rope-only", action="store_true",
                    help="time only RoPE fused with the append on the continuous-batching global "
                         "and sliding layers' new tokens (prints that measurement)")
    return ap.parse_args()


def workload_spec(args):
    spec = synth.CONFIGS[args.config]
    if args.batch:
        spec = synth.shrink(spec, batch=args.batch)
    if args.split_tokens is not None:
        spec = synth.shrink(spec, split_tokens=args.split_tokens)
    return spec


# ------------------------------------------------------------------ helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Sources each decode kernel is compiled from: a recorded DRAM-traffic figure
# stays valid while these files are unchanged.
KERNEL_SOURCES = {
    "cuda_core": ("pkv_decode.cu", "pkv_device.cuh", "pkv_internal.h"),
    "tensor_core": ("pkv_decode_tc.cu", "pkv_device.cuh", "pkv_internal.h"),
}


def csrc_sha(names=None) -> str:
    h = hashlib.sha256()
    base = os.path.join(ROOT, "paged_kv_decode_03_gb300", "csrc")
    for name in sorted(names if names is not None else os.listdir(base)):
        with open(os.path.join(base, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str):
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, if it was taken on the current sources of that kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(config)
        if e and e.get("sources_sha") == csrc_sha(KERNEL_SOURCES[e["kernel_family"]]):
            return e.get("bytes_per_launch")
    except Exception:
        pass
    return None


def layout_bytes(spec) -> int:
    """Algorithmic bytes of one decode of the workload (KV once, q, out),
    from its layout alone (no K/V values are drawn)."""
    layout = synth.make_layout(spec, np.random.default_rng(spec.seed))
    d = bytes_model.decode_bytes(spec, layout.seq_lens, layout.block_table)
    return int(d["kv"] + d["q"] + d["out"])


def record_traffic(args) -> dict:
    """profiles/traffic.json entry of --config: DRAM bytes of the captured
    launch (dram__bytes_read.sum + dram__bytes_write.sum, one launch) times
    full-batch / captured-batch algorithmic bytes, keyed by the kernel's
    source hash."""
    import csv
    with open(args.record_traffic) as f:
        rows = [r for r in csv.reader(f)]
    hdr, vals = rows[0], rows[2]
    col = {h: i for i, h in enumerate(hdr)}
    unit = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}

    def metric(name):
        return float(vals[col[name]].replace(",", "")) * unit[rows[1][col[name]]]

    dram = metric("dram__bytes_read.sum") + metric("dram__bytes_write.sum")
    kernel = vals[col["Kernel Name"]]
    family = "tensor_core" if "decode_tc_kernel" in kernel else "cuda_core"
    full = synth.CONFIGS[args.config]
    cap = workload_spec(args)
    a_cap, a_full = layout_bytes(cap), layout_bytes(full)
    entry = {
        "kernel_family": family,
        "sources_sha": csrc_sha(KERNEL_SOURCES[family]),
        "bytes_per_launch": int(round(dram * a_full / a_cap)),
        "kernel": kernel.split("(")[0].strip(),
        "source": f"ncu capture of one launch on {args.config} with batch {cap.batch} "
                  f"(dram__bytes_read.sum + dram__bytes_write.sum), scaled to batch "
                  f"{full.batch} by the ratio of algorithmic bytes",
        "capture_dram_bytes": int(round(dram)),
        "capture_algorithmic_bytes": a_cap,
    }
    path = getattr(args, "traffic_path", None) or os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        d = {}
    d[args.config] = entry
    with open(path, "w") as f:
        json.dump(d, f, indent=1, sort_keys=True)
        f.write("\n")
    return entry


def workload_desc(spec) -> str:
    lens = spec.lens
    if lens[0] == "uniform":
        ls = f"lens U[{lens[1]},{lens[2]}]"
    elif lens[0] == "const":
        ls = f"lens {lens[1]}"
    elif lens[0] == "lognormal":
        ls = f"lens lognormal(median {lens[1]}, sigma {lens[2]}) clipped [{lens[3]},{lens[4]}]"
    else:
        ls = f"lens {list(lens[1])}"
    kv = {"bf16": "bf16 KV", "int8_token": "int8 KV per-token scales",
          "int8_head": "int8 KV per-head scales"}[spec.kv]
    return (f"{spec.name}: B={spec.batch}, H_q={spec.num_q_heads}, H_kv={spec.num_kv_heads}, "
            f"D={spec.head_dim}, window={spec.window or 'none (global)'}, {kv}"
            f"{', K=V one tensor' if spec.alias else ''}, block {spec.block_size}, {ls}")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during a region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed"
        if not inside:
            inside, window = rows, "whole run (timed region shorter than the sample period)"
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# ------------------------------------------------------------- our arm
def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value of x over all ranks (the job's time is its slowest
    rank's); x itself on one rank."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: float, ms_per_step: float, world: int) -> float:
    """Whole-job throughput: every rank moves bytes_per_rank_step per step
    (weak scaling, one independent batch per GPU) and a step takes the slowest
    rank's ms_per_step."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def _dbits(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _dnum(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def device_pool(spec, w, dev, hist=True):
    """A poisoned device pool for the workload, with its history appended."""
    import torch
    import paged_kv_decode_03_gb300 as pkv
    P, D = spec.block_size, spec.head_dim
    shape = (w.layout.num_blocks, P, spec.num_kv_heads, D)
    if spec.kv == "bf16":
        k_pool = torch.full(shape, int(np.int16(synth.BF16_NAN.view(np.int16))), dtype=torch.int16,
                            device=dev).view(torch.bfloat16)
    else:
        k_pool = torch.full(shape, int(synth.INT8_POISON), dtype=torch.int8, device=dev)
    v_pool = None if spec.alias else k_pool.clone()
    ks = vs = None
    mode = pkv.SCALE_NONE
    if spec.kv == "int8_token":
        mode = pkv.SCALE_PER_TOKEN
        ks = torch.full((w.layout.num_blocks * P,), float("nan"), device=dev)
        vs = None if spec.alias else ks.clone()
    elif spec.kv == "int8_head":
        mode = pkv.SCALE_PER_HEAD
        ks = _dnum(w.k_head_scale, dev)
        vs = None if spec.alias else _dnum(w.v_head_scale, dev)
    pool = pkv.PagedKVPool(k=k_pool, v=v_pool, k_scale=ks, v_scale=vs, scale_mode=mode,
                           ring_blocks=spec.ring_blocks)
    if hist:
        T = len(w.hist_pos)
        bt = _dnum(w.block_table, dev)
        for s in range(0, T, 1 << 16):
            e = min(T, s + (1 << 16))
            if w.hist_slots is not None:
                slots = _dnum(w.hist_slots[s:e], dev)
            else:  # ring layout: the library's own address map
                slots = torch.empty(e - s, dtype=torch.int64, device=dev)
                pkv.paged_kv_slot_mapping(pool, bt, _dnum(w.hist_pos[s:e], dev), slots,
                                          seq_ids=_dnum(w.hist_seq[s:e], dev))
            pkv.paged_kv_append(_dbits(w.hist_k[s:e], dev),
                                None if w.hist_v is None else _dbits(w.hist_v[s:e], dev),
                                slots, pool)
    return pool


def config_dict(spec, w, st, ns, split_api, world):
    """The workload as both arms describe it (the reference arm's line
    carries the same dict, so the two lines can be compared key by key)."""
    dbytes_kv = bytes_model.decode_bytes(spec, w.seq_lens, w.block_table)["kv"]
    return {
        "workload": workload_desc(spec),
        "batch": int(spec.batch), "num_q_heads": spec.num_q_heads,
        "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim, "window": spec.window,
        "block_size": spec.block_size, "num_blocks": int(w.layout.num_blocks),
        "kv": spec.kv, "k_equals_v": bool(spec.alias),
        "split_tokens": int(st), "num_splits": int(ns),
        "step": ("append 1 token/seq + decode (split partial + combine)" if split_api
                 else "append 1 token/seq + paged_decode_attention"),
        "l2": f"inputs larger than L2 ({dbytes_kv / 1e6:.0f} MB of KV read per step vs 129 MB L2); no flush",
        "parallelism": "one batch" if world == 1 else f"replicas: one independent batch per GPU x{world}",
    }


class LayerRun:
    """Device buffers of one layer's decode step and its captured graphs:
    append, decode (one paged_decode_attention call, or the split partial
    call when ``split_api``) and, for the split path, the combine."""

    def __init__(self, spec, w, dev, req_split, split_api_allowed=True):
        import torch
        import paged_kv_decode_03_gb300 as pkv
        self.spec, self.w = spec, w
        B, Hq, D = w.q.shape
        self.pool = device_pool(spec, w, dev)
        self.q = _dbits(w.q, dev)
        self.bt = _dnum(w.block_table, dev)
        self.sl = _dnum(w.seq_lens, dev)
        self.k_new = _dbits(w.new_k, dev)
        self.v_new = None if w.new_v is None else _dbits(w.new_v, dev)
        # ring layouts: the step maps each new token's position (seq_lens - 1)
        # to its ring slot on the device before appending it
        self.ring = spec.ring_blocks > 0
        self.positions = _dnum(w.seq_lens.astype(np.int64) - 1, dev) if self.ring else None
        self.slots = (torch.empty(B, dtype=torch.int64, device=dev) if self.ring
                      else _dnum(w.new_slots, dev))
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
        self.max_len = int(w.seq_lens.max())
        self.scale = float(np.float32(spec.softmax_scale))
        # a workload that names its split length (or --split-tokens) runs the
        # two split-KV calls; otherwise one paged_decode_attention call
        self.split_api = split_api_allowed and req_split != pkv.SPLIT_AUTO and req_split > 0
        self.st = pkv.paged_decode_split_tokens(B, Hq, spec.num_kv_heads, self.max_len,
                                                spec.window, req_split)
        self.ns = pkv.paged_decode_num_splits(self.max_len, spec.window, self.st) if self.st > 0 else 1
        self.split_api = self.split_api and self.st > 0
        ws_bytes = pkv.paged_decode_workspace_bytes(B, Hq, spec.num_kv_heads, D, self.max_len,
                                                    spec.window, self.st)
        self.ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.pws = torch.empty(max(pkv.paged_decode_partial_workspace_bytes(B, Hq, spec.num_kv_heads, D),
                                   256), dtype=torch.uint8, device=dev)
        self.lse = torch.empty((B, self.ns, Hq), dtype=torch.float32, device=dev)
        self.po = torch.empty((B, self.ns, Hq, D), dtype=torch.float32, device=dev)
        self.tc = pkv.uses_tensor_cores(self.pool, Hq)
        dbytes = bytes_model.decode_bytes(spec, w.seq_lens, w.block_table)
        self.dbytes = dbytes
        self.abytes = bytes_model.append_bytes(spec, int((w.seq_lens > 0).sum()))
        self.step_bytes = dbytes["kv"] + dbytes["q"] + dbytes["out"] + self.abytes
        self.decode_kernel_bytes = dbytes["kv"] + dbytes["q"] + (dbytes["out"] if not self.split_api else 0)
        self.graphs = None

    def append(self):
        import paged_kv_decode_03_gb300 as pkv
        if self.ring:
            pkv.paged_kv_slot_mapping(self.pool, self.bt, self.positions, self.slots)
        pkv.paged_kv_append(self.k_new, self.v_new, self.slots, self.pool)

    def decode(self):
        import paged_kv_decode_03_gb300 as pkv
        s = self.spec
        if self.split_api:
            pkv.paged_decode_split_partial(self.q, self.pool, self.bt, self.sl, s.window, self.scale,
                                           self.st, self.lse, self.po, self.out, self.max_len,
                                           workspace=self.pws)
        else:
            pkv.paged_decode_attention(self.q, self.pool, self.bt, self.sl, s.window, self.scale,
                                       self.out, self.max_len, split_tokens=self.st,
                                       workspace=self.ws)

    def combine(self):
        import paged_kv_decode_03_gb300 as pkv
        pkv.paged_decode_lse_combine(self.lse, self.po, self.sl, self.spec.window, self.st, self.out)

    def step(self):
        self.append()
        self.decode()
        if self.split_api:
            self.combine()

    def launches_per_step(self):
        import paged_kv_decode_03_gb300 as pkv
        n = 0
        if self.ring:
            pkv.paged_kv_slot_mapping(self.pool, self.bt, self.positions, self.slots)
            n += pkv.last_launch_count()
            pkv.paged_kv_append(self.k_new, self.v_new, self.slots, self.pool)
            n += pkv.last_launch_count()
        else:
            self.append()
            n += pkv.last_launch_count()
        for part in ([self.decode] + ([self.combine] if self.split_api else [])):
            part()
            n += pkv.last_launch_count()
        return n

    def capture(self):
        """The whole step as one CUDA graph (what the step time is taken on,
        as an engine replays a captured step), and its parts as graphs of
        their own, replayed with events between them for the per-part device
        times; replays measure the GPU and not the Python loop."""
        import torch
        parts = [None, None, None]
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            for i, fn in enumerate([self.append, self.decode] + ([self.combine] if self.split_api else [])):
                parts[i] = torch.cuda.CUDAGraph()
                with torch.cuda.graph(parts[i], stream=cap):
                    fn()
            self.step_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.step_graph, stream=cap):
                self.step()
        torch.cuda.current_stream().wait_stream(cap)
        torch.cuda.synchronize()
        self.graphs = parts

    def part_times(self, steps):
        """Per-part device times (us): append, decode, combine -- each part's
        graph replayed back to back between two events (every replay redoes
        the same work: the same tokens into the same slots, the same
        outputs)."""
        import torch
        times = []
        for g in self.graphs:
            if g is None:
                times.append(0.0)
                continue
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            start.record()
            for _ in range(steps):
                g.replay()
            end.record()
            torch.cuda.synchronize()
            times.append(start.elapsed_time(end) / steps * 1e3)
        app, dec, cmb = times
        return app, dec, (cmb if self.split_api else 0.0)


def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_decode_03_gb300 as pkv

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pkv.load_library()
    spec = workload_spec(args)
    w = synth.make_workload(spec)
    B, Hq, D = w.q.shape
    P = spec.block_size
    req = args.split_tokens if args.split_tokens is not None else (spec.split_tokens
                                                                    or pkv.SPLIT_AUTO)
    run = LayerRun(spec, w, dev, req)
    pool, q, bt, sl = run.pool, run.q, run.bt, run.sl
    k_new, v_new, slots, out = run.k_new, run.v_new, run.slots, run.out
    max_len, scale, split_api, st, ns = run.max_len, run.scale, run.split_api, run.st, run.ns
    ws, pws, lse, po, tc = run.ws, run.pws, run.lse, run.po, run.tc
    torch.cuda.synchronize()
    pkv.device_status(clear=True)
    dbytes, abytes, step_bytes = run.dbytes, run.abytes, run.step_bytes
    decode_kernel_bytes = run.decode_kernel_bytes
    launches_per_step = run.launches_per_step()
    for _ in range(max(3, args.warmup)):
        run.step()
    torch.cuda.synchronize()
    run.capture()

    for _ in range(3):
        run.step_graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record()
    for i in range(args.steps):
        run.step_graph.replay()
    end.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop(t0, t1) if sampler else None
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    status = pkv.device_status(clear=True)
    # per-kernel times for the roofline: the parts' graphs with events between
    app_us, dec_us, cmb_us = run.part_times(args.steps)
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_gbs(step_bytes, ms_per_step, world)

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        # the step's host inputs travel in one pinned buffer and one copy
        # (each at a 256-byte offset); the calls take device views of it
        parts = [("q", w.q.view(np.uint8)), ("k", w.new_k.view(np.uint8)),
                 ("v", None if w.new_v is None else w.new_v.view(np.uint8)),
                 ("slots", w.new_slots.view(np.uint8)), ("bt", w.block_table.view(np.uint8)),
                 ("sl", w.seq_lens.view(np.uint8))]
        offs, total = {}, 0
        for name, a in parts:
            if a is not None:
                offs[name] = total
                total += (a.nbytes + 255) // 256 * 256
        stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
        for name, a in parts:
            if a is not None:
                stage_h[offs[name]:offs[name] + a.nbytes].copy_(torch.from_numpy(np.ascontiguousarray(a).reshape(-1)))
        stage_d = torch.empty(total, dtype=torch.uint8, device=dev)

        def view(name, dtype, shape):
            n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            return stage_d[offs[name]:offs[name] + n].view(dtype).view(*shape)

        q_e = view("q", torch.bfloat16, w.q.shape)
        k_e = view("k", torch.bfloat16, w.new_k.shape)
        v_e = None if w.new_v is None else view("v", torch.bfloat16, w.new_v.shape)
        slots_e = view("slots", torch.int64, w.new_slots.shape)
        bt_e = view("bt", torch.int32, w.block_table.shape)
        sl_e = view("sl", torch.int32, w.seq_lens.shape)
        out_h = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
        h2d = sum(a.nbytes for _, a in parts if a is not None)
        d2h = out_h.numel() * out_h.element_size()

        def e2e_step():
            stage_d.copy_(stage_h, non_blocking=True)
            pkv.paged_kv_append(k_e, v_e, slots_e, pool)
            if split_api:  # the same calls as the device-timed step
                pkv.paged_decode_split_partial(q_e, pool, bt_e, sl_e, spec.window, scale, st, lse,
                                               po, out, max_len, workspace=pws)
                pkv.paged_decode_lse_combine(lse, po, sl_e, spec.window, st, out)
            else:
                pkv.paged_decode_attention(q_e, pool, bt_e, sl_e, spec.window, scale, out, max_len,
                                           split_tokens=st, workspace=ws)
            out_h.copy_(out, non_blocking=True)

        for _ in range(max(3, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        s2 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        s2.record()
        for _ in range(args.steps):
            e2e_step()
        e2.record()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s2.elapsed_time(e2), world, dev)
        e2e = {"value": whole_job_gbs(step_bytes, e2e_ms / args.steps, world), "unit": "GB/s",
               "ms_per_step": e2e_ms / args.steps, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h),
               "api": ("paged_kv_append + paged_decode_split_partial + paged_decode_lse_combine"
                       if split_api else "paged_kv_append + paged_decode_attention")
                      + " (C ABI), the step's inputs in one pinned host buffer and one copy"}

    if rank != 0:
        return None
    peak, peak_kind = peaks()
    achieved = decode_kernel_bytes / (dec_us * 1e-6) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(spec, w, step_bytes, args.cpu_seconds)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if spec.kv == "bf16" else "int8 KV / bf16 q",
        "data": "synthetic (seeded N(0,1) bf16 K/V/q; shuffled physical blocks)",
        "config": config_dict(spec, w, st, ns, split_api, world),
        "method": {
            "timing": ("one CUDA graph per step (append + decode), CUDA events around the "
                       "timed replays; per-kernel times from each part's graph replayed back "
                       "to back between two events"),
            "decode_kernel": ("tensor cores (tcgen05), persistent stream-K" if tc
                              else "CUDA cores"),
        },
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_peak": round(100 * value / world / peak, 2),
        "seq_layer_steps_per_s": round(world * B / (ms_per_step * 1e-3), 1),
        "bytes_per_step": {"kv": dbytes["kv"], "q": dbytes["q"], "out": dbytes["out"],
                           "append": abytes, "total": step_bytes},
        "kernels_us": {"append": round(app_us, 3), "decode": round(dec_us, 3),
                       "combine": round(cmb_us, 3)},
        "roofline": {"bound": "hbm",
                     "kernel": ("decode_tc_kernel (+ plan)" if tc else "decode_kernel")
                     + (" split partial" if split_api else ""),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": decode_kernel_bytes,
                     "traffic": recorded_traffic(args.config + ("_split_calls" if split_api
                                                                else ""))},
        "gpu_launches": launches_per_step * args.steps,
        "device_error_word": status,
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in e2e.items()}
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if (world == 1 and not args.no_per_config and args.config == "c2" and not args.batch
            and args.split_tokens is None):
        main = {"workload": workload_desc(spec), "call": "paged_decode_attention",
                "decode_kernel": line["method"]["decode_kernel"],
                "kernels_us": line["kernels_us"], "ms_per_step": line["ms_per_step"],
                "algorithmic_bytes_per_launch": decode_kernel_bytes,
                "achieved_gbs": round(achieved, 1), "frac_of_measured": round(achieved / peak, 4),
                "pct_of_8tbs": round(100 * achieved / NOMINAL_HBM_GBS, 2),
                "traffic": recorded_traffic("c2"),
                "seq_layer_steps_per_s": round(B / (ms_per_step * 1e-3), 1),
                "device_error_word": status}
        del run, pool, q, bt, sl, k_new, v_new, slots, out, ws, pws, lse, po
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["per_config"] = per_config(args, dev, main, spec, w)
    return line


# ------------------------------------------------------- every workload
def oracle_full_run(spec, w, layers=None):
    """One full step of the oracle (append every sequence's new token, decode
    every row) with all host threads and with one thread, in seconds.  For a
    multi-layer step, ``layers`` are the per-layer workloads (layers sharing
    history values share one oracle pool: the timing does not depend on the
    appended token's values)."""
    import oracle
    layers = layers or [w]
    pools = {}
    for lw in layers:
        if id(lw.hist_k) not in pools:
            pools[id(lw.hist_k)] = oracle_setup(lw.spec, lw)
    threads = oracle.max_threads()
    times = {}
    for label, nt in (("all_threads_s", 0), ("one_thread_s", 1)):
        t = 0.0
        for lw in layers:
            pool = pools[id(lw.hist_k)]
            s = lw.spec
            t0 = time.perf_counter()
            oracle.append(lw.new_k, lw.new_v, oracle_new_slots(lw, pool), pool)
            oracle.decode(lw.q, pool, lw.block_table, lw.seq_lens, s.num_q_heads, s.window,
                          np.float32(s.softmax_scale), num_threads=nt)
            t += time.perf_counter() - t0
        times[label] = round(t, 4)
    return {"kind": "oracle", "threads": threads, **times,
            "sample": f"one full step: {len(layers)} layer(s) x (append {w.spec.batch} tokens + "
                      f"decode {w.spec.batch}x{w.spec.num_q_heads} rows), fp64 C oracle"}


def measure_layer(spec, w, dev, req, steps, warmup, split_api_allowed=True):
    """Decode-kernel timing of one workload as the main line takes it."""
    import torch
    import paged_kv_decode_03_gb300 as pkv
    run = LayerRun(spec, w, dev, req, split_api_allowed)
    launches = run.launches_per_step()
    for _ in range(max(3, warmup)):
        run.step()
    torch.cuda.synchronize()
    run.capture()
    for _ in range(3):
        run.step_graph.replay()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for i in range(steps):
        run.step_graph.replay()
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    app, dec, cmb = run.part_times(steps)
    peak, _ = peaks()
    achieved = run.decode_kernel_bytes / (dec * 1e-6) / 1e9
    B = spec.batch
    entry = {
        "workload": workload_desc(spec),
        "call": ("paged_decode_split_partial + paged_decode_lse_combine" if run.split_api
                 else "paged_decode_attention") + (f", split_tokens {run.st}" if run.st else ""),
        "decode_kernel": ("tensor cores (tcgen05), persistent stream-K" if run.tc else "CUDA cores"),
        "kernels_us": {"append": round(app, 3), "decode": round(dec, 3),
                       "combine": round(cmb if run.split_api else 0.0, 3)},
        "ms_per_step": round(ms, 6),
        "algorithmic_bytes_per_launch": run.decode_kernel_bytes,
        "achieved_gbs": round(achieved, 1), "frac_of_measured": round(achieved / peak, 4),
        "pct_of_8tbs": round(100 * achieved / NOMINAL_HBM_GBS, 2),
        "step_gbs": round(run.step_bytes / (ms * 1e-3) / 1e9, 1),
        "seq_layer_steps_per_s": round(B / (ms * 1e-3), 1),
        "gpu_launches_per_step": launches,
        "device_error_word": pkv.device_status(clear=True),
    }
    del run
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def rope_theta(spec):
    """(base, theta) of a layer's RoPE in the benchmark: every pair with base
    10^4 on sliding layers, p-RoPE on the first quarter of the pairs with
    base 10^6 on global layers; theta_i = base^(-2i/D) (RoFormer)."""
    D = spec.head_dim
    base, pairs = (1e4, D // 2) if spec.window else (1e6, D // 8)
    return base, (base ** (-2.0 * np.arange(D // 2) / D))[:pairs].astype(np.float64)


def measure_step(dev, steps, warmup, rope=False):
    """The six-layer continuous-batching step (five int8 per-head sliding
    layers, one bf16 global layer, one ragged layout with shared prefix
    blocks): one paged_decode_step call captured as one CUDA graph and
    replayed; events around each replay.  With ``rope`` every layer's append
    is RoPE fused with the append (q rotated into its own buffer)."""
    import torch
    import paged_kv_decode_03_gb300 as pkv
    layers = synth.make_step(share_history=True)
    w0 = layers[0]
    pools, base = [], {}
    for lw in layers:
        key = id(lw.hist_k)
        if key not in base:
            base[key] = device_pool(lw.spec, lw, dev)
            pools.append(base[key])
        else:
            b = base[key]
            pools.append(pkv.PagedKVPool(k=b.k.clone(), v=None if b.v is None else b.v.clone(),
                                         k_scale=b.k_scale, v_scale=b.v_scale,
                                         scale_mode=b.scale_mode))
    del base
    slots, bt, sl = _dnum(w0.new_slots, dev), _dnum(w0.block_table, dev), _dnum(w0.seq_lens, dev)
    max_len = int(w0.seq_lens.max())
    extra, rope_bytes = [{} for _ in layers], 0
    if rope:
        for i, lw in enumerate(layers):
            _, theta = rope_theta(lw.spec)
            table = pkv.paged_rope_cos_sin_table(_dnum(theta, dev), max_len)
            extra[i] = dict(rope_table=table, q_rotated=torch.empty(lw.q.shape, dtype=torch.bfloat16,
                                                                   device=dev))
            rope_bytes += 2 * lw.q.size * 2 + len(lw.seq_lens) * len(theta) * 8
    dl = [pkv.DecodeLayer(pool=gp, q=_dbits(lw.q, dev), k_new=_dbits(lw.new_k, dev),
                          v_new=None if lw.new_v is None else _dbits(lw.new_v, dev),
                          out=torch.empty(lw.q.shape, dtype=torch.bfloat16, device=dev),
                          window=lw.spec.window, softmax_scale=float(np.float32(lw.spec.softmax_scale)),
                          **extra[i])
          for i, (lw, gp) in enumerate(zip(layers, pools))]
    ws = torch.empty(max(256, pkv.paged_decode_step_workspace_bytes(dl, max_len)),
                     dtype=torch.uint8, device=dev)

    def call():
        pkv.paged_decode_step(dl, slots, bt, sl, max_len, workspace=ws)

    call()
    launches = pkv.last_launch_count()
    for _ in range(max(3, warmup)):
        call()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            call()
    torch.cuda.current_stream().wait_stream(cap)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record()
    for i in range(steps):
        graph.replay()
        evs[i + 1].record()
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    ms = evs[0].elapsed_time(evs[-1]) / steps
    step_bytes = 0
    for lw in layers:
        d = bytes_model.decode_bytes(lw.spec, lw.seq_lens, lw.block_table)
        step_bytes += d["kv"] + d["q"] + d["out"]
        step_bytes += bytes_model.append_bytes(lw.spec, int((lw.new_slots >= 0).sum()))
    step_bytes += rope_bytes  # rotated q written and read again, table rows
    peak, _ = peaks()
    gbs = step_bytes / (ms * 1e-3) / 1e9
    B = w0.spec.batch
    entry = {
        "workload": (f"c5 continuous-batching step: {len(layers)} layers "
                     f"({''.join(synth.C5_LAYERS)}) over one layout; sliding: "
                     f"{workload_desc(layers[0].spec)}; global: {workload_desc(layers[-1].spec)}; "
                     "history values shared by the sliding layers, each its own pool"),
        "call": ("paged_decode_step (every layer's RoPE + append, then decode), one CUDA graph; "
                 "RoPE: every pair, theta base 1e4, on sliding layers; the first quarter of the "
                 "pairs, base 1e6, on the global layer" if rope else
                 "paged_decode_step (every layer's append + decode), one CUDA graph"),
        "ms_per_step": round(ms, 6), "ms_per_step_median": round(statistics.median(per), 6),
        "bytes_per_step": int(step_bytes),
        "step_gbs": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4),
        "pct_of_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
        "seq_layer_steps_per_s": round(B * len(layers) / (ms * 1e-3), 1),
        "gpu_launches_per_step": launches,
        "device_error_word": pkv.device_status(clear=True),
    }
    del dl, pools, ws, graph, extra
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry, layers


def measure_prefill(spec, q_len, dev, steps, warmup, with_oracle):
    """Chunk attention (q_len > 1): every sequence's last ``q_len`` tokens
    attend their cache (chunked prefill), one paged_prefill_attention call
    captured in a CUDA graph; events around each replay."""
    import torch
    import paged_kv_decode_03_gb300 as pkv
    w = synth.make_chunk_workload(spec, q_len)
    B, G = spec.batch, spec.group
    pool = device_pool(spec, synth.Workload(spec, w.layout, w.q, w.hist_k, w.hist_v, w.hist_slots,
                                            w.new_k, w.new_v, w.new_slots, None, None,
                                            None, None), dev, hist=False)
    for k_, v_, sl_ in ((w.hist_k, w.hist_v, w.hist_slots), (w.new_k, w.new_v, w.new_slots)):
        for s0 in range(0, len(sl_), 1 << 16):
            e0 = min(len(sl_), s0 + (1 << 16))
            pkv.paged_kv_append(_dbits(k_[s0:e0], dev), None if v_ is None else _dbits(v_[s0:e0], dev),
                                _dnum(sl_[s0:e0], dev), pool)
    q = _dbits(w.q, dev)
    qs, bt, sl = _dnum(w.q_start, dev), _dnum(w.block_table, dev), _dnum(w.seq_lens, dev)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    max_len, max_q = int(w.seq_lens.max()), int(np.diff(w.q_start).max())
    scale = float(np.float32(spec.softmax_scale))

    def call():
        pkv.paged_prefill_attention(q, qs, pool, bt, sl, spec.window, scale, out, max_len, max_q)

    call()
    launches = pkv.last_launch_count()
    for _ in range(max(3, warmup)):
        call()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            call()
    torch.cuda.current_stream().wait_stream(cap)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record()
    for i in range(steps):
        graph.replay()
        evs[i + 1].record()
    torch.cuda.synchronize()
    us = evs[0].elapsed_time(evs[-1]) / steps * 1e3
    # algorithmic work: every (query, head) row against the keys its mask
    # allows, two contractions of head_dim each; bytes: the unique KV rows
    # the chunks read, Q and the output
    n = np.diff(w.q_start).astype(np.int64)
    lens = w.seq_lens.astype(np.int64)
    keys = 0
    for b in range(B):
        pos = lens[b] - n[b] + np.arange(n[b])
        lo = np.maximum(0, pos - spec.window) if spec.window else np.zeros_like(pos)
        keys += int((pos - lo + 1).sum())
    flops = 4 * keys * spec.num_q_heads * spec.head_dim
    kv = 0
    for b in range(B):
        first = lens[b] - n[b]
        lo = max(0, first - spec.window) if spec.window else 0
        kv += int(lens[b] - lo)
    kv_bytes = kv * bytes_model.bytes_per_key(spec.num_kv_heads, spec.head_dim, spec.kv, spec.alias)
    qo_bytes = 2 * int(n.sum()) * spec.num_q_heads * spec.head_dim * 2
    peaks_d = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks_d = json.load(f)
    except Exception:
        pass
    tf_peak = float(peaks_d.get("bf16_tflops", 1900.0))
    hbm_peak, _ = peaks()
    tflops = flops / (us * 1e-6) / 1e12
    gbs = (kv_bytes + qo_bytes) / (us * 1e-6) / 1e9
    entry = {
        "workload": f"{workload_desc(spec)}; chunks of {q_len} tokens per sequence (chunked prefill)",
        "call": "paged_prefill_attention, one CUDA graph",
        "decode_kernel": "tensor cores (tcgen05): S = Q K^T, O += P V in TMEM, 128 query rows per CTA",
        "kernel_us": round(us, 3),
        "query_tokens_per_s": round(int(n.sum()) / (us * 1e-6), 1),
        "algorithmic_tflop": round(flops / 1e12, 4),
        "achieved_tflops": round(tflops, 2), "bf16_peak_tflops": tf_peak,
        "frac_of_bf16_peak": round(tflops / tf_peak, 4),
        "hbm_gbs": round(gbs, 1), "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
        "gpu_launches_per_step": launches,
        "device_error_word": pkv.device_status(clear=True),
    }
    if with_oracle:
        import oracle
        sub = synth.make_chunk_workload(synth.shrink(spec, batch=4), q_len)
        k_, v_, _, _ = synth.empty_pool_arrays(sub.spec, sub.layout)
        opool = oracle.OraclePool(k=k_, v=v_)
        oracle.append(sub.hist_k, sub.hist_v, sub.hist_slots, opool)
        oracle.append(sub.new_k, sub.new_v, sub.new_slots, opool)
        t0 = time.perf_counter()
        oracle.prefill(sub.q, opool, sub.block_table, sub.seq_lens, sub.q_start, spec.num_q_heads,
                       spec.window, np.float32(spec.softmax_scale))
        t = time.perf_counter() - t0
        entry["oracle"] = {"kind": "oracle", "threads": oracle.max_threads(),
                           "all_threads_s": round(t, 4),
                           "query_tokens_per_s": round(int(sub.q_start[-1]) / t, 1),
                           "sample": f"4 of {B} sequences, chunks of {q_len}, fp64 C oracle"}
    del pool, q, out, graph
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def measure_rope_append(spec, base, pairs, dev, steps, warmup, with_oracle):
    """RoPE fused with the append for one decode step's new tokens (one per
    sequence, at position seq_len - 1): paged_kv_append_rope in a CUDA graph,
    beside the plain paged_kv_append of the same tokens.  theta_i =
    base^(-2i/D) for the first ``pairs`` pairs (p-RoPE keeps the highest
    frequencies), halves pairing."""
    import torch
    import paged_kv_decode_03_gb300 as pkv
    w = synth.make_workload(spec)
    B, D = spec.batch, spec.head_dim
    pool = device_pool(spec, w, dev, hist=False)
    npos = int(w.seq_lens.max())
    theta = (base ** (-2.0 * np.arange(D // 2) / D))[:pairs].astype(np.float64)  # RoFormer
    table = pkv.paged_rope_cos_sin_table(_dnum(theta, dev), npos)
    q = _dbits(w.q, dev)
    q_out = torch.empty_like(q)
    k = _dbits(w.new_k, dev)
    v = None if w.new_v is None else _dbits(w.new_v, dev)
    pos = _dnum(w.seq_lens.astype(np.int64) - 1, dev)
    slots = _dnum(w.new_slots, dev)
    calls = {
        "fused": lambda: pkv.paged_kv_append_rope(q, q_out, k, v, pos, slots, pool, table),
        "append_only": lambda: pkv.paged_kv_append(k, v, slots, pool),
    }
    us = {}
    for name, call in calls.items():
        for _ in range(max(3, warmup)):
            call()
        torch.cuda.synchronize()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                call()
        torch.cuda.current_stream().wait_stream(cap)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        evs[0].record()
        for i in range(steps):
            graph.replay()
            evs[i + 1].record()
        torch.cuda.synchronize()
        us[name] = evs[0].elapsed_time(evs[-1]) / steps * 1e3
        del graph
    # bytes: q in and out, the new k (and v) rows in, the pool rows out (bf16
    # or int8 codes), one table row per token, positions and slots
    row = spec.num_kv_heads * D
    kv_in = B * row * 2 * (1 if spec.alias else 2)
    elem = 2 if spec.kv == "bf16" else 1
    kv_out = B * row * elem * (1 if spec.alias else 2)
    moved = 2 * B * spec.num_q_heads * D * 2 + kv_in + kv_out + B * pairs * 8 + B * 16
    hbm_peak, _ = peaks()
    entry = {
        "workload": f"{workload_desc(spec)}; one new token per sequence at position seq_len - 1, "
                    f"RoPE theta = {base:g}^(-2i/{D}) on the first {pairs} of {D // 2} pairs",
        "call": "paged_kv_append_rope, one CUDA graph (beside paged_kv_append of the same tokens)",
        "kernel_us": round(us["fused"], 3),
        "append_only_us": round(us["append_only"], 3),
        "bytes_moved": moved,
        "hbm_gbs": round(moved / (us["fused"] * 1e-6) / 1e9, 1),
        "frac_of_measured_hbm": round(moved / (us["fused"] * 1e-6) / 1e9 / hbm_peak, 4),
        "device_error_word": pkv.device_status(clear=True),
    }
    if with_oracle:
        import oracle
        k_, v_, ks_, vs_ = synth.empty_pool_arrays(spec, w.layout)
        mode = {"bf16": oracle.SCALE_NONE, "int8_token": oracle.SCALE_PER_TOKEN,
                "int8_head": oracle.SCALE_PER_HEAD}[spec.kv]
        if spec.kv == "int8_head":
            ks_, vs_ = w.k_head_scale.copy(), None if spec.alias else w.v_head_scale.copy()
        opool = oracle.OraclePool(k=k_, v=v_, k_scale=ks_, v_scale=vs_, scale_mode=mode)
        otable, _ = oracle.rope_table(theta, npos)
        t0 = time.perf_counter()
        oracle.append_rope(w.q, w.new_k, w.new_v, w.seq_lens.astype(np.int64) - 1, w.new_slots,
                           opool, otable)
        t = time.perf_counter() - t0
        entry["oracle"] = {"kind": "oracle", "threads": 1, "all_threads_s": round(t, 5),
                           "sample": f"the whole step ({B} tokens), fp32-rounded C oracle "
                                     "(table built outside the timing)"}
    del pool, table, q, q_out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def per_config(args, dev, main_entry, main_spec, main_w):
    """Every workload at its full size: the decode kernel's time and roofline
    fraction (CUDA events over CUDA-graph replays), the six-layer step, and
    one full run of the oracle per workload at all host threads and at one
    thread."""
    import paged_kv_decode_03_gb300 as pkv
    out = {}
    steps, warm = args.per_config_steps, 5
    cpu = not args.no_cpu_baseline
    out["c2"] = main_entry
    if cpu:
        out["c2"]["oracle"] = oracle_full_run(main_spec, main_w)
    for name in ("c1", "c3", "c4", "c5s", "c5g", "c2r", "c5sr"):
        spec = synth.CONFIGS[name]
        w = synth.make_workload(spec)
        req = spec.split_tokens or pkv.SPLIT_AUTO
        # the library's decode call (paged_decode_attention) with the
        # workload's split length
        out[name] = measure_layer(spec, w, dev, req, steps, warm, split_api_allowed=False)
        out[name]["traffic"] = recorded_traffic(name)
        if spec.split_tokens:
            # and the two split-KV calls with that split length
            out[name + "_split_calls"] = measure_layer(spec, w, dev, req, steps, warm)
            out[name + "_split_calls"]["traffic"] = recorded_traffic(name + "_split_calls")
        if cpu:
            out[name]["oracle"] = oracle_full_run(spec, w)
        del w
    entry, layers = measure_step(dev, max(20, steps // 2), warm)
    out["c5"] = entry
    if cpu:
        out["c5"]["oracle"] = oracle_full_run(layers[0].spec, layers[0], layers)
    del layers
    out["c5_rope"], _ = measure_step(dev, max(20, steps // 2), warm, rope=True)
    out["c2_chunk128"] = measure_prefill(synth.C2, 128, dev, steps, warm, cpu)
    # RoPE fused with the append: the global layer with p-RoPE on a quarter
    # of the pairs, the int8 sliding layer with every pair turning
    out["c5g_rope_append"] = measure_rope_append(synth.C5_GLOBAL, 1e6, synth.C5_GLOBAL.head_dim // 8,
                                                 dev, steps, warm, cpu)
    out["c5s_rope_append"] = measure_rope_append(synth.C5_SLIDING, 1e4,
                                                 synth.C5_SLIDING.head_dim // 2, dev, steps, warm,
                                                 cpu)
    return out


# --------------------------------------------------------- CPU baseline
def oracle_setup(spec, w):
    import oracle
    k, v, ks, vs = synth.empty_pool_arrays(spec, w.layout)
    mode = {"bf16": oracle.SCALE_NONE, "int8_token": oracle.SCALE_PER_TOKEN,
            "int8_head": oracle.SCALE_PER_HEAD}[spec.kv]
    if spec.kv == "int8_head":
        ks = w.k_head_scale.copy()
        vs = None if spec.alias else w.v_head_scale.copy()
    pool = oracle.OraclePool(k=k, v=v, k_scale=ks, v_scale=vs, scale_mode=mode,
                             ring_blocks=spec.ring_blocks)
    hist = (w.hist_slots if w.hist_slots is not None
            else oracle.slot_mapping(pool, w.block_table, w.hist_seq, w.hist_pos))
    if len(hist):
        oracle.append(w.hist_k, w.hist_v, hist, pool)
    return pool


def oracle_new_slots(w, pool):
    """The step's new-token slots (the oracle's own address map for rings)."""
    import oracle
    if w.new_slots is not None:
        return w.new_slots
    B = len(w.seq_lens)
    return oracle.slot_mapping(pool, w.block_table, np.arange(B, dtype=np.int32),
                               w.seq_lens.astype(np.int64) - 1)


def cpu_baseline(spec, w, step_bytes, budget_s):
    """The oracle as it stands, on the host cores, over repetitions of the
    full step (append the new tokens + decode every row) for about
    ``budget_s`` seconds."""
    import oracle
    pool = oracle_setup(spec, w)
    threads = oracle.max_threads()
    reps, t = 0, 0.0
    while reps == 0 or t < budget_s:
        t0 = time.perf_counter()
        oracle.append(w.new_k, w.new_v, oracle_new_slots(w, pool), pool)
        oracle.decode(w.q, pool, w.block_table, w.seq_lens, spec.num_q_heads, spec.window,
                      np.float32(spec.softmax_scale))
        t += time.perf_counter() - t0
        reps += 1
    return {"value": round(step_bytes * reps / t / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "seconds": round(t, 2),
            "sample": f"{reps} full step(s) of {spec.name} (append {spec.batch} tokens + "
                      f"decode {spec.batch}x{spec.num_q_heads} rows), fp64 C oracle, "
                      f"{threads} OpenMP threads"}


def reference_config(spec, w):
    """The config dict of our arm's line for the same workload (split length
    and split count resolved by the library's host-side sizing calls)."""
    import paged_kv_decode_03_gb300 as pkv
    B, Hq = w.q.shape[:2]
    max_len = int(w.seq_lens.max())
    req = spec.split_tokens or pkv.SPLIT_AUTO
    st = pkv.paged_decode_split_tokens(B, Hq, spec.num_kv_heads, max_len, spec.window, req)
    ns = pkv.paged_decode_num_splits(max_len, spec.window, st) if st > 0 else 1
    split_api = req != pkv.SPLIT_AUTO and req > 0 and st > 0
    return config_dict(spec, w, st, ns, split_api, 1)


def run_reference(args, rank):
    """The oracle timed as the reference arm: each step a bounded sample of
    the workload (whole sequences, all heads), sized so that warmup + steps
    take about two minutes."""
    if rank != 0:
        return None
    import oracle
    spec = workload_spec(args)
    w = synth.make_workload(spec)
    pool = oracle_setup(spec, w)
    threads = oracle.max_threads()
    B, Hq, _ = w.q.shape
    order = np.argsort(-w.seq_lens)  # deterministic sample: longest first

    def sample_step(nseq):
        idx = np.sort(order[:nseq])
        rows = np.array([(b, h) for b in idx for h in range(Hq)], np.int32)
        oracle.append(w.new_k[idx], None if w.new_v is None else w.new_v[idx],
                      oracle_new_slots(w, pool)[idx], pool)
        oracle.decode(w.q, pool, w.block_table, w.seq_lens, Hq, spec.window,
                      np.float32(spec.softmax_scale), rows=rows)
        return idx

    t0 = time.perf_counter()
    sample_step(1)
    t_one = max(time.perf_counter() - t0, 1e-4)
    budget = 120.0 / max(1, args.steps + args.warmup)
    nseq = int(max(1, min(B, budget // t_one)))
    for _ in range(max(3, args.warmup)):
        sample_step(nseq)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        idx = sample_step(nseq)
    dt = (time.perf_counter() - t0) / args.steps
    dbytes = bytes_model.decode_bytes(spec, w.seq_lens[idx], w.block_table[idx])
    abytes = bytes_model.append_bytes(spec, len(idx))
    sbytes = dbytes["kv"] + dbytes["q"] + dbytes["out"] + abytes
    value = sbytes / dt / 1e9
    sample = (f"{len(idx)} of {B} sequences of {spec.name} per step (longest first), all "
              f"{Hq} heads: append + decode, fp64 C oracle")
    return {
        "metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": reference_config(spec, w),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.record_traffic:
        print(json.dumps(record_traffic(args)), flush=True)
        return 0
    if args.impl == "reference":
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if args.chunk_only:
        import torch
        import paged_kv_decode_03_gb300 as pkv
        torch.cuda.set_device(local_rank)
        pkv.load_library()
        entry = measure_prefill(workload_spec(args), args.chunk_only, torch.device("cuda", local_rank),
                                args.steps, args.warmup, not args.no_cpu_baseline)
        print(json.dumps(entry), flush=True)
        return 0
    if args.rope_only:
        import torch
        import paged_kv_decode_03_gb300 as pkv
        torch.cuda.set_device(local_rank)
        pkv.load_library()
        dev = torch.device("cuda", local_rank)
        cpu = not args.no_cpu_baseline
        entry = {
            "c5g_rope_append": measure_rope_append(synth.C5_GLOBAL, 1e6, synth.C5_GLOBAL.head_dim // 8,
                                                   dev, args.steps, args.warmup, cpu),
            "c5s_rope_append": measure_rope_append(synth.C5_SLIDING, 1e4,
                                                   synth.C5_SLIDING.head_dim // 2, dev, args.steps,
                                                   args.warmup, cpu)}
        print(json.dumps(entry), flush=True)
        return 0
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
