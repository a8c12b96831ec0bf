"""Host-side pieces of bench.py that need no GPU: the DRAM-traffic record
written from an ncu capture, and its invalidation when the kernel sources
change."""
from __future__ import annotations

import argparse
import csv
import json

import bench
from paged_kv_decode_03_gb300 import synth


def _raw_csv(path, kernel, read_mb, write_mb):
    """A raw-page CSV as `ncu -i REPORT --page raw --csv` writes it: names,
    units, then one row per launch."""
    with open(path, "w", newline="") as f:
        w = csv.writer(f)
        w.writerow(["ID", "Kernel Name", "dram__bytes_read.sum", "dram__bytes_write.sum"])
        w.writerow(["", "", "Mbyte", "Kbyte"])
        w.writerow(["0", kernel, f"{read_mb}", f"{write_mb * 1000}"])


def _args(tmp_path, config, batch, csv_path):
    return argparse.Namespace(config=config, batch=batch, split_tokens=0,
                              record_traffic=str(csv_path),
                              traffic_path=str(tmp_path / "traffic.json"))


def test_record_traffic_scales_by_algorithmic_bytes(tmp_path):
    raw = tmp_path / "raw.csv"
    _raw_csv(raw, "void pkv::decode_kernel<256, 2, 0>(DecodeParams, CUtensorMap_st, CUtensorMap_st)",
             272.95, 2.99)
    e = bench.record_traffic(_args(tmp_path, "c2", 32, raw))
    cap = bench.layout_bytes(synth.shrink(synth.C2, batch=32))
    full = bench.layout_bytes(synth.C2)
    dram = 272.95e6 + 2.99e6
    assert e["kernel_family"] == "cuda_core"
    assert e["capture_algorithmic_bytes"] == cap
    assert e["capture_dram_bytes"] == round(dram)
    assert e["bytes_per_launch"] == round(dram * full / cap)
    assert e["sources_sha"] == bench.csrc_sha(bench.KERNEL_SOURCES["cuda_core"])
    d = json.loads((tmp_path / "traffic.json").read_text())
    assert d["c2"] == e


def test_record_traffic_tensor_core_family_and_merge(tmp_path):
    (tmp_path / "traffic.json").write_text(json.dumps({"c2": {"kept": 1}}))
    raw = tmp_path / "raw.csv"
    _raw_csv(raw, "void pkv::decode_tc_kernel<256, 16>(DecodeParams, CUtensorMap_st, CUtensorMap_st, "
                  "CUtensorMap_st)", 132.05, 2.97)
    e = bench.record_traffic(_args(tmp_path, "c3", 16, raw))
    assert e["kernel_family"] == "tensor_core"
    assert e["sources_sha"] == bench.csrc_sha(bench.KERNEL_SOURCES["tensor_core"])
    d = json.loads((tmp_path / "traffic.json").read_text())
    assert d["c2"] == {"kept": 1} and d["c3"] == e


def test_recorded_traffic_only_for_current_sources():
    """The committed record is read back only while its sources_sha matches
    the kernel's current sources."""
    with open(bench.os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for name, e in d.items():
        current = e["sources_sha"] == bench.csrc_sha(bench.KERNEL_SOURCES[e["kernel_family"]])
        assert (bench.recorded_traffic(name) == e["bytes_per_launch"]) == current, name
