"""Host-side logic of bench.py, on CPU: the reference arm's JSON line, the flop and byte
accounting, and the rule that recorded ncu traffic is reported only while the kernel
sources still match the hash stored with it."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np

import bench
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "GFLOP/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["n_gpus"] == 1 and line["steps"] == 2
    assert line["config"]["workload"] == bench.DESCRIPTION["tiny"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_accounting_counts_what_the_step_does():
    """Flops are 2*nnz*N (SpMM) plus 2*nnz*kd (SDDMM); the compulsory bytes read the B and BT
    rows of the columns that occur and the A rows that hold entries, counted here by brute
    force over the entries."""
    w = wl.generate("tiny")
    acc = bench.accounting(w)
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    nnz, N, kd = len(col), w.B.shape[1], w.A.shape[1]
    assert acc["spmm"]["flops"] == 2 * nnz * N
    assert acc["sddmm"]["flops"] == 2 * nnz * kd
    assert bench.step_flops(acc) == 2 * nnz * (N + kd)
    used_cols = set(int(c) for c in col)
    rows_with_entries = sum(1 for i in range(w.m) if ro[i + 1] > ro[i])
    b = w.values.element_size()
    # B rows of used columns and all of C
    spmm_dense = len(used_cols) * N * b + w.m * N * b
    assert acc["spmm"]["bytes"] - spmm_dense == nnz * (b + 2) + 4 * (w.m + 1) + 2 * w.m
    sddmm_dense = rows_with_entries * kd * b + len(used_cols) * kd * b
    assert acc["sddmm"]["bytes"] - sddmm_dense == nnz * 2 + 4 * (w.m + 1) + 2 * w.m + nnz * b
    assert acc["csr_add"]["bytes"] >= 2 * w.m * w.n * b
    assert np.isclose(acc["csr_add"]["bytes"] - 2 * w.m * w.n * b, nnz * (b + 2) + 4 * (w.m + 1))


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash("k.cu")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.md").write_text(
        "| workload | op | sources | sha256[:16] | bytes |\n|---|---|---|---|---|\n"
        f"| rosa | spmm | k.cu | {h} | 12345 |\n")
    assert bench.recorded_traffic("spmm", "rosa") == {"bytes": 12345, "read": None, "write": None}
    assert bench.recorded_traffic("sddmm", "rosa") is None
    assert bench.recorded_traffic("spmm", "llama_mlp") is None
    # rows with read and write columns
    (tmp_path / "profiles" / "traffic.md").write_text(
        "| workload | op | sources | sha256[:16] | read | write | bytes |\n|---|---|---|---|---|---|---|\n"
        f"| butterfly | sddmm | k.cu | {h} | 100 | 20 | 120 |\n")
    assert bench.recorded_traffic("sddmm", "butterfly") == {"bytes": 120, "read": 100, "write": 20}
    # rows that also give the L2 write bytes
    (tmp_path / "profiles" / "traffic.md").write_text(
        "| workload | op | sources | sha256[:16] | read | write | bytes | L2 write bytes |\n"
        "|---|---|---|---|---|---|---|---|\n"
        f"| butterfly | sddmm | k.cu | {h} | 100 | 20 | 120 | 300 |\n")
    assert bench.recorded_traffic("sddmm", "butterfly") == {"bytes": 120, "read": 100, "write": 20, "l2_write": 300}
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.recorded_traffic("sddmm", "butterfly") is None


def test_committed_traffic_table_parses():
    """Every row of the committed table names existing sources and a 16-digit hash."""
    rows = [ln for ln in open(os.path.join(ROOT, "profiles", "traffic.md")) if "/csrc/" in ln]
    assert rows
    for ln in rows:
        cells = [p.strip() for p in ln.strip().strip("|").split("|")]
        assert len(cells) in (5, 7, 8), ln  # | read | write | bytes | (L2 write bytes |)
        wk, op, srcs, h = cells[:4]
        assert wk in wl.SPECS and op in ("sort_rows", "plan", "spmm", "sddmm", "csr_add")
        assert len(h) == 16 and int(cells[4 if len(cells) == 5 else 6]) > 0
        if len(cells) >= 7:
            assert int(cells[4]) + int(cells[5]) == int(cells[6])
        if len(cells) == 8:
            assert int(cells[7]) >= 0
        for p in srcs.split("+"):
            assert os.path.exists(os.path.join(ROOT, p)), p


def test_reference_arm_config_matches_the_gpu_arm():
    """The reference arm's config object is the one the GPU arm prints for its headline
    workload (both come from bench.config_dict), and the default run's headline is the
    butterfly layer, the largest configuration."""
    import argparse
    args = argparse.Namespace(workload="all", sddmm_backend="structure_aware", spmm_path="auto")
    assert bench.headline_name(args) == "butterfly"
    assert bench.workload_list(args)[:5] == wl.CONFIG_ORDER
    w = wl.generate("tiny")
    cfg = bench.config_dict("tiny", w, args)
    assert cfg["workload"] == bench.DESCRIPTION["tiny"] and cfg["N"] == 64 and cfg["kd"] == 64
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert out.returncode == 0, out.stderr[-2000:]
    assert json.loads(out.stdout.strip().splitlines()[-1])["config"] == cfg
