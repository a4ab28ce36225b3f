"""Host logic of bench.py on CPU: byte models, clock summaries, the traffic
record's staleness check, max-over-ranks with gloo (world size 2), and the
reference arm (the CPU oracle) printing its JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_byte_models():
    R, S = 8, 256 << 20
    assert bench.algo_bytes("twoshot", R, S) == {"compulsory": 16 * S, "logical": 16 * S}
    assert bench.algo_bytes("oneshot", R, S)["logical"] == 72 * S
    assert bench.algo_bytes("twoshot_pull", R, S)["logical"] == 23 * S


def test_clock_summary_and_percentile():
    s = [{"sm_mhz": 1900.0, "reasons": ["sw_power_cap"]}, {"sm_mhz": 1800.0, "reasons": []},
         {"sm_mhz": 300.0, "reasons": ["gpu_idle"]}]
    c = bench.summarize_clocks(s, 2070.0)
    assert c["sm_mhz"] == 1850.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["gpu_idle", "sw_power_cap"]
    assert bench.percentile([1, 2, 3, 4, 5], 0.5) == 3
    assert bench.percentile([1.0, 3.0], 0.5) == 2.0


def test_traffic_record_goes_stale(tmp_path, monkeypatch):
    rec = {"R": 8, "bytes_per_rank": 1 << 20, "dram_bytes_per_launch": 16 << 20,
           "source_sha256": bench.kernel_source_hash()}
    p = tmp_path / "t.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    assert bench.recorded_traffic(8, 256 << 20) == 16 * (256 << 20)
    rec["source_sha256"] = "0" * 16
    p.write_text(json.dumps(rec))
    assert bench.recorded_traffic(8, 256 << 20) is None


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


_WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
r = dist.get_rank()
bench.barrier()
m = bench.max_over_ranks(10.0 + 5 * r)
bench.barrier()
print("RESULT", r, m, flush=True)
dist.destroy_process_group()
"""


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", _WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    vals = sorted(tuple(l.split()[1:]) for o, _ in outs for l in o.splitlines() if l.startswith("RESULT"))
    assert vals == [("0", "15.0"), ("1", "15.0")]


def test_reference_arm_prints_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3"], env=env, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["metric"] == bench.METRIC
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # the same workload as the GPU arm's line, timed whole every step
    assert d["config"] == bench._config(bench.R_DEFAULT, bench.N_DEFAULT)
    assert "whole workload" in d["cpu_baseline"]["sample"]


def test_reference_arm_nonzero_rank_is_silent():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3"], env=env, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_parse_dram_csv(tmp_path):
    """ncu --csv launch lists: per launch, dram read + write bytes summed, in launch order."""
    p = tmp_path / "l.csv"
    hdr = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size",'
           '"Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n')
    rows = []
    for i, (name, rd, wr) in enumerate([("k_bump_epoch(unsigned int *)", 64, 0),
                                        ("void k_twoshot_st<F32T, OpSum, 8, 1>(ArArgs)", 1000, 900),
                                        ("void k_oneshot<F32T, OpSum, 8, 2>(ArArgs)", 10, 20)]):
        for metric, v in (("dram__bytes_read.sum", rd), ("dram__bytes_write.sum", wr)):
            rows.append(f'"{i}","1","python3","h","{name}","1","7","(256, 1, 1)","(1, 1, 1)","0","10.3",'
                        f'"Command line profiler metrics","{metric}","byte","{v}"\n')
    p.write_text("==PROF== Connected\n" + hdr + "".join(rows))
    got = bench.parse_dram_csv(str(p))
    assert [n.split("<")[0].split("(")[0].split()[-1] for n, _ in got] == [
        "k_bump_epoch", "k_twoshot_st", "k_oneshot"]
    assert [b for _, b in got] == [64.0, 1900.0, 30.0]


def test_table_rows_cover_every_config():
    rows = bench.table_rows()
    labels = {r[1] for r in rows}
    assert labels == {1, 2, 3, 4, 5}
    assert len({(r[0], r[2], r[3]) for r in rows}) == len(rows)          # no duplicate row
    sweep = [r for r in rows if r[1] == 4]
    assert sorted({r[4] * 4 for r in sweep}) == [1024 * 4 ** k for k in range(11)]
    assert {r[2] for r in rows if r[1] == 3} == {"twoshot", "twoshot_pull"}
    assert {r[5] for r in rows if r[1] == 5} == {1, 8, 64}
    assert set(bench._MAIN_KERNEL) >= {r[2] for r in rows}


def test_format_table_flags_l2_served_rows():
    base = {"label": "3", "algo": "twoshot", "dtype": "f32", "R": 8, "bytes_per_rank": 1 << 28,
            "t_ms": 0.6, "algbw": 400.0, "compulsory_gbs": 7000.0, "parity": True,
            "oracle_1t_ms": 200.0, "oracle_nt_ms": 16.0, "l2_resident": False}
    rows = [dict(base, logical_gbs=7000.0, dram_gbs=6900.0),
            dict(base, algo="twoshot_pull", logical_gbs=9600.0, dram_gbs=6600.0),
            dict(base, label="1", logical_gbs=100.0, dram_gbs=50.0, l2_resident=True),
            dict(base, label="5", algo="put_signal", logical_gbs=100.0, parity=False, oracle_nt_ms=None)]
    md = bench.format_table(rows, 6789.0, "measured", 16, "cpu").splitlines()
    assert "oracle 16-thread" in md[0]
    assert "| 1.01 |" in md[2] and "L2-served" not in md[2]
    assert "1.45 (L2-served)" in md[3]
    assert "L2-resident (n/m)" in md[4]
    assert "**MISMATCH**" in md[5] and "(compulsory)" in md[5]
