"""The committed ncu summaries (profiles/) against the bench that reads them:
each names the full command it came from (committed files only, clocks left
alone), its traffic line is the DRAM read + write bytes its own metric table
shows, its algorithmic bytes are the bench's figure for that kernel and
workload, launch-list shares add up, and the bench drops a summary's traffic
once the kernel sources differ from the ones it was taken on."""
import os
import re
import sys

import pytest

from qwen3_gated_attention_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")
sys.path.insert(0, ROOT)
import bench  # noqa: E402

UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
SUMMARIES = sorted(f for f in os.listdir(PROFILES) if f.endswith(".md")) if os.path.isdir(PROFILES) else []
KERNEL_SUMMARIES = [f for f in SUMMARIES if not f.startswith("launches_")]
LAUNCH_SUMMARIES = [f for f in SUMMARIES if f.startswith("launches_")]


def _text(name):
    with open(os.path.join(PROFILES, name)) as f:
        return f.read()


def _command(text):
    block = re.search(r"```\n(.*?)```", text, re.S).group(1)
    return " ".join(l.rstrip("\\").strip() for l in block.splitlines())


def _workload_and_kv(cmd):
    w = re.search(r"--workload (\S+)", cmd).group(1)
    kv = re.search(r"--kv (\S+)", cmd)
    return w, kv.group(1) if kv else "bf16"


def test_there_are_kernel_and_launch_summaries():
    assert KERNEL_SUMMARIES and LAUNCH_SUMMARIES


@pytest.mark.parametrize("name", SUMMARIES)
def test_summary_names_its_command_and_sources(name):
    t = _text(name)
    cmd = _command(t)
    assert cmd.startswith("ncu ") and "--clock-control none" in cmd
    assert "python bench.py" in cmd and "_work" not in cmd
    assert re.search(r"^sources: [0-9a-f]{16}$", t, re.M)
    w, kv = _workload_and_kv(cmd)
    assert w in synth.WORKLOADS
    # the file is named for the kernel (or launch list), the workload and the cache format
    stem = name[:-3]
    assert stem.endswith(w if kv == "bf16" else f"{w}_{kv}")


@pytest.mark.parametrize("name", KERNEL_SUMMARIES)
def test_traffic_line_is_the_dram_bytes_of_the_table(name):
    t = _text(name)
    traffic = float(re.search(r"^traffic_bytes_per_launch: (\d+)$", t, re.M).group(1))
    rd = re.search(r"`dram__bytes_read.sum` \| ([\d.]+) (\w+)", t)
    wr = re.search(r"`dram__bytes_write.sum` \| ([\d.]+) (\w+)", t)
    total = float(rd.group(1)) * UNITS[rd.group(2)] + float(wr.group(1)) * UNITS[wr.group(2)]
    # the table prints six to seven significant digits
    assert abs(traffic - total) <= 1e-6 * traffic + 1


@pytest.mark.parametrize("name", KERNEL_SUMMARIES)
def test_algorithmic_bytes_are_the_bench_figure(name):
    t = _text(name)
    w, kv = _workload_and_kv(_command(t))
    kernel = name.split("_" + w)[0]
    stated = int(re.search(r"Algorithmic bytes per launch: ([\d,]+)", t).group(1).replace(",", ""))
    _, per = bench.algorithmic_bytes(synth.WORKLOADS[w], kv=kv)
    assert per[kernel] == stated


@pytest.mark.parametrize("name", LAUNCH_SUMMARIES)
def test_launch_list_shares_add_up(name):
    rows = [l for l in _text(name).splitlines() if l.startswith("| ") and not l.startswith("| kernel")
            and not l.startswith("|---")]
    shares, totals = [], []
    for r in rows:
        cells = [c.strip() for c in r.strip("|").split("|")]
        launches, avg, total, share = int(cells[2]), float(cells[3]), float(cells[4]), float(cells[5])
        assert abs(launches * avg - total) <= 0.01 * total + 0.1
        shares.append(share)
        totals.append(total)
    assert abs(sum(shares) - 1.0) <= 0.01
    for s, tot in zip(shares, totals):
        assert abs(s - tot / sum(totals)) <= 0.002


def test_bench_drops_traffic_taken_on_other_sources(monkeypatch):
    name = KERNEL_SUMMARIES[0]
    t = _text(name)
    w, kv = _workload_and_kv(_command(t))
    kernel = name.split("_" + w)[0]
    key = w if kv == "bf16" else f"{w}_{kv}"
    src = re.search(r"^sources: (\w+)$", t, re.M).group(1)
    traffic = float(re.search(r"^traffic_bytes_per_launch: (\d+)$", t, re.M).group(1))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: src)
    assert bench.profiled_traffic(kernel, key) == traffic
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.profiled_traffic(kernel, key) is None
