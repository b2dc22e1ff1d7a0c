"""The bench's JSON contract on the CPU: the reference arm (the oracle timed on
the host) prints one line with every key the contract asks for, only rank 0
prints, and the algorithmic-bytes accounting follows the cache formats."""
import json
import os
import subprocess
import sys

import pytest

from qwen3_gated_attention_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _reference_line(*extra, env=None):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           "tiny", "--steps", "1", "--warmup", "0", *extra]
    e = dict(os.environ)
    e.update(env or {})
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=e, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


@pytest.mark.parametrize("extra", [(), ("--kv", "turbo4v"), ("--kv", "turbo4"), ("--block",)])
def test_reference_arm_prints_one_complete_line(extra):
    lines = _reference_line(*extra)
    assert len(lines) == 1
    d = lines[0]
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_on_rank_zero_only():
    assert _reference_line(env={"RANK": "1", "WORLD_SIZE": "2"}) == []


def test_algorithmic_bytes_follow_the_cache_format():
    spec = synth.WORKLOADS["batched_9b"]
    d, Hk, R = spec.head_dim, spec.num_kv_heads, spec.q_len
    pos = spec.positions().astype(int)
    attended = int(((pos + R) * Hk).sum())            # (token, KV head) pairs read
    bf16, per_bf16 = bench.algorithmic_bytes(spec)
    t4v, per_t4v = bench.algorithmic_bytes(spec, kv="turbo4v")
    t4, per_t4 = bench.algorithmic_bytes(spec, kv="turbo4")
    quant = d // 2 + d // 16                            # codes + E4M3 scales per row
    # the attention's K/V read shrinks by exactly the per-row byte difference
    assert per_bf16["attn"] - per_t4v["attn"] == attended * (2 * d - quant)
    assert per_t4v["attn"] - per_t4["attn"] == attended * (2 * d - quant)
    # weights and x/out are the same; the step changes by the read and the written rows
    M = spec.batch * spec.q_len
    assert bf16 - t4v == (attended + M * Hk) * (2 * d - quant)
    assert t4v - t4 == (attended + M * Hk) * (2 * d - quant)
    # the decoder block adds the two norm vectors and the normed output to the step
    blk, per_blk = bench.algorithmic_bytes(spec, block=True)
    assert blk - bf16 == 2 * spec.hidden * 2 + M * spec.hidden * 2
    assert set(per_blk) == set(per_bf16) | {"postnorm"}


def test_reference_arm_under_torchrun_prints_one_line():
    """Launched the way a multi-GPU run launches it (torchrun, two ranks on
    127.0.0.1): rank 0 alone prints, the other rank exits 0 without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2
