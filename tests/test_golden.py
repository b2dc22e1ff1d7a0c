"""Numbers the source pages print (tests/golden/, each file citing its page):
the 4B-class geometry, rotary dimension counts, the verify head-chunk plans
around the route's boundaries, and the KV cache sizes of the bf16, Turbo4 and
Bf16KTurbo4V formats.  Each is checked against the oracle, the library's host
entry points and the synthetic workloads, none of which the fixtures came from."""
import os
import sys

import numpy as np
import pytest

import oracle as orc
from qwen3_gated_attention_gb300 import gattn, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.split("#", 1)[0].strip() for l in f if l.split("#", 1)[0].strip()]


def _keyed(name):
    return {k: v for k, v in (l.split(None, 1) for l in _lines(name))}


# ------------------------------------------------------------ geometry

def test_4b_workload_has_the_printed_geometry():
    g = _keyed("qwen35_4b_geometry.txt")
    s = synth.WORKLOADS["decode_4b"]
    assert s.hidden == int(g["hidden"])
    assert s.num_heads == int(g["num_heads"]) and s.num_kv_heads == int(g["num_kv_heads"])
    assert s.head_dim == int(g["head_dim"])
    assert set(s.group) == {int(g["group_size"])} and set(s.bits) == {int(g["bits"])}
    assert s.rms_eps == float(g["rms_eps"]) and s.rope_theta == float(g["rope_theta"])
    assert s.partial_rotary_factor == float(g["partial_rotary_factor"])
    assert s.n_q == int(g["q_total"])


def test_4b_rotary_dims_in_the_oracle_and_the_library():
    g = _keyed("qwen35_4b_geometry.txt")
    d, prf = int(g["head_dim"]), float(g["partial_rotary_factor"])
    assert orc.rotary_dims(d, prf) == int(g["rotary_dim"])
    cfg = gattn.make_cfg(int(g["hidden"]), int(g["num_heads"]), int(g["num_kv_heads"]), d, prf,
                         float(g["rope_theta"]), float(g["rms_eps"]), (int(g["bits"]),) * 4,
                         (int(g["group_size"]),) * 4, x_dtype="bf16", max_batch=1, max_q_len=4)
    gattn.cfg_validate(cfg)                       # the library serves this geometry
    assert gattn.rotary_dims(cfg) == int(g["rotary_dim"])


@pytest.mark.parametrize("row", _lines("rope_dims.txt"))
def test_printed_rotary_dim_counts(row):
    d, prf, want = row.split()
    assert orc.rotary_dims(int(d), float(prf)) == int(want)
    cfg = gattn.make_cfg(128, 1, 1, int(d), float(prf), 1e4, 1e-6, (4,) * 4, (64,) * 4)
    assert gattn.rotary_dims(cfg) == int(want)


# ------------------------------------------------------------ head-chunk plans

def _plans():
    out = []
    for l in _lines("ds4_113_plan.txt"):
        head, chunks = l.split(":", 1)
        q, h, hk, on = (int(t) for t in head.split())
        want = [tuple(int(t) for t in c.split(":")) for c in chunks.split()]
        out.append((q, h, hk, on, want))
    return out


@pytest.mark.parametrize("q,h,hk,on,want", _plans())
def test_head_chunk_plans_worked_by_hand(q, h, hk, on, want):
    assert orc.head_chunk_plan(q, h, hk, bool(on)) == want
    assert gattn.head_chunk_plan(q, h, hk, bool(on)) == want


def test_the_shipped_verify_case_is_the_verify_workload():
    """DS4Server issue 113's case: 24 query / 2 KV heads, d 256, four rows after 46 tokens."""
    s = synth.WORKLOADS["verify_2k_p46"]
    assert (s.num_heads, s.num_kv_heads, s.head_dim, s.q_len) == (24, 2, 256, 4)
    assert int(s.positions()[0]) == 46
    q, h, hk, on, want = _plans()[0]
    assert (q, h, hk, on) == (s.q_len, s.num_heads, s.num_kv_heads, 1)


# ------------------------------------------------------------ KV cache sizes

def _kv_sizes():
    g = _lines("kv_cache_bytes.txt")
    kv = {}
    for l in g:
        t = l.split()
        if t[0] in ("bf16", "turbo4", "turbo4v"):
            kv[t[0]] = tuple(int(v) for v in t[1:])
        else:
            kv[t[0]] = float(t[1])
    return kv


def _cache_spec(kv):
    s = synth.WORKLOADS["decode_4b"]
    assert s.num_kv_heads * s.head_dim == int(kv["kv_dim"])
    return s


def test_synthetic_caches_have_the_printed_sizes():
    kv = _kv_sizes()
    s = _cache_spec(kv)
    cap = int(kv["max_seq"])
    ck, cv = synth.cache(s, cap)
    assert (ck.nbytes, cv.nbytes) == kv["bf16"][:2]
    vc, vs = synth.turbo4v_cache(s, cap)
    kc, ks = synth.turbo4v_cache(s, cap, plane="k")
    assert (kc.nbytes, vc.nbytes, ks.nbytes, vs.nbytes) == kv["turbo4"]
    assert (ck.nbytes, vc.nbytes, 0, vs.nbytes) == kv["turbo4v"]


def test_oracle_quantizer_writes_the_printed_bytes_per_row():
    kv = _kv_sizes()
    s = _cache_spec(kv)
    rows = int(kv["max_seq"]) * s.num_kv_heads
    v = synth.f32_to_bf16_bits(np.random.default_rng(0).standard_normal((8, s.head_dim)).astype(np.float32))
    codes, scales = orc.turbo4_quantize_rows(v)
    assert codes.dtype == np.uint8 and scales.dtype == np.uint8
    _, vb, _, vsb = kv["turbo4"]
    assert codes.shape[1] * rows == vb and scales.shape[1] * rows == vsb


def test_turbo4_ratio_is_the_printed_one():
    kv = _kv_sizes()
    bf = sum(kv["bf16"])
    t4 = sum(kv["turbo4"])
    assert round(bf / t4, 2) == kv["turbo4_ratio"]


@pytest.mark.parametrize("fmt", ["bf16", "turbo4v", "turbo4"])
def test_bench_accounting_reads_the_whole_printed_cache(fmt):
    """A decode step at the last position reads every cache row once: the
    attention's algorithmic bytes minus its q rows equal the printed cache size,
    and the merge moves the gate rows (fp32) and the gated operand (fp16)."""
    kv = _kv_sizes()
    s = _cache_spec(kv)
    assert int(s.positions()[0]) + s.q_len == int(kv["max_seq"]) and s.batch == 1
    _, per = bench.algorithmic_bytes(s, kv=fmt)
    rows = s.batch * s.q_len * s.num_heads * s.head_dim
    assert per["attn"] - rows * 2 == sum(kv[fmt])
    assert per["merge"] == rows * (4 + 2)
