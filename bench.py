"""Throughput of the gated full-attention layer step on GB300.

One "step" is one layer step (q/k/v dequant projections with the norm / rotary
/ append epilogue, causal GQA attention with the gate, o_proj) over one batch
of synthetic input.  Default workload: the 4B-class decode layer (hidden 2560,
16/4 heads, head_dim 256, rotary 64, 8-bit group-64 weights, one sequence, one
new row, cache length 4096).

Device timing: a CUDA graph of consecutive steps cycling over enough distinct
layer instances (weights + caches) that their bytes exceed 4x the L2 cache, so
every step streams from HBM; CUDA events on the launching stream.  A second
pass records per-kernel events (no programmatic overlap) for the roofline of
the dominant kernel.  e2e: the same steps through the C ABI from pinned host
buffers (gattn_layer_step_host: x and cache_pos copied in, the step, out read
back, every step; the decoder block copies around gattn_layer_step_block).

--impl reference times the float64 CPU oracle (the reference arm) on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from qwen3_gated_attention_gb300 import synth  # noqa: E402

METRIC = "gated-attn layer steps/s & tokens/s; achieved HBM GB/s vs GB300 peak"
UNIT = "layer-steps/s"


def algorithmic_bytes(spec, block=False, kv="bf16", x_folded=False):
    """Per-step and per-kernel algorithmic bytes (packed weights + bf16
    scales/biases, KV read over every attended position, KV rows written, x,
    out and the small intermediates each kernel must move).  block: the
    decoder-block step, which adds the two norm weight vectors and the
    post-norm output to the step (x is still read once).  kv="turbo4v": V rows
    are d/2 code bytes + d/16 E4M3 scale bytes instead of 2d.  x_folded: the
    q|k|v kernel converts x itself (it reads x; no x prep kernel, no fp16 copy)."""
    H, Hk, d, Hd, B, R = (spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.hidden,
                          spec.batch, spec.q_len)
    M = B * R

    def wbytes(N, K, bits, group):
        return N * K * bits // 8 + N * (K // group) * 4

    wq = wbytes(spec.n_q, Hd, spec.bits[0], spec.group[0])
    wk = wbytes(spec.n_kv, Hd, spec.bits[1], spec.group[1])
    wv = wbytes(spec.n_kv, Hd, spec.bits[2], spec.group[2])
    wo = wbytes(Hd, H * d, spec.bits[3], spec.group[3])
    pos = spec.positions().astype(np.int64)
    quant = d // 2 + d // 16                  # a Turbo4 row: codes + E4M3 scales
    row_kv = (quant if kv == "turbo4" else d * 2) + (quant if kv in ("turbo4v", "turbo4") else d * 2)
    kv_read = int(((pos + R) * Hk * row_kv).sum())
    kv_write = M * Hk * row_kv
    xb = M * Hd * (4 if spec.x_dtype == "f32" else 2)
    outb = M * Hd * 2
    x16 = M * Hd * 2
    qn = M * H * d * 2
    gate = M * H * d * 4
    o16 = M * H * d * 2
    per_kernel = {
        "xprep": xb + x16,
        "proj_qkv": wq + wk + wv + x16 + qn + gate + kv_write,
        "attn": kv_read + qn,
        "merge": gate + o16,                        # the chunk merge and the output gate
        "proj_o": wo + o16 + outb,
    }
    if x_folded:
        per_kernel["proj_qkv"] += xb - x16
        del per_kernel["xprep"]
    step = wq + wk + wv + wo + kv_read + kv_write + xb + outb
    if block:
        lnb = Hd * 2
        per_kernel["xprep"] += lnb
        per_kernel["proj_o"] += xb                   # the residual rows
        per_kernel["postnorm"] = outb + lnb + outb
        step += 2 * lnb + outb
    return step, per_kernel


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "qwen3_gated_attention_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    src_hash, traffic = None, None
    with open(path) as f:
        for line in f:
            if line.startswith("sources:"):
                src_hash = line.split(":", 1)[1].strip()
            if line.startswith("traffic_bytes_per_launch:"):
                traffic = float(line.split(":", 1)[1].strip())
    if src_hash != kernel_source_hash():
        return None
    return traffic


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"gattn_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------- cpu baseline

def oracle_sample(spec, budget_s=15.0, max_steps=64, block=False, kv="bf16"):
    """Time the oracle as it stands on a bounded sample of the workload: whole
    layer (or decoder-block) steps of the same shapes, one core."""
    import oracle as orc
    wf = synth.weights_f32(spec)
    op = [orc.quantize_affine(w.astype(np.float64), spec.bits[i], spec.group[i])
          for i, w in enumerate(wf)]
    qn, kn = synth.norm_weights_bf16(spec)
    W = orc.OracleWeights([p for p, _, _ in op], [s for _, s, _ in op], [b for _, _, b in op],
                          qn, kn, list(spec.bits), list(spec.group))
    cap = spec.capacity()
    ck, cv = synth.cache(spec, cap)
    vq = synth.turbo4v_cache(spec, cap) if kv in ("turbo4v", "turbo4") else None
    kq = synth.turbo4v_cache(spec, cap, plane="k") if kv == "turbo4" else None
    x = synth.x_values(spec, synth.layer_input(spec))
    pos = spec.positions()
    il, pl = synth.block_norm_weights_bf16(spec)
    steps = 0
    t0 = time.perf_counter()
    while steps < max_steps:
        k2, v2 = ck.copy(), cv.copy()
        ts = time.perf_counter()
        if kv == "turbo4":
            orc.layer_step_ext(spec, W, x, None, None, pos, turbo=(vq[0].copy(), vq[1].copy()),
                               turbo_k=(kq[0].copy(), kq[1].copy()))
        elif kv == "turbo4v":
            orc.layer_step_turbo4v(spec, W, x, k2, vq[0].copy(), vq[1].copy(), pos)
        elif block:
            orc.block_step(spec, W, x, il, pl, k2, v2, pos)
        else:
            orc.layer_step(spec, W, x, k2, v2, pos)
        steps += 1
        if time.perf_counter() - t0 + (time.perf_counter() - ts) > budget_s:
            break
    el = time.perf_counter() - t0
    return steps / el, steps, el


def reference_arm(args, spec):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    K, W = args.steps, max(args.warmup, 0)
    budget = min(120.0, max(10.0, 2.0 * (K + W)))
    rate, n, el = oracle_sample(spec, budget_s=budget, max_steps=max(1, K + W), block=args.block,
                                kv=args.kv)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT,
        "n_gpus": args.gpus, "steps": n, "warmup": 0, "ms_per_step": 1000.0 / rate,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(spec, args),
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{n} whole {unit_name(args)} steps of {spec.name} in "
                                   f"{el:.1f} s"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def unit_name(args):
    return "decoder-block" if args.block else "layer"


def config_dict(spec, args, extra=None):
    d = {"workload": spec.name, "hidden": spec.hidden, "num_heads": spec.num_heads,
         "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
         "rotary_dim": int(spec.head_dim * spec.partial_rotary_factor),
         "bits": list(spec.bits), "group": list(spec.group), "batch": spec.batch,
         "q_len": spec.q_len, "cache_len": int(spec.positions().max()) + spec.q_len,
         "head_chunk": not args.no_head_chunk, "parallelism": f"replicas x{args.gpus}",
         "step": "decoder block (input RMSNorm, layer, residual, post-norm)" if args.block
         else "attention layer",
         "kv_cache": {"turbo4v": "bf16 K, Turbo4 V (WHT basis, 4-bit Lloyd-Max codes, E4M3 "
                                 "group-16 scales)",
                      "turbo4": "Turbo4 K and V (WHT basis, 4-bit Lloyd-Max codes, E4M3 group-16 "
                                "scales)"}.get(args.kv, "bf16 K and V")}
    if extra:
        d.update(extra)
    return d


# ------------------------------------------------------------------ ours

# ----------------------------------------------------- replicas across ranks

def max_over_ranks(value, dist, device):
    """The largest of every rank's value (a time: the job ends with its slowest
    replica); the value itself when there is one rank."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, elapsed_ms, world):
    """Whole-job throughput: the units all replicas processed over the job's
    (slowest rank's) time."""
    return world * units_per_rank / (elapsed_ms / 1e3)


# workloads whose numbers ride along in the default line, next to the headline
PER_WORKLOAD = ("verify_2k_p46", "verify_2k_p2048", "batched_9b", "long_verify_mixed")


def cpu_baseline_entry(spec, args, budget_s, max_steps):
    rate, n, el = oracle_sample(spec, budget_s=budget_s, max_steps=max_steps, block=args.block,
                                kv=args.kv)
    return {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} whole {unit_name(args)} step{'s' if n != 1 else ''} of {spec.name} "
                      f"({el:.1f} s, one core)"}


def measure_workload(spec, args, dev, world, dist, l2, full=True):
    """Device-timed throughput of one workload: a CUDA graph of `args.steps`
    consecutive steps over rotating layer instances, replayed at least
    `args.replays` times (each replay timed with CUDA events on the launching
    stream; the median replay gives ms_per_step); then a per-kernel pass
    (events between the step's kernels, programmatic overlap off) whose
    per-kernel medians give the dominant kernel's roofline; with full=True also
    the end-to-end rate through the C ABI from pinned host buffers and the
    clocks sampled during the timed replays."""
    import torch

    from qwen3_gated_attention_gb300 import gattn
    from qwen3_gated_attention_gb300.device import DeviceLayer, x_to_device

    local = dev.index or 0
    step_bytes, kernel_bytes = algorithmic_bytes(spec, args.block, args.kv)
    n_inst = max(2, math.ceil(4 * l2 / step_bytes))
    if args.instances:
        n_inst = args.instances

    # one instance's inputs on the host, replicated across instances on the device
    wf = synth.weights_f32(spec)
    packed = [gattn.pack_affine_host(w, spec.bits[i], spec.group[i]) for i, w in enumerate(wf)]
    del wf
    qn, kn = synth.norm_weights_bf16(spec)
    cap = spec.capacity()
    ck, cv = synth.cache(spec, cap)
    vq = synth.turbo4v_cache(spec, cap) if args.kv in ("turbo4v", "turbo4") else None
    kq = synth.turbo4v_cache(spec, cap, plane="k") if args.kv == "turbo4" else None
    pos = spec.positions()
    x = synth.layer_input(spec)
    layers = []
    for _ in range(n_inst):
        dl = DeviceLayer(spec, packed, qn, kn, cap, head_chunk=not args.no_head_chunk,
                         device=dev, kv_format=args.kv)
        dl._w = None          # interchange copies are no longer needed after repacking
        dl.load_cache(kq if args.kv == "turbo4" else ck,
                      vq if args.kv in ("turbo4v", "turbo4") else cv)
        layers.append(dl)
    del ck, cv, vq, kq
    xd = x_to_device(spec, x, dev)
    pd = torch.from_numpy(pos).to(dev)
    outs = [torch.empty((spec.batch, spec.q_len, spec.hidden), dtype=torch.bfloat16, device=dev)
            for _ in range(n_inst)]
    il, pl = synth.block_norm_weights_bf16(spec)
    ild = torch.from_numpy(il.view(np.int16)).to(dev)
    pld = torch.from_numpy(pl.view(np.int16)).to(dev)
    normed = torch.empty_like(outs[0])
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream

    def step_call(dl, xp, pp, op):
        if args.block:
            gattn.layer_step_block(dl.h, xp, dl.kv, pp, spec.batch, spec.q_len, ild.data_ptr(),
                                   pld.data_ptr(), op, normed.data_ptr(), sh)
        else:
            gattn.layer_step(dl.h, xp, dl.kv, pp, spec.batch, spec.q_len, op, sh)

    def enqueue(i):
        step_call(layers[i % n_inst], xd.data_ptr(), pd.data_ptr(), outs[i % n_inst].data_ptr())

    # eager warm-up (also checks status), then the graph
    with torch.cuda.stream(stream):
        for i in range(n_inst):
            enqueue(i)
    stream.synchronize()
    for dl in layers:
        gattn.layer_poll_status(dl.h, sh)
    launches = gattn.layer_launches_per_step(layers[0].h)

    K = args.steps
    W = max(args.warmup, 3)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        graph.capture_begin()
        for i in range(K):
            enqueue(i)
        graph.capture_end()

    # warm-up: W steps (whole replays)
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(W / K))):
            graph.replay()
    stream.synchronize()

    # timed replays: at least args.replays, and at least args.min_timed_s of work
    est_ms = None
    with torch.cuda.stream(stream):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    stream.synchronize()
    est_ms = max(e0.elapsed_time(e1), 1e-3)
    n_rep = max(args.replays, int(math.ceil(args.min_timed_s * 1e3 / est_ms)) if full else 0)
    n_rep = min(n_rep, 100000)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
    clocks = ClockSampler(local) if full else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.start()
        time.sleep(0.3)
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for r in range(n_rep):
            graph.replay()
            evs[r + 1].record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    clk = clocks.stop() if clocks else None
    rep_ms = sorted(evs[r].elapsed_time(evs[r + 1]) for r in range(n_rep))
    med_ms = statistics.median(rep_ms)
    med_ms = max_over_ranks(med_ms, dist if world > 1 else None, dev)
    if world > 1:
        dist.barrier()
    ms_per_step = med_ms / K
    steps_per_s = job_rate(K, med_ms, world)
    for dl in layers:
        gattn.layer_poll_status(dl.h, sh)

    # per-kernel pass: events between the step's kernels (programmatic overlap off)
    names = gattn.layer_step_kernels(layers[0].h)
    if "xprep" not in names:               # x converted inside the q|k|v kernel
        kernel_bytes = dict(algorithmic_bytes(spec, args.block, args.kv, x_folded=True)[1])
    if "postnorm" not in names and "postnorm" in kernel_bytes:       # post-norm inside the o_proj
        kernel_bytes["proj_o"] += kernel_bytes.pop("postnorm")
    kernel_bytes = {n: kernel_bytes[n] for n in names}
    nper = max(args.replays, n_inst)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(launches + 1)] for _ in range(nper)]
    per_kernel_ms = {n: [] for n in names}
    with torch.cuda.stream(stream):
        for row in kev:
            for e in row:
                e.record(stream)          # creates the underlying cudaEvent_t
    stream.synchronize()
    with torch.cuda.stream(stream):
        for i in range(nper):
            dl = layers[i % n_inst]
            gattn.layer_set_events(dl.h, [e.cuda_event for e in kev[i]])
            enqueue(i)
            gattn.layer_set_events(dl.h, [])
    stream.synchronize()
    for i in range(nper):
        for j, n in enumerate(names):
            per_kernel_ms[n].append(kev[i][j].elapsed_time(kev[i][j + 1]))
    kernel_med_ms = {n: statistics.median(v) for n, v in per_kernel_ms.items()}
    dominant = max(kernel_bytes, key=lambda n: kernel_bytes[n])
    peak, peak_kind = load_peaks()
    achieved = kernel_bytes[dominant] / (kernel_med_ms[dominant] / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": profiled_traffic(dominant, spec.name + ("" if args.kv == "bf16"
                                                                   else "_" + args.kv)),
                "kernel": dominant, "peak_source": peak_kind, "kernel_launches_timed": nper,
                "kernel_median_us": {n: 1e3 * v for n, v in kernel_med_ms.items()},
                "kernel_bytes": kernel_bytes}

    res = {"value": steps_per_s, "ms_per_step": ms_per_step, "steps": K, "warmup": W,
           "replays": n_rep, "replay_ms": {"median": med_ms, "min": rep_ms[0], "max": rep_ms[-1]},
           "tokens_per_s": steps_per_s * spec.batch * spec.q_len,
           "hbm_gbs": steps_per_s / world * step_bytes / 1e9,
           "hbm_frac_of_peak": steps_per_s / world * step_bytes / 1e9 / peak,
           "bytes_per_step": step_bytes, "roofline": roofline, "launches": launches,
           "kernels": names,
           "n_inst": n_inst, "inst_bytes": n_inst * step_bytes, "clocks": clk}

    if full:
        # e2e through the C ABI with pinned host buffers, copies inside the timed region
        xh = torch.from_numpy(np.ascontiguousarray(xd.cpu().view(torch.int16).numpy())).pin_memory() \
            if spec.x_dtype != "f32" else xd.cpu().pin_memory()
        ph = torch.from_numpy(pos.copy()).pin_memory()
        oh = torch.empty(outs[0].shape, dtype=torch.bfloat16).pin_memory()
        xdev = torch.empty_like(xd)
        pdev = torch.empty_like(pd)
        n_e2e = max(1, args.e2e_steps)     # consecutive steps, independent of K
        h2d = xh.numel() * xh.element_size() + ph.numel() * ph.element_size()
        d2h = oh.numel() * oh.element_size()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(n_e2e):
                dl = layers[i % n_inst]
                if not args.block:
                    # one C call: x and cache_pos in, the step, out back
                    gattn.layer_step_host(dl.h, xh.data_ptr(), dl.kv, ph.data_ptr(), spec.batch,
                                          spec.q_len, oh.data_ptr(), sh)
                    continue
                xdev.view(torch.int16 if spec.x_dtype != "f32" else torch.float32).copy_(
                    xh, non_blocking=True)
                pdev.copy_(ph, non_blocking=True)
                step_call(dl, xdev.data_ptr(), pdev.data_ptr(), outs[i % n_inst].data_ptr())
                oh.copy_(normed, non_blocking=True)
            e1.record(stream)
        stream.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist if world > 1 else None, dev)
        res["e2e"] = {"value": job_rate(n_e2e, e2e_ms, world), "unit": UNIT,
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e}
    del graph
    for dl in layers:
        dl.close()
    del layers, outs, xd, pd
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return res


def our_arm(args, spec):
    import torch
    import torch.distributed as dist

    from qwen3_gated_attention_gb300 import build as libbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    others = [w for w in PER_WORKLOAD if w != spec.name] \
        if (args.per_workload and not args.block and args.kv == "bf16") \
        else []

    # CPU baselines first (rank 0, N = 1): the oracle as it stands, before any
    # GPU work; one bounded oracle step for each ride-along workload
    cpu, cpu_other = None, {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_entry(spec, args, args.cpu_budget, 64)
        for w in others:
            cpu_other[w] = cpu_baseline_entry(synth.WORKLOADS[w], args, 1.0, 1)

    if rank == 0:
        libbuild.build()
    if world > 1:
        dist.init_process_group("nccl")
        dist.barrier()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 129 * 2 ** 20

    r = measure_workload(spec, args, dev, world, dist, l2, full=True)
    per = {}
    for w in others:
        o = measure_workload(synth.WORKLOADS[w], args, dev, world, dist, l2, full=False)
        per[w] = {"value": o["value"], "unit": UNIT, "ms_per_step": o["ms_per_step"],
                  "tokens_per_s": o["tokens_per_s"], "hbm_gbs": o["hbm_gbs"],
                  "hbm_frac_of_peak": o["hbm_frac_of_peak"], "bytes_per_step": o["bytes_per_step"],
                  "steps": o["steps"], "replays": o["replays"], "roofline": o["roofline"],
                  "config": config_dict(synth.WORKLOADS[w], args),
                  "cpu_baseline": cpu_other.get(w)}

    line = {
        "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world, "steps": r["steps"],
        "warmup": r["warmup"], "ms_per_step": r["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(spec, args, {
            "l2": f"rotating {r['n_inst']} layer instances, {r['inst_bytes'] / 2**20:.0f} MiB "
                  f"> 4x L2 ({l2 / 2**20:.0f} MiB)",
            "arith": "bf16/fp16 tensor-core operands, fp32 accumulate; 8/4/6/3-bit codes",
            "path": f"{r['launches']} kernels per step ({', '.join(r['kernels'])})",
            "timing": f"median of {r['replays']} timed replays of a {r['steps']}-step graph"}),
        "replays": r["replays"], "replay_ms": r["replay_ms"],
        "tokens_per_s": r["tokens_per_s"], "hbm_gbs": r["hbm_gbs"],
        "hbm_frac_of_peak": r["hbm_frac_of_peak"], "bytes_per_step": r["bytes_per_step"],
        "roofline": r["roofline"], "cpu_baseline": cpu, "e2e": r["e2e"],
        "gpu_launches": r["launches"] * r["steps"] * r["replays"],
        "clocks": r["clocks"],
    }
    if per:
        line["per_workload"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20, help="steps per timed graph replay")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_4b", choices=list(synth.WORKLOADS))
    ap.add_argument("--instances", type=int, default=0)
    ap.add_argument("--replays", type=int, default=20,
                    help="timed replays of the step graph, at least (median reported)")
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="replay the graph for at least this long (seconds) in the timed region")
    ap.add_argument("--no-per-workload", dest="per_workload", action="store_false",
                    help="time only the selected workload (no per_workload entries)")
    ap.add_argument("--e2e-steps", type=int, default=200,
                    help="consecutive steps of the end-to-end leg")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-head-chunk", action="store_true")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "turbo4v", "turbo4"],
                    help="KV cache format: bf16, bf16 K with a Turbo4 V cache, or Turbo4 K and V")
    ap.add_argument("--block", action="store_true",
                    help="time the decoder-block step (input RMSNorm + layer + residual + "
                         "post-attention RMSNorm) instead of the layer alone")
    args = ap.parse_args()
    spec = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        reference_arm(args, spec)
    else:
        our_arm(args, spec)


if __name__ == "__main__":
    main()
