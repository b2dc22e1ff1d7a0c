"""Builds one parity case: the same seeded inputs for the CUDA library (packed
by the library's host packer) and for the oracle (packed by its own packer),
and runs either side."""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle as orc
from qwen3_gated_attention_gb300 import gattn, synth
from qwen3_gated_attention_gb300.synth import bf16_bits_to_f32


@dataclass
class Case:
    spec: object
    lib_packed: list
    orc_weights: object
    qn: np.ndarray
    kn: np.ndarray
    x: np.ndarray
    cap: int
    pos: np.ndarray
    ck: np.ndarray
    cv: np.ndarray


def make_case(spec, fill=0x3F80, capacity=None, with_cache=True) -> Case:
    wf = synth.weights_f32(spec)
    lib_packed, op, os_, ob = [], [], [], []
    for i, w in enumerate(wf):
        lib_packed.append(gattn.pack_affine_host(w, spec.bits[i], spec.group[i]))
        p, s, b = orc.quantize_affine(w.astype(np.float64), spec.bits[i], spec.group[i])
        op.append(p), os_.append(s), ob.append(b)
    qn, kn = synth.norm_weights_bf16(spec)
    W = orc.OracleWeights(op, os_, ob, qn, kn, list(spec.bits), list(spec.group))
    cap = capacity or spec.capacity()
    pos = spec.positions()
    ck = cv = None
    if with_cache:
        ck, cv = synth.cache(spec, cap, fill)
    return Case(spec, lib_packed, W, qn, kn, synth.layer_input(spec), cap, pos, ck, cv)


def oracle_run(case: Case, head_chunk=True, batches=None, x=None, pos=None, ck=None, cv=None,
               spec=None):
    """Oracle on all sequences or on the listed ones.  Returns dict of arrays
    (caches as [B'][Hk][cap][d] bf16 bits after the step)."""
    spec = spec or case.spec
    idx = list(range(spec.batch)) if batches is None else list(batches)
    x = case.x if x is None else x
    pos = case.pos if pos is None else pos
    ck = case.ck if ck is None else ck
    cv = case.cv if cv is None else cv
    sub = spec.with_(batch=len(idx))
    xs = np.ascontiguousarray(synth.x_values(spec, x)[idx])
    k2 = np.ascontiguousarray(ck[idx]).copy()
    v2 = np.ascontiguousarray(cv[idx]).copy()
    p2 = np.ascontiguousarray(pos[idx])
    out, y, attn = orc.layer_step(sub, case.orc_weights, xs, k2, v2, p2, head_chunk=head_chunk,
                                  taps=True)
    return dict(out=out, y=y, attn=attn, k=k2, v=v2, pos=p2)


def new_rows(cache_bits, pos, R):
    """[B][Hk][R][d] float64 values of the rows written at pos .. pos+R-1."""
    return np.stack([bf16_bits_to_f32(cache_bits[b, :, pos[b]:pos[b] + R]).astype(np.float64)
                     for b in range(len(pos))])


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps (monotone integer mapping of the bit patterns)."""
    def key(h):
        h = h.astype(np.int32)
        return np.where(h & 0x8000, 0x8000 - (h & 0x7FFF), 0x8000 + h)
    return np.abs(key(a_bits) - key(b_bits))

