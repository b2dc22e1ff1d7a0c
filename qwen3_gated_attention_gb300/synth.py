"""Seeded synthetic inputs for the gated full-attention layer.

This module only draws numbers: it holds none of the layer's arithmetic (no
quantizer, no norm, no rotary, no attention).  Both the CUDA path and the CPU
oracle take their inputs from here.

Recipe (every tensor has its own substream ``numpy.random.default_rng([seed, id, ...])``):

* weights  ``N(0, 0.02)`` drawn in float64, stored float32 (each side quantizes
  them with its own packer);
* ``x``    ``N(0, 1)``, float32 for the tiny layer, bf16 (nearest-even) otherwise;
* ``q_norm``/``k_norm``  ``bf16(1 + 0.1 N(0, 1))`` (the pages fix no values);
* prior cache rows ``[0, cache_pos)`` ``N(0, 1)`` bf16, raw (not normed or
  rotated); slots at and past ``cache_pos`` hold ``fill`` (a bf16 bit pattern);
* batched lengths ``U{lo..hi}``; ``cache_pos = length - q_len``.

The workloads are the five shapes the layer is exercised on: a tiny correctness
layer, a 4B-class decode, a 2k-hidden speculative verify, a 9B-class batched
decode and a long-context mixed-width verify.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

# substream ids
(_X, _WQ, _WK, _WV, _WO, _QN, _KN, _CK, _CV, _LEN, _IN_LN, _POST_LN, _VQC, _VQS, _KQC,
 _KQS) = range(1, 17)


@dataclass(frozen=True)
class LayerSpec:
    name: str
    hidden: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    partial_rotary_factor: float
    rope_theta: float
    rms_eps: float
    bits: tuple          # (q, k, v, o)
    group: tuple         # (q, k, v, o)
    batch: int
    q_len: int
    x_dtype: str         # "f32" | "bf16"
    cache_pos: tuple | None = None      # fixed first-new-position per sequence
    length_range: tuple | None = None   # (lo, hi): final attended lengths U{lo..hi}
    seed: int = 0

    @property
    def gqa(self):
        return self.num_heads // self.num_kv_heads

    @property
    def n_q(self):           # doubled q_proj width: query and gate of every head
        return 2 * self.num_heads * self.head_dim

    @property
    def n_kv(self):
        return self.num_kv_heads * self.head_dim

    def positions(self) -> np.ndarray:
        """First new cache position of each sequence."""
        if self.cache_pos is not None:
            cp = np.asarray(self.cache_pos, np.int64)
            if cp.size == 1:
                cp = np.full(self.batch, int(cp[0]), np.int64)
            return cp.astype(np.int32)
        lo, hi = self.length_range
        rng = np.random.default_rng([self.seed, _LEN])
        lengths = rng.integers(lo, hi + 1, size=self.batch)
        return (lengths - self.q_len).astype(np.int32)

    def capacity(self) -> int:
        last = int(self.positions().max()) + self.q_len
        return ((last + 63) // 64) * 64

    def with_(self, **kw) -> "LayerSpec":
        return replace(self, **kw)


def _spec(name, hidden, H, Hk, d, bits, group, batch, q_len, x_dtype, **kw):
    return LayerSpec(name=name, hidden=hidden, num_heads=H, num_kv_heads=Hk, head_dim=d,
                     partial_rotary_factor=0.25, rope_theta=1e7, rms_eps=1e-6,
                     bits=bits, group=group, batch=batch, q_len=q_len, x_dtype=x_dtype, **kw)


WORKLOADS = {
    # tiny correctness layer: rotary 16, cache_pos 31
    "tiny": _spec("tiny", 256, 4, 2, 64, (4,) * 4, (64,) * 4, 1, 1, "f32", cache_pos=(31,)),
    # 4B-class decode: 8-bit g64, cache length 4096
    "decode_4b": _spec("decode_4b", 2560, 16, 4, 256, (8,) * 4, (64,) * 4, 1, 1, "bf16",
                       cache_pos=(4096 - 1,)),
    # speculative verify, 4 new rows, gqa 12, at cache_pos 46 and 2048
    "verify_2k_p46": _spec("verify_2k_p46", 2048, 24, 2, 256, (4,) * 4, (64,) * 4, 1, 4, "bf16",
                           cache_pos=(46,)),
    "verify_2k_p2048": _spec("verify_2k_p2048", 2048, 24, 2, 256, (4,) * 4, (64,) * 4, 1, 4,
                             "bf16", cache_pos=(2048,)),
    # the same verify at 32 new rows (a short prefill / wide speculative verify:
    # the head-chunk route's upper bound on q_len)
    "verify_2k_r32": _spec("verify_2k_r32", 2048, 24, 2, 256, (4,) * 4, (64,) * 4, 1, 32,
                           "bf16", cache_pos=(2048,)),
    # 9B-class batched decode: 32 sequences, lengths U{512..8192}
    "batched_9b": _spec("batched_9b", 4096, 32, 8, 256, (4,) * 4, (64,) * 4, 32, 1, "bf16",
                        length_range=(512, 8192)),
    # long-context verify, mixed widths: q/k/v 6-bit g128, o 3-bit g32, length 32768
    "long_verify_mixed": _spec("long_verify_mixed", 4096, 32, 8, 256, (6, 6, 6, 3),
                               (128, 128, 128, 32), 8, 4, "bf16", cache_pos=(32768 - 4,)),
}


# ------------------------------------------------------------------ helpers

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Nearest-even bf16 bit patterns of float32 values (NaN kept quiet)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    rounded = ((u + np.uint32(0x7FFF) + ((u >> 16) & np.uint32(1))) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        rounded = np.where(nan, np.uint16(0x7FC0), rounded)
    return rounded


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(seed, *ids, n, scale=1.0, dtype=np.float64):
    rng = np.random.default_rng([seed, *ids])
    if dtype == np.float64:
        return rng.standard_normal(n) * scale
    return rng.standard_normal(n, dtype=np.float32) * np.float32(scale)


# ----------------------------------------------------------------- tensors

def weights_f32(spec: LayerSpec):
    """Unquantized q/k/v/o weights, float32, [N][K] each."""
    s = spec.seed
    shapes = [(spec.n_q, spec.hidden), (spec.n_kv, spec.hidden), (spec.n_kv, spec.hidden),
              (spec.hidden, spec.num_heads * spec.head_dim)]
    out = []
    for sid, (n, k) in zip((_WQ, _WK, _WV, _WO), shapes):
        out.append(_normal(s, sid, n=n * k, scale=0.02).astype(np.float32).reshape(n, k))
    return out


def norm_weights_bf16(spec: LayerSpec):
    qn = f32_to_bf16_bits((1.0 + 0.1 * _normal(spec.seed, _QN, n=spec.head_dim)).astype(np.float32))
    kn = f32_to_bf16_bits((1.0 + 0.1 * _normal(spec.seed, _KN, n=spec.head_dim)).astype(np.float32))
    return qn, kn


def block_norm_weights_bf16(spec: LayerSpec):
    """input_ln and post_ln of the decoder block around the layer, bf16 bits
    [hidden], 1 + 0.1 N(0, 1) like the QK norms (no values are given)."""
    il = f32_to_bf16_bits((1.0 + 0.1 * _normal(spec.seed, _IN_LN, n=spec.hidden)).astype(np.float32))
    pl = f32_to_bf16_bits((1.0 + 0.1 * _normal(spec.seed, _POST_LN, n=spec.hidden)).astype(np.float32))
    return il, pl


def layer_input(spec: LayerSpec, step: int = 0):
    """x [B][R][hidden]: float32 array for f32 layers, bf16 bits for bf16 layers.
    ``step`` selects an independent draw (successive steps of one layer)."""
    n = spec.batch * spec.q_len * spec.hidden
    v = _normal(spec.seed, _X, step, n=n).astype(np.float32).reshape(spec.batch, spec.q_len,
                                                                     spec.hidden)
    return v if spec.x_dtype == "f32" else f32_to_bf16_bits(v)


def x_values(spec: LayerSpec, x: np.ndarray) -> np.ndarray:
    """The exact float64 values an x array stands for."""
    if spec.x_dtype == "f32":
        return np.asarray(x, np.float64)
    return bf16_bits_to_f32(x).astype(np.float64)


def cache_sequence(spec: LayerSpec, b: int, pos: int, capacity: int, fill: int = 0):
    """Prior K and V of sequence b: [Hk][capacity][d] bf16 bits."""
    Hk, d = spec.num_kv_heads, spec.head_dim
    k = np.full((Hk, capacity, d), fill, np.uint16)
    v = np.full((Hk, capacity, d), fill, np.uint16)
    for kh in range(Hk):
        k[kh, :pos] = f32_to_bf16_bits(
            _normal(spec.seed, _CK, b, kh, n=pos * d, dtype=np.float32)).reshape(pos, d)
        v[kh, :pos] = f32_to_bf16_bits(
            _normal(spec.seed, _CV, b, kh, n=pos * d, dtype=np.float32)).reshape(pos, d)
    return k, v


def cache(spec: LayerSpec, capacity: int | None = None, fill: int = 0, batches=None):
    """Prior caches [B'][Hk][capacity][d] bf16 bits for the sequences in ``batches``
    (all by default)."""
    cap = capacity or spec.capacity()
    pos = spec.positions()
    idx = range(spec.batch) if batches is None else list(batches)
    ks, vs = [], []
    for b in idx:
        k, v = cache_sequence(spec, b, int(pos[b]), cap, fill)
        ks.append(k)
        vs.append(v)
    return np.stack(ks), np.stack(vs)


def turbo4v_cache(spec: LayerSpec, capacity: int | None = None, stale_code: int = 0xFF,
                  stale_scale: int = 0x7F, batches=None, plane: str = "v"):
    """Prior Bf16KTurbo4V V planes for the sequences in ``batches``: codes
    [B'][Hk][cap][d/2] uint8 (uniform random nibbles) and E4M3 scales
    [B'][Hk][cap][d/16] uint8, uniform over the bytes 0x30..0x3F (0.5 to
    1.875, the scale of a unit-variance group) for positions < cache_pos;
    every later slot holds ``stale_code`` / ``stale_scale`` (0x7F is an E4M3
    NaN, so a kernel that reads a stale slot shows it).  Random bytes only:
    no quantizer arithmetic here.  plane="k" draws the K planes of a symmetric
    Turbo4 cache from their own substreams."""
    ic, isc = (_VQC, _VQS) if plane == "v" else (_KQC, _KQS)
    cap = capacity or spec.capacity()
    pos = spec.positions()
    Hk, d = spec.num_kv_heads, spec.head_dim
    idx = range(spec.batch) if batches is None else list(batches)
    cs, ss = [], []
    for b in idx:
        p = int(pos[b])
        c = np.full((Hk, cap, d // 2), stale_code, np.uint8)
        sc = np.full((Hk, cap, d // 16), stale_scale, np.uint8)
        for kh in range(Hk):
            rng = np.random.default_rng([spec.seed, ic, b, kh])
            c[kh, :p] = rng.integers(0, 256, size=(p, d // 2), dtype=np.uint8)
            rng = np.random.default_rng([spec.seed, isc, b, kh])
            sc[kh, :p] = rng.integers(0x30, 0x40, size=(p, d // 16), dtype=np.uint8)
        cs.append(c)
        ss.append(sc)
    return np.stack(cs), np.stack(ss)
