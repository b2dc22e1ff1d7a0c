"""ctypes face of the float64 CPU oracle (``gattn_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` load this module.  The CUDA library never
imports it and shares no code with it.

Every function cites the page and section it restates; the C file carries the
readings taken where the pages are silent.  All weight inputs are the packed
interchange layout (LSB-first code bitstream per row, bf16 scales/biases
``[N][K/group]``) produced by the oracle's own quantizer.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gattn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

MUTATIONS = {
    "none": 0,
    "no_gate": 1,
    "rotate_all": 2,
    "pair_adjacent": 3,
    "gqa_modulo": 4,
    "freq_base_d": 5,
    "no_causal": 6,
    "split_alternate": 7,
    "no_knorm": 8,
    "no_bf16_cache": 9,
    "turbo_no_iwht": 10,
}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, IEEE semantics: no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
             "-Wall", "-Wextra", "-Wno-unused-parameter", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _declare(_lib)
    return _lib


_p = C.c_void_p
_i64 = C.c_int64
_i = C.c_int


class _OrcLayer(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("num_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("partial_rotary_factor", C.c_double),
                ("rope_theta", C.c_double), ("rms_eps", C.c_double),
                ("bits", C.c_int32 * 4), ("group", C.c_int32 * 4),
                ("head_chunk", C.c_int32), ("mutate", C.c_int32)]


class _OrcStepExt(C.Structure):
    _fields_ = [("v_codes", _p), ("v_scales", _p), ("k_codes", _p), ("k_scales", _p),
                ("mask", _p), ("mask_heads", C.c_int32),
                ("mask_row", _i64), ("mask_head", _i64), ("mask_batch", _i64),
                ("mask_len", C.c_int32)]


class _OrcWeights(C.Structure):
    _fields_ = [("packed", _p * 4), ("scales", _p * 4), ("biases", _p * 4),
                ("q_norm", _p), ("k_norm", _p)]


def _declare(L):
    L.orc_bf16_to_double.argtypes = [C.c_uint16]
    L.orc_bf16_to_double.restype = C.c_double
    L.orc_bf16_from_double.argtypes = [C.c_double]
    L.orc_bf16_from_double.restype = C.c_uint16
    L.orc_quantize_affine.argtypes = [_p, _i64, _i64, _i, _i, _p, _p, _p]
    L.orc_unpack_codes.argtypes = [_p, _i64, _i64, _i, _p]
    L.orc_dequantize.argtypes = [_p, _p, _p, _i64, _i64, _i, _i, _p]
    L.orc_qmatvec.argtypes = [_p, _p, _p, _i64, _i64, _i, _i, _p, _i, _p]
    L.orc_rms_norm.argtypes = [_p, _i, _p, C.c_double, _p]
    L.orc_rms_norm.restype = None
    L.orc_rotary_dims.argtypes = [_i, C.c_double]
    L.orc_rope.argtypes = [_p, _i, _i, C.c_double, C.c_double]
    L.orc_rope.restype = None
    L.orc_head_chunk_plan.argtypes = [_i, _i, _i, _i, _p, _p, _i]
    L.orc_sdpa.argtypes = [_p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _p]
    L.orc_layer_step.argtypes = [C.POINTER(_OrcLayer), C.POINTER(_OrcWeights), _p, _p, _p, _i,
                                 _p, _i, _i, _p, _p, _p]
    L.orc_block_step.argtypes = [C.POINTER(_OrcLayer), C.POINTER(_OrcWeights), _p, _i, _p, _p,
                                 _p, _p, _i, _p, _i, _i, _p, _p]
    L.orc_e4m3_to_double.argtypes = [C.c_uint8]
    L.orc_e4m3_to_double.restype = C.c_double
    L.orc_e4m3_from_float.argtypes = [C.c_float]
    L.orc_e4m3_from_float.restype = C.c_uint8
    L.orc_turbo4_codebook.argtypes = [_p]
    L.orc_turbo4_codebook.restype = None
    L.orc_turbo4_tables_f32.argtypes = [_p, _p]
    L.orc_turbo4_tables_f32.restype = None
    L.orc_turbo4_quantize_rows.argtypes = [_p, _i64, _i, _p, _p]
    L.orc_turbo4_dequant_rows.argtypes = [_p, _p, _i64, _i, _i, _p]
    L.orc_layer_step_masked.argtypes = [C.POINTER(_OrcLayer), C.POINTER(_OrcWeights), _p, _p, _p,
                                        _i, _p, _i, _i, _p, _i, _i64, _i64, _i64, _p, _p, _p]
    L.orc_layer_step_ext.argtypes = [C.POINTER(_OrcLayer), C.POINTER(_OrcWeights), _p, _p, _p, _i,
                                     _p, _i, _i, C.POINTER(_OrcStepExt), _p, _p, _p]
    L.orc_block_step_ext.argtypes = [C.POINTER(_OrcLayer), C.POINTER(_OrcWeights), _p, _i, _p, _p,
                                     _p, _p, _i, _p, _i, _i, C.POINTER(_OrcStepExt), _p, _p]
    L.orc_layer_step_turbo4v.argtypes = [C.POINTER(_OrcLayer), C.POINTER(_OrcWeights), _p, _p, _p,
                                         _p, _i, _p, _i, _i, _p, _p, _p]


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


class MaskRouteError(ValueError):
    """A head-specific mask met the head-chunked attention route ([DS4#113]:
    the route hands the mask unchanged to every head chunk, so only a
    broadcast mask fits)."""


def _check(rc, what):
    if rc == 3:
        raise MaskRouteError(f"oracle {what}: a head-specific mask cannot take the head-chunk route")
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


# ------------------------------------------------------------------ scalars

def bf16_to_double(h: int) -> float:
    return lib().orc_bf16_to_double(int(h))


def bf16_from_double(x: float) -> int:
    return int(lib().orc_bf16_from_double(float(x)))


# ------------------------------------------------------------ quantization

def quantize_affine(w: np.ndarray, bits: int, group: int):
    """Affine group quantizer for synthetic weights ([TF#503] Option C: packed-row
    affine decoder, 2-8 bit, groups 32/64/128).  Returns (packed u32 [N][K*bits/32],
    scales bf16 [N][K/group], biases bf16 [N][K/group])."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    N, K = w.shape
    packed = np.zeros((N, K * bits // 32), np.uint32)
    scales = np.zeros((N, K // group), np.uint16)
    biases = np.zeros((N, K // group), np.uint16)
    _check(lib().orc_quantize_affine(_ptr(w), N, K, bits, group, _ptr(packed), _ptr(scales),
                                     _ptr(biases)), "quantize")
    return packed, scales, biases


def unpack_codes(packed: np.ndarray, N: int, K: int, bits: int) -> np.ndarray:
    codes = np.zeros((N, K), np.uint8)
    _check(lib().orc_unpack_codes(_ptr(np.ascontiguousarray(packed)), N, K, bits, _ptr(codes)),
           "unpack")
    return codes


def dequantize(packed, scales, biases, N, K, bits, group) -> np.ndarray:
    W = np.zeros((N, K), np.float64)
    _check(lib().orc_dequantize(_ptr(packed), _ptr(scales), _ptr(biases), N, K, bits, group,
                                _ptr(W)), "dequantize")
    return W


def qmatvec(packed, scales, biases, N, K, bits, group, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    y = np.zeros((x.shape[0], N), np.float64)
    _check(lib().orc_qmatvec(_ptr(packed), _ptr(scales), _ptr(biases), N, K, bits, group,
                             _ptr(x), x.shape[0], _ptr(y)), "qmatvec")
    return y


# ---------------------------------------------------------- norm / rotary

def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    w = np.ascontiguousarray(w, np.float64)
    y = np.zeros_like(x)
    lib().orc_rms_norm(_ptr(x), x.size, _ptr(w), float(eps), _ptr(y))
    return y


def rotary_dims(head_dim: int, prf: float) -> int:
    return int(lib().orc_rotary_dims(head_dim, float(prf)))


def rope(x: np.ndarray, rd: int, pos: float, theta: float) -> np.ndarray:
    y = np.array(x, np.float64, copy=True)
    lib().orc_rope(_ptr(y), y.size, rd, float(pos), float(theta))
    return y


def head_chunk_plan(q_len: int, num_heads: int, num_kv_heads: int, enabled: bool = True):
    cap = max(num_heads, 1)
    first = np.zeros(cap, np.int32)
    ln = np.zeros(cap, np.int32)
    n = lib().orc_head_chunk_plan(q_len, num_heads, num_kv_heads, int(bool(enabled)),
                                  _ptr(first), _ptr(ln), cap)
    if n < 0:
        raise ValueError("bad plan arguments")
    return list(zip(first[:n].tolist(), ln[:n].tolist()))


def sdpa(q, cache_k, cache_v, num_heads, h0, pos0):
    """q [n_heads][R][d]; cache [Hk][cap][d] bf16 bits; row r attends t <= pos0 + r."""
    q = np.ascontiguousarray(q, np.float64)
    n_heads, R, d = q.shape
    Hk, cap, d2 = cache_k.shape
    assert d2 == d
    out = np.zeros_like(q)
    _check(lib().orc_sdpa(_ptr(q), _ptr(np.ascontiguousarray(cache_k)),
                          _ptr(np.ascontiguousarray(cache_v)), num_heads, Hk, d, cap, h0,
                          n_heads, R, pos0, _ptr(out)), "sdpa")
    return out


# --------------------------------------------------------------- the layer

@dataclass
class OracleWeights:
    """Packed interchange weights for q, k, v, o plus bf16 q_norm/k_norm."""
    packed: list
    scales: list
    biases: list
    q_norm: np.ndarray
    k_norm: np.ndarray
    bits: list = field(default_factory=list)
    group: list = field(default_factory=list)


def _layer_structs(spec, weights: OracleWeights, head_chunk: bool, mutate: str):
    """The C structs of a layer; `keep` holds the arrays they point into."""
    L = _OrcLayer()
    L.hidden, L.num_heads, L.num_kv_heads, L.head_dim = (spec.hidden, spec.num_heads,
                                                         spec.num_kv_heads, spec.head_dim)
    L.partial_rotary_factor = float(np.float32(spec.partial_rotary_factor))
    L.rope_theta = float(np.float32(spec.rope_theta))
    L.rms_eps = float(np.float32(spec.rms_eps))
    for i in range(4):
        L.bits[i] = weights.bits[i]
        L.group[i] = weights.group[i]
    L.head_chunk = int(bool(head_chunk))
    L.mutate = MUTATIONS[mutate]
    Wt = _OrcWeights()
    keep = []
    for i in range(4):
        for arr, slot in ((weights.packed[i], Wt.packed), (weights.scales[i], Wt.scales),
                          (weights.biases[i], Wt.biases)):
            a = np.ascontiguousarray(arr)
            keep.append(a)
            slot[i] = _ptr(a)
    qn = np.ascontiguousarray(weights.q_norm, np.uint16)
    kn = np.ascontiguousarray(weights.k_norm, np.uint16)
    keep += [qn, kn]
    Wt.q_norm, Wt.k_norm = _ptr(qn), _ptr(kn)
    return L, Wt, keep


def layer_step(spec, weights: OracleWeights, x: np.ndarray, cache_k: np.ndarray,
               cache_v: np.ndarray, cache_pos: np.ndarray, head_chunk: bool = True,
               mutate: str = "none", taps: bool = False, mask: np.ndarray | None = None):
    """One gated full-attention layer step ([mlxd#99] Summary: doubled q_proj ->
    split query/gate -> o_proj(attn * sigmoid(gate)); [atlas-mod] KV append at
    cache_pos, attention over cache_pos + 1 per row).

    x: [B][R][hidden] float64 values; cache_k/v: [B][Hk][cap][d] bf16 bits,
    updated in place.  mask (optional, [DS4#113] broadcast / head-specific
    masks): uint8 [B][1 or H][R][T >= max(cache_pos) + R], nonzero = attend;
    it replaces the causal rule.  Returns out [B][R][hidden] (and the taps
    when asked)."""
    B, R, Hd = x.shape
    L, Wt, keep = _layer_structs(spec, weights, head_chunk, mutate)
    x = np.ascontiguousarray(x, np.float64)
    assert cache_k.flags["C_CONTIGUOUS"] and cache_v.flags["C_CONTIGUOUS"]
    cap = cache_k.shape[2]
    cp = np.ascontiguousarray(cache_pos, np.int32)
    out = np.zeros((B, R, Hd), np.float64)
    H, Hk, d = spec.num_heads, spec.num_kv_heads, spec.head_dim
    ty = np.zeros((B, R, 2 * H * d + 2 * Hk * d), np.float64) if taps else None
    ta = np.zeros((B, R, H, d), np.float64) if taps else None
    if mask is None:
        rc = lib().orc_layer_step(C.byref(L), C.byref(Wt), _ptr(x), _ptr(cache_k), _ptr(cache_v),
                                  cap, _ptr(cp), B, R, _ptr(out), _ptr(ty), _ptr(ta))
    else:
        mk = np.ascontiguousarray(mask, np.uint8)
        assert mk.ndim == 4 and mk.shape[0] == B and mk.shape[2] == R
        assert int(np.max(cp)) + R <= mk.shape[3]
        rc = lib().orc_layer_step_masked(C.byref(L), C.byref(Wt), _ptr(x), _ptr(cache_k),
                                         _ptr(cache_v), cap, _ptr(cp), B, R, _ptr(mk), mk.shape[1],
                                         mk.strides[2], mk.strides[1], mk.strides[0], _ptr(out),
                                         _ptr(ty), _ptr(ta))
    _check(rc, "layer_step")
    if taps:
        return out, ty, ta
    return out


# ------------------------------------------------- Turbo4 V cache ([atlas-mod])

def e4m3_to_double(b: int) -> float:
    """Value of an FP8 E4M3 byte ([atlas-mod] MetalKvDtype: FP8 group scales)."""
    return lib().orc_e4m3_to_double(int(b))


def e4m3_from_float(x: float) -> int:
    """Nearest E4M3 byte of an fp32 value (ties to even, saturating at 448)."""
    return int(lib().orc_e4m3_from_float(float(np.float32(x))))


def turbo4_codebook() -> np.ndarray:
    """The 16 Lloyd-Max levels of N(0, 1), ascending, float64 ([atlas-mod]
    MetalKvDtype::Turbo4: 4-bit Lloyd-Max codebook indices)."""
    c = np.zeros(16, np.float64)
    lib().orc_turbo4_codebook(_ptr(c))
    return c


def turbo4_tables_f32():
    """(levels fp32 [16], decision thresholds fp32 [15]) the quantizer uses."""
    lv = np.zeros(16, np.float32)
    th = np.zeros(15, np.float32)
    lib().orc_turbo4_tables_f32(_ptr(lv), _ptr(th))
    return lv, th


def turbo4_quantize_rows(v_bf16: np.ndarray):
    """bf16 bits [..., d] -> (codes uint8 [..., d/2], scales uint8 [..., d/16]):
    WHT rotation, per-16 RMS-normalized nearest Lloyd-Max level, matched-norm
    E4M3 scale; decisions in fp32 in the order the C source states."""
    v = np.ascontiguousarray(v_bf16, np.uint16)
    d = v.shape[-1]
    n = v.size // d
    codes = np.zeros(v.shape[:-1] + (d // 2,), np.uint8)
    scales = np.zeros(v.shape[:-1] + (d // 16,), np.uint8)
    _check(lib().orc_turbo4_quantize_rows(_ptr(v), n, d, _ptr(codes), _ptr(scales)),
           "turbo4_quantize_rows")
    return codes, scales


def turbo4_dequant_rows(codes: np.ndarray, scales: np.ndarray, mutate: str = "none") -> np.ndarray:
    """(codes [..., d/2], scales [..., d/16]) -> float64 rows [..., d] in the
    original basis (the inverse rotation applied)."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    d = codes.shape[-1] * 2
    n = codes.size // (d // 2)
    out = np.zeros(codes.shape[:-1] + (d,), np.float64)
    _check(lib().orc_turbo4_dequant_rows(_ptr(codes), _ptr(scales), n, d, MUTATIONS[mutate],
                                         _ptr(out)), "turbo4_dequant_rows")
    return out


def layer_step_turbo4v(spec, weights: OracleWeights, x: np.ndarray, cache_k: np.ndarray,
                       v_codes: np.ndarray, v_scales: np.ndarray, cache_pos: np.ndarray,
                       head_chunk: bool = True, mutate: str = "none", taps: bool = False):
    """layer_step over a Bf16KTurbo4V cache ([atlas-mod] MetalKvDtype,
    LayerKvCache): K bf16 [B][Hk][cap][d]; V codes [B][Hk][cap][d/2] and
    E4M3 scales [B][Hk][cap][d/16], all updated in place."""
    B, R, Hd = x.shape
    L, Wt, keep = _layer_structs(spec, weights, head_chunk, mutate)
    x = np.ascontiguousarray(x, np.float64)
    for a in (cache_k, v_codes, v_scales):
        assert a.flags["C_CONTIGUOUS"]
    cap = cache_k.shape[2]
    assert v_codes.dtype == np.uint8 and v_scales.dtype == np.uint8
    cp = np.ascontiguousarray(cache_pos, np.int32)
    out = np.zeros((B, R, Hd), np.float64)
    H, Hk, d = spec.num_heads, spec.num_kv_heads, spec.head_dim
    ty = np.zeros((B, R, 2 * H * d + 2 * Hk * d), np.float64) if taps else None
    ta = np.zeros((B, R, H, d), np.float64) if taps else None
    rc = lib().orc_layer_step_turbo4v(C.byref(L), C.byref(Wt), _ptr(x), _ptr(cache_k),
                                      _ptr(v_codes), _ptr(v_scales), cap, _ptr(cp), B, R,
                                      _ptr(out), _ptr(ty), _ptr(ta))
    _check(rc, "layer_step_turbo4v")
    if taps:
        return out, ty, ta
    return out


def _step_ext(turbo, mask, keep, turbo_k=None):
    """orc_step_ext for a Turbo4 V cache (codes, scales), the K planes of a
    symmetric Turbo4 cache, and/or a mask [B][1|H][R][T]."""
    e = _OrcStepExt()
    for planes, names in ((turbo, ("v_codes", "v_scales")), (turbo_k, ("k_codes", "k_scales"))):
        if planes is not None:
            codes, scales = planes
            assert codes.dtype == np.uint8 and scales.dtype == np.uint8
            assert codes.flags["C_CONTIGUOUS"] and scales.flags["C_CONTIGUOUS"]
            setattr(e, names[0], _ptr(codes))
            setattr(e, names[1], _ptr(scales))
    if mask is not None:
        mk = np.ascontiguousarray(mask, np.uint8)
        keep.append(mk)
        e.mask, e.mask_heads = _ptr(mk), mk.shape[1]
        e.mask_row, e.mask_head, e.mask_batch = mk.strides[2], mk.strides[1], mk.strides[0]
        e.mask_len = mk.shape[3]           # positions from T on are not attended
    return e


def layer_step_ext(spec, weights: OracleWeights, x: np.ndarray, cache_k, cache_v,
                   cache_pos: np.ndarray, turbo=None, mask=None, head_chunk: bool = True,
                   taps: bool = False, turbo_k=None):
    """layer_step with the optional parts together: turbo = (codes, scales) of a
    Bf16KTurbo4V cache (cache_v unused, may be None); turbo_k = the K planes of
    the symmetric Turbo4 cache ([atlas-mod] MetalKvDtype::Turbo4; needs turbo,
    cache_k unused); mask as in layer_step, except that its rows may be shorter
    than cache_pos + R: positions from T on are not attended (the library's
    mask rows of `positions` bytes).  Planes are updated in place."""
    B, R, Hd = x.shape
    L, Wt, keep = _layer_structs(spec, weights, head_chunk, "none")
    x = np.ascontiguousarray(x, np.float64)
    cp = np.ascontiguousarray(cache_pos, np.int32)
    e = _step_ext(turbo, mask, keep, turbo_k)
    cap = (turbo_k[0] if turbo_k is not None else cache_k).shape[2]
    out = np.zeros((B, R, Hd), np.float64)
    H, Hk, d = spec.num_heads, spec.num_kv_heads, spec.head_dim
    ty = np.zeros((B, R, 2 * H * d + 2 * Hk * d), np.float64) if taps else None
    ta = np.zeros((B, R, H, d), np.float64) if taps else None
    rc = lib().orc_layer_step_ext(C.byref(L), C.byref(Wt), _ptr(x), _ptr(cache_k), _ptr(cache_v),
                                  cap, _ptr(cp), B, R, C.byref(e), _ptr(out), _ptr(ty), _ptr(ta))
    _check(rc, "layer_step_ext")
    return (out, ty, ta) if taps else out


def block_step(spec, weights: OracleWeights, x: np.ndarray, input_ln: np.ndarray,
               post_ln, cache_k: np.ndarray, cache_v, cache_pos: np.ndarray,
               head_chunk: bool = True, turbo=None, mask=None):
    """The decoder block around the layer ([atlas-mod] forward_full_attention:
    input RMSNorm -> layer -> residual add -> post-attention RMSNorm): returns
    out = x + layer(RMSNorm(x) * input_ln) and, when post_ln is given,
    RMSNorm(bf16(out)) * post_ln (else None).  The normed input h is rounded
    to bf16 for a bf16 layer (spec.x_dtype), kept exact for an fp32 one.
    input_ln / post_ln: bf16 bits [hidden]; caches as in layer_step (updated
    in place)."""
    B, R, Hd = x.shape
    L, Wt, keep = _layer_structs(spec, weights, head_chunk, "none")
    x = np.ascontiguousarray(x, np.float64)
    iw = np.ascontiguousarray(input_ln, np.uint16)
    pw = None if post_ln is None else np.ascontiguousarray(post_ln, np.uint16)
    assert cache_k.flags["C_CONTIGUOUS"]
    assert turbo is not None or cache_v.flags["C_CONTIGUOUS"]
    e = _step_ext(turbo, mask, keep)
    cp = np.ascontiguousarray(cache_pos, np.int32)
    out = np.zeros((B, R, Hd), np.float64)
    on = np.zeros((B, R, Hd), np.float64) if pw is not None else None
    rc = lib().orc_block_step_ext(C.byref(L), C.byref(Wt), _ptr(x),
                                  1 if spec.x_dtype == "bf16" else 0, _ptr(iw), _ptr(pw),
                                  _ptr(cache_k), _ptr(cache_v), cache_k.shape[2], _ptr(cp), B, R,
                                  C.byref(e), _ptr(out), _ptr(on))
    _check(rc, "block_step")
    return out, on
