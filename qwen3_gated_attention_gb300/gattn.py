"""ctypes binding of libgattn.so (C ABI in include/gattn.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Device buffers are passed as integer addresses (e.g. a torch
tensor's ``data_ptr()``), streams as integer ``cudaStream_t`` handles.  There is
no fallback: if the shared library is missing this module raises on import of
the library.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgattn.so")

GATTN_OK = 0
STATUS_NAMES = {0: "GATTN_OK", 1: "GATTN_E_INVALID_ARG", 2: "GATTN_E_UNSUPPORTED",
                3: "GATTN_E_CUDA", 4: "GATTN_E_DEVICE_RANGE", 5: "GATTN_E_STATE",
                6: "GATTN_E_DEVICE_TIMEOUT"}
DTYPE_F32, DTYPE_BF16 = 0, 1
PROJ_Q, PROJ_K, PROJ_V, PROJ_O = 0, 1, 2, 3
# kernels of a step (gattn_layer_step_kernels)
KERNEL_NAMES = {1: "xprep", 2: "proj_qkv", 3: "attn", 4: "merge", 5: "proj_o", 6: "postnorm"}

# every symbol include/gattn.h declares
EXPORTS = (
    "gattn_cfg_validate", "gattn_rotary_dims", "gattn_layer_create", "gattn_layer_set_weights",
    "gattn_kv_register", "gattn_layer_step", "gattn_layer_poll_status", "gattn_layer_set_taps",
    "gattn_layer_destroy", "gattn_kv_destroy", "gattn_last_error", "gattn_pack_affine_host",
    "gattn_unpack_codes_device", "gattn_layer_dequant_device", "gattn_head_chunk_plan",
    "gattn_layer_launches_per_step", "gattn_layer_set_events", "gattn_layer_dequant_device_static",
    "gattn_layer_step_block", "gattn_kv_register_turbo4v",
    "gattn_turbo4_codebook", "gattn_turbo4_quantize_device", "gattn_layer_set_mask",
    "gattn_kv_register_turbo4", "gattn_layer_step_kernels", "gattn_layer_set_test_wait",
    "gattn_layer_step_host",
)


class GattnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class gattn_cfg(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("num_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("partial_rotary_factor", C.c_float),
                ("rope_theta", C.c_float), ("rms_eps", C.c_float), ("bits", C.c_int32),
                ("group_size", C.c_int32), ("proj_bits", C.c_int32 * 4),
                ("proj_group", C.c_int32 * 4), ("x_dtype", C.c_int32), ("max_batch", C.c_int32),
                ("max_q_len", C.c_int32), ("head_chunk", C.c_int32)]


class gattn_proj(C.Structure):
    _fields_ = [("packed", C.c_void_p), ("scales", C.c_void_p), ("biases", C.c_void_p)]


class gattn_weights(C.Structure):
    _fields_ = [("proj", gattn_proj * 4), ("q_norm", C.c_void_p), ("k_norm", C.c_void_p)]


class gattn_kv_desc(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("batch", C.c_int32),
                ("capacity", C.c_int32), ("stride_token", C.c_int64), ("stride_head", C.c_int64),
                ("stride_batch", C.c_int64)]


class gattn_kv_turbo4v_desc(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v_codes", C.c_void_p), ("v_scales", C.c_void_p),
                ("batch", C.c_int32), ("capacity", C.c_int32),
                ("k_stride_token", C.c_int64), ("k_stride_head", C.c_int64),
                ("k_stride_batch", C.c_int64), ("code_stride_head", C.c_int64),
                ("code_stride_batch", C.c_int64), ("scale_stride_head", C.c_int64),
                ("scale_stride_batch", C.c_int64)]


class gattn_kv_turbo4_desc(C.Structure):
    _fields_ = [("k_codes", C.c_void_p), ("k_scales", C.c_void_p), ("v_codes", C.c_void_p),
                ("v_scales", C.c_void_p), ("batch", C.c_int32), ("capacity", C.c_int32),
                ("code_stride_head", C.c_int64), ("code_stride_batch", C.c_int64),
                ("scale_stride_head", C.c_int64), ("scale_stride_batch", C.c_int64)]


class gattn_mask(C.Structure):
    _fields_ = [("mask", C.c_void_p), ("heads", C.c_int32), ("positions", C.c_int32),
                ("stride_row", C.c_int64), ("stride_head", C.c_int64), ("stride_batch", C.c_int64)]


class gattn_taps(C.Structure):
    _fields_ = [("y", C.c_void_p), ("attn", C.c_void_p)]


_lib = None


def lib():
    """Load libgattn.so once (raises OSError when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: build it with "
                          "`python -m qwen3_gated_attention_gb300.build`")
        L = C.CDLL(LIB_PATH)
        p, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
        L.gattn_cfg_validate.argtypes = [C.POINTER(gattn_cfg)]
        L.gattn_rotary_dims.argtypes = [C.POINTER(gattn_cfg)]
        L.gattn_rotary_dims.restype = i32
        L.gattn_layer_create.argtypes = [C.POINTER(gattn_cfg), C.POINTER(p)]
        L.gattn_layer_set_weights.argtypes = [p, C.POINTER(gattn_weights), p]
        L.gattn_kv_register.argtypes = [p, C.POINTER(gattn_kv_desc), C.POINTER(p)]
        L.gattn_layer_step.argtypes = [p, p, p, p, i32, i32, p, p]
        L.gattn_layer_poll_status.argtypes = [p, p]
        L.gattn_layer_set_taps.argtypes = [p, C.POINTER(gattn_taps)]
        L.gattn_layer_destroy.argtypes = [p]
        L.gattn_layer_destroy.restype = None
        L.gattn_kv_destroy.argtypes = [p]
        L.gattn_kv_destroy.restype = None
        L.gattn_last_error.restype = C.c_char_p
        L.gattn_pack_affine_host.argtypes = [p, i64, i64, i32, i32, p, p, p]
        L.gattn_unpack_codes_device.argtypes = [p, i64, i64, i32, p, p]
        L.gattn_layer_dequant_device.argtypes = [p, i32, p, p]
        L.gattn_layer_dequant_device_static.argtypes = [p, i32, p, p]
        L.gattn_head_chunk_plan.argtypes = [i32, i32, i32, i32, p, p, i32]
        L.gattn_head_chunk_plan.restype = i32
        L.gattn_layer_launches_per_step.argtypes = [p]
        L.gattn_layer_launches_per_step.restype = i32
        L.gattn_layer_step_kernels.argtypes = [p, p, i32]
        L.gattn_layer_step_kernels.restype = i32
        L.gattn_layer_set_events.argtypes = [p, p, i32]
        L.gattn_layer_step_block.argtypes = [p, p, p, p, i32, i32, p, p, p, p, p]
        L.gattn_kv_register_turbo4v.argtypes = [p, C.POINTER(gattn_kv_turbo4v_desc), C.POINTER(p)]
        L.gattn_turbo4_codebook.argtypes = [p, p]
        L.gattn_turbo4_quantize_device.argtypes = [p, i64, i32, p, p, p]
        L.gattn_layer_set_mask.argtypes = [p, C.POINTER(gattn_mask)]
        L.gattn_kv_register_turbo4.argtypes = [p, C.POINTER(gattn_kv_turbo4_desc), C.POINTER(p)]
        L.gattn_layer_set_test_wait.argtypes = [p, i64, i32]
        L.gattn_layer_step_host.argtypes = [p, p, p, p, i32, i32, p, p]
        for name in ("gattn_cfg_validate", "gattn_layer_create", "gattn_layer_set_weights",
                     "gattn_kv_register", "gattn_layer_step", "gattn_layer_poll_status",
                     "gattn_layer_set_taps", "gattn_pack_affine_host", "gattn_unpack_codes_device",
                     "gattn_layer_dequant_device", "gattn_layer_set_events",
                     "gattn_layer_dequant_device_static",
                     "gattn_layer_step_block", "gattn_kv_register_turbo4v",
                     "gattn_turbo4_codebook", "gattn_turbo4_quantize_device",
                     "gattn_layer_set_mask", "gattn_kv_register_turbo4",
                     "gattn_layer_set_test_wait", "gattn_layer_step_host"):
            getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


def last_error() -> str:
    return lib().gattn_last_error().decode()


def _check(status: int):
    if status != GATTN_OK:
        raise GattnError(status, last_error())


# ------------------------------------------------------------------- cfg

def make_cfg(hidden, num_heads, num_kv_heads, head_dim, partial_rotary_factor, rope_theta, rms_eps,
             bits, group, x_dtype="bf16", max_batch=1, max_q_len=1, head_chunk=True) -> gattn_cfg:
    """bits/group: an int (all projections) or a 4-tuple (q, k, v, o)."""
    c = gattn_cfg()
    c.hidden, c.num_heads, c.num_kv_heads, c.head_dim = hidden, num_heads, num_kv_heads, head_dim
    c.partial_rotary_factor, c.rope_theta, c.rms_eps = partial_rotary_factor, rope_theta, rms_eps
    bt = tuple(bits) if isinstance(bits, (tuple, list)) else (bits,) * 4
    gt = tuple(group) if isinstance(group, (tuple, list)) else (group,) * 4
    c.bits, c.group_size = bt[0], gt[0]
    for i in range(4):
        c.proj_bits[i] = bt[i]
        c.proj_group[i] = gt[i]
    c.x_dtype = DTYPE_F32 if x_dtype == "f32" else DTYPE_BF16
    c.max_batch, c.max_q_len, c.head_chunk = max_batch, max_q_len, int(bool(head_chunk))
    return c


def cfg_validate(cfg: gattn_cfg) -> None:
    _check(lib().gattn_cfg_validate(C.byref(cfg)))


def rotary_dims(cfg: gattn_cfg) -> int:
    return int(lib().gattn_rotary_dims(C.byref(cfg)))


# ------------------------------------------------------------------ layer

def layer_create(cfg: gattn_cfg) -> int:
    h = C.c_void_p()
    _check(lib().gattn_layer_create(C.byref(cfg), C.byref(h)))
    return h.value


def layer_set_weights(layer: int, proj_ptrs, q_norm: int, k_norm: int, stream: int = 0) -> None:
    """proj_ptrs: four (packed, scales, biases) device-address triples (q, k, v, o)."""
    w = gattn_weights()
    for i, (pk, sc, bi) in enumerate(proj_ptrs):
        w.proj[i].packed, w.proj[i].scales, w.proj[i].biases = pk, sc, bi
    w.q_norm, w.k_norm = q_norm, k_norm
    _check(lib().gattn_layer_set_weights(layer, C.byref(w), stream))


def kv_register(layer: int, k: int, v: int, batch: int, capacity: int, stride_token: int,
                stride_head: int, stride_batch: int) -> int:
    d = gattn_kv_desc(k, v, batch, capacity, stride_token, stride_head, stride_batch)
    h = C.c_void_p()
    _check(lib().gattn_kv_register(layer, C.byref(d), C.byref(h)))
    return h.value


def kv_register_turbo4v(layer: int, k: int, v_codes: int, v_scales: int, batch: int,
                        capacity: int, k_strides, code_strides, scale_strides) -> int:
    """Register a Bf16KTurbo4V cache.  k_strides: (token, head, batch) in
    elements; code_strides / scale_strides: (head, batch) in bytes."""
    d = gattn_kv_turbo4v_desc(k, v_codes, v_scales, batch, capacity, *k_strides, *code_strides,
                              *scale_strides)
    h = C.c_void_p()
    _check(lib().gattn_kv_register_turbo4v(layer, C.byref(d), C.byref(h)))
    return h.value


def layer_set_mask(layer: int, mask: int | None, heads: int = 1, positions: int = 0,
                   strides=(0, 0, 0)) -> None:
    """Attention mask of the following steps (device bytes; None clears it).
    strides: (row, head, batch) in bytes."""
    if not mask:
        _check(lib().gattn_layer_set_mask(layer, None))
        return
    m = gattn_mask(mask, heads, positions, *strides)
    _check(lib().gattn_layer_set_mask(layer, C.byref(m)))


def kv_register_turbo4(layer: int, k_codes: int, k_scales: int, v_codes: int, v_scales: int,
                       batch: int, capacity: int, code_strides, scale_strides) -> int:
    """Register a symmetric Turbo4 cache; strides (head, batch) in bytes, shared by K and V."""
    d = gattn_kv_turbo4_desc(k_codes, k_scales, v_codes, v_scales, batch, capacity,
                             *code_strides, *scale_strides)
    h = C.c_void_p()
    _check(lib().gattn_kv_register_turbo4(layer, C.byref(d), C.byref(h)))
    return h.value


def turbo4_codebook():
    """(levels fp32 [16], thresholds fp32 [15]) as the kernels use them (host call)."""
    import numpy as np
    lv = np.zeros(16, np.float32)
    th = np.zeros(15, np.float32)
    _check(lib().gattn_turbo4_codebook(lv.ctypes.data, th.ctypes.data))
    return lv, th


def turbo4_quantize_device(v: int, rows: int, d: int, codes: int, scales: int,
                           stream: int = 0) -> None:
    """Quantize bf16 rows (device) into Turbo4 codes and E4M3 scales (device)."""
    _check(lib().gattn_turbo4_quantize_device(v, rows, d, codes, scales, stream))


def layer_step(layer: int, x: int, kv: int, cache_pos: int, batch: int, q_len: int, out: int,
               stream: int = 0) -> None:
    _check(lib().gattn_layer_step(layer, x, kv, cache_pos, batch, q_len, out, stream))


def layer_step_host(layer: int, x_host: int, kv: int, cache_pos_host: int, batch: int,
                    q_len: int, out_host: int, stream: int = 0) -> None:
    """gattn_layer_step from host buffers (x, cache_pos in; out back), enqueued
    on the stream; out_host holds the result once the stream has reached it."""
    _check(lib().gattn_layer_step_host(layer, x_host, kv, cache_pos_host, batch, q_len, out_host,
                                       stream))


def layer_poll_status(layer: int, stream: int = 0) -> None:
    _check(lib().gattn_layer_poll_status(layer, stream))


def layer_poll_status_code(layer: int, stream: int = 0) -> int:
    return int(lib().gattn_layer_poll_status(layer, stream))


def layer_set_taps(layer: int, y: int | None = None, attn: int | None = None) -> None:
    t = gattn_taps(y, attn)
    _check(lib().gattn_layer_set_taps(layer, C.byref(t)))


def layer_destroy(layer: int) -> None:
    if layer:
        lib().gattn_layer_destroy(layer)


def kv_destroy(kv: int) -> None:
    if kv:
        lib().gattn_kv_destroy(kv)


def layer_launches_per_step(layer: int) -> int:
    return int(lib().gattn_layer_launches_per_step(layer))


def layer_step_kernels(layer: int) -> list:
    """Names of the kernels the layer's last step launched, in order."""
    arr = (C.c_int32 * 8)()
    n = int(lib().gattn_layer_step_kernels(layer, C.addressof(arr), 8))
    if n < 0:
        raise GattnError(1, "bad arguments")
    return [KERNEL_NAMES.get(int(arr[i]), "?") for i in range(min(n, 8))]


def layer_step_block(layer: int, x: int, kv: int, cache_pos: int, batch: int, q_len: int,
                     input_ln: int, post_ln: int | None, out: int, out_normed: int | None,
                     stream: int | None = None) -> None:
    """Decoder-block step: out = x + layer(RMSNorm(x) * input_ln); out_normed =
    RMSNorm(out) * post_ln when given (device pointers)."""
    _check(lib().gattn_layer_step_block(layer, x, kv, cache_pos, batch, q_len, input_ln, post_ln,
                                        out, out_normed, stream))


def layer_set_events(layer: int, events) -> None:
    """events: sequence of cudaEvent_t handles (ints), or empty to turn off."""
    arr = (C.c_void_p * max(1, len(events)))(*events)
    _check(lib().gattn_layer_set_events(layer, C.addressof(arr) if events else None, len(events)))


def layer_set_test_wait(layer: int, wait_limit_ns: int = 0, withhold_stage: bool = False) -> None:
    """Failure-detection test hook: the bound of the projection kernels' device
    waits (0 restores the default) and whether CTA 0 of the q|k|v projection
    withholds its last weight stage so that one wait runs out."""
    _check(lib().gattn_layer_set_test_wait(layer, int(wait_limit_ns), 1 if withhold_stage else 0))


# ------------------------------------------------------------ host helpers

def pack_affine_host(w: np.ndarray, bits: int, group: int):
    """float32 [N][K] -> (packed u32 [N][K*bits/32], scales bf16 [N][K/group], biases)."""
    w = np.ascontiguousarray(w, np.float32)
    N, K = w.shape
    packed = np.zeros((N, K * bits // 32), np.uint32)
    scales = np.zeros((N, K // group), np.uint16)
    biases = np.zeros((N, K // group), np.uint16)
    _check(lib().gattn_pack_affine_host(w.ctypes.data, N, K, bits, group, packed.ctypes.data,
                                        scales.ctypes.data, biases.ctypes.data))
    return packed, scales, biases


def unpack_codes_device(packed: int, N: int, K: int, bits: int, codes: int, stream: int = 0):
    _check(lib().gattn_unpack_codes_device(packed, N, K, bits, codes, stream))


def layer_dequant_device(layer: int, proj: int, w: int, stream: int = 0):
    _check(lib().gattn_layer_dequant_device(layer, proj, w, stream))


def layer_dequant_device_static(layer: int, proj: int, w: int, stream: int = 0):
    """Like layer_dequant_device but allocation-free (fixed device staging array,
    no synchronization); see include/gattn.h for the size limit."""
    _check(lib().gattn_layer_dequant_device_static(layer, proj, w, stream))


def head_chunk_plan(q_len: int, num_heads: int, num_kv_heads: int, enabled: bool = True):
    cap = max(1, num_heads)
    first = (C.c_int32 * cap)()
    ln = (C.c_int32 * cap)()
    n = lib().gattn_head_chunk_plan(q_len, num_heads, num_kv_heads, int(bool(enabled)),
                                    C.addressof(first), C.addressof(ln), cap)
    if n < 0:
        raise GattnError(1, "bad plan arguments")
    return [(first[i], ln[i]) for i in range(min(n, cap))]
