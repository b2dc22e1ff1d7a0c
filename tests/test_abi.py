"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, validates configurations, and its host-side helpers (packer, rotary
dims, head-chunk plan) agree with the oracle."""
import os
import re

import numpy as np
import pytest

import oracle as orc
from qwen3_gated_attention_gb300 import gattn, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from qwen3_gated_attention_gb300 import build
    build.build()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "gattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gattn_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    decl = _declared_functions()
    assert len(decl) >= 16
    assert sorted(gattn.EXPORTS) == decl
    L = gattn.lib()
    for name in decl:
        assert hasattr(L, name), name


def _cfg(spec, **kw):
    args = dict(x_dtype=spec.x_dtype, max_batch=spec.batch, max_q_len=spec.q_len)
    args.update(kw)
    return gattn.make_cfg(spec.hidden, spec.num_heads, spec.num_kv_heads, spec.head_dim,
                          spec.partial_rotary_factor, spec.rope_theta, spec.rms_eps,
                          tuple(spec.bits), tuple(spec.group), **args)


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_configs_are_admitted(name):
    spec = synth.WORKLOADS[name]
    c = _cfg(spec)
    gattn.cfg_validate(c)
    assert gattn.rotary_dims(c) == orc.rotary_dims(spec.head_dim, float(np.float32(spec.partial_rotary_factor)))


@pytest.mark.parametrize("change,status", [
    (dict(partial_rotary_factor=0.0), 1),
    (dict(partial_rotary_factor=1.5), 1),
    (dict(partial_rotary_factor=0.01), 1),       # trunc(64*0.01) = 0 rotary dims
    (dict(partial_rotary_factor=3 / 64), 1),     # 3 rotary dims: odd
    (dict(num_kv_heads=3), 1),                   # 4 % 3
    (dict(bits=7), 1),
    (dict(group=16), 1),
    (dict(head_dim=96), 2),
    (dict(hidden=200), 2),
    (dict(max_batch=64), 2),
    (dict(bits=(4, 8, 4, 4)), 2),                # q/k/v widths must match
    # sizes past the kernels' 32-bit indexes, and products of fields that would
    # overflow a 32-bit int if they were formed before the bounds are checked
    (dict(hidden=16384 + 128), 2),
    (dict(num_heads=2 ** 23, num_kv_heads=2 ** 23, head_dim=256), 2),
    (dict(max_batch=2, max_q_len=2 ** 31 - 1), 2),
    (dict(max_batch=2 ** 30, max_q_len=2 ** 30), 2),
    (dict(max_batch=1, max_q_len=33), 2),
])
def test_inadmissible_configs_are_rejected(change, status):
    spec = synth.WORKLOADS["tiny"]
    kw = dict(hidden=spec.hidden, num_heads=spec.num_heads, num_kv_heads=spec.num_kv_heads,
              head_dim=spec.head_dim, partial_rotary_factor=spec.partial_rotary_factor,
              rope_theta=spec.rope_theta, rms_eps=spec.rms_eps, bits=spec.bits, group=spec.group)
    extra = {}
    for k, v in change.items():
        if k in kw:
            kw[k] = v
        else:
            extra[k] = v
    c = gattn.make_cfg(**kw, **extra)
    with pytest.raises(gattn.GattnError) as ei:
        gattn.cfg_validate(c)
    assert ei.value.status == status
    assert gattn.last_error()


@pytest.mark.parametrize("bits,group", [(2, 32), (3, 32), (4, 64), (5, 128), (6, 128), (8, 64)])
def test_host_packer_matches_oracle_packer_bit_exactly(bits, group):
    rng = np.random.default_rng(bits)
    w = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    w[5, :group] = 0.03125                      # constant group (scale 0)
    w[6] *= 1e-30                               # tiny values: bf16 subnormal scales
    w[7] *= 1e30
    a = gattn.pack_affine_host(w, bits, group)
    b = orc.quantize_affine(w.astype(np.float64), bits, group)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_host_packer_on_a_workload_matrix():
    spec = synth.WORKLOADS["tiny"]
    for i, w in enumerate(synth.weights_f32(spec)):
        a = gattn.pack_affine_host(w, spec.bits[i], spec.group[i])
        b = orc.quantize_affine(w.astype(np.float64), spec.bits[i], spec.group[i])
        assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_head_chunk_plan_matches_oracle():
    for q_len in range(1, 34):
        for gqa in (1, 2, 3, 4, 5, 8, 12, 16, 31, 64):
            for Hk in (1, 2, 4):
                for on in (True, False):
                    H = gqa * Hk
                    assert gattn.head_chunk_plan(q_len, H, Hk, on) == \
                        orc.head_chunk_plan(q_len, H, Hk, on)


def test_step_rejects_null_arguments_without_a_gpu():
    with pytest.raises(gattn.GattnError) as ei:
        gattn.layer_step(0, 0, 0, 0, 1, 1, 0, 0)
    assert ei.value.status == 1


def test_turbo4_codebook_matches_oracle_bit_exactly():
    """The library derives its Turbo4 tables (Lloyd-Max levels of N(0, 1) and
    the thresholds between them) by its own iteration; the fp32 values the
    kernels decide with equal the oracle's bit for bit, so both sides take the
    same quantization decisions."""
    lv, th = gattn.turbo4_codebook()
    olv, oth = orc.turbo4_tables_f32()
    assert np.array_equal(lv.view(np.uint32), olv.view(np.uint32))
    assert np.array_equal(th.view(np.uint32), oth.view(np.uint32))
    assert th[7] == 0.0 and np.array_equal(lv, -lv[::-1])


def test_turbo4_quantize_rejects_bad_arguments_without_a_gpu():
    with pytest.raises(gattn.GattnError) as e:
        gattn.turbo4_quantize_device(0, 4, 96, 0, 0)
    assert e.value.status == 1                                  # GATTN_E_INVALID_ARG
    with pytest.raises(gattn.GattnError):
        gattn.turbo4_quantize_device(0, 4, 128, 0, 0)          # NULL pointers


def test_documented_errors_that_need_no_gpu():
    """Every entry point's argument errors as the header states them, taken
    before any CUDA call, so they hold on a machine without a GPU."""
    import ctypes as C
    L = gattn.lib()
    null = None

    def status(rc, want):
        assert rc == want, (rc, want)
        assert gattn.last_error()

    # create refuses an inadmissible config with the validator's status and no handle
    spec = synth.WORKLOADS["tiny"]
    bad = gattn.make_cfg(spec.hidden, spec.num_heads, spec.num_kv_heads, 96,
                         spec.partial_rotary_factor, spec.rope_theta, spec.rms_eps,
                         tuple(spec.bits), tuple(spec.group))
    h = C.c_void_p(1)
    status(L.gattn_layer_create(C.byref(bad), C.byref(h)), 2)
    assert h.value is None
    status(L.gattn_layer_create(C.byref(_cfg(spec)), null), 1)
    # NULL handles
    status(L.gattn_layer_set_weights(null, null, null), 1)
    status(L.gattn_kv_register(null, null, null), 1)
    status(L.gattn_kv_register_turbo4v(null, null, null), 1)
    status(L.gattn_kv_register_turbo4(null, null, null), 1)
    status(L.gattn_layer_poll_status(null, null), 1)
    status(L.gattn_layer_set_taps(null, null), 1)
    status(L.gattn_layer_set_mask(null, null), 1)
    status(L.gattn_layer_set_events(null, null, 0), 1)
    status(L.gattn_layer_step_block(null, null, null, null, 1, 1, null, null, null, null, null), 1)
    status(L.gattn_layer_dequant_device(null, 0, null, null), 1)
    status(L.gattn_layer_dequant_device_static(null, 0, null, null), 1)
    status(L.gattn_unpack_codes_device(null, 1, 32, 4, null, null), 1)
    status(L.gattn_turbo4_codebook(null, null), 1)
    status(L.gattn_pack_affine_host(null, 4, 64, 4, 64, null, null, null), 1)
    # the plain-value queries
    assert L.gattn_rotary_dims(null) == -1
    assert L.gattn_layer_launches_per_step(null) == -1
    first = (C.c_int32 * 4)()
    assert L.gattn_head_chunk_plan(0, 4, 2, 1, first, first, 4) == -1
    assert L.gattn_head_chunk_plan(4, 6, 4, 1, first, first, 4) == -1      # 6 % 4
    assert L.gattn_head_chunk_plan(4, 4, 2, 1, null, null, 4) == -1
    assert L.gattn_head_chunk_plan(4, 4, 2, 1, null, null, 0) == 2         # count only
    # destroy(NULL) is a no-op
    L.gattn_layer_destroy(null)
    L.gattn_kv_destroy(null)
