"""The built rows together on the GPU against the oracle: a Bf16KTurbo4V cache
with an attention mask, and the decoder-block step over a Turbo4 cache and
with a mask."""
import numpy as np
import pytest
import torch

import oracle as orc
from qwen3_gated_attention_gb300 import synth
from qwen3_gated_attention_gb300.device import DeviceLayer, x_to_device
from tests import refs
from tests.cases import make_case
from tests.test_gpu_block import _clear_of_midpoints, _u16
from tests.test_gpu_layer import SMALL, assert_rows_close
from tests.test_gpu_mask import _mask
from tests.test_gpu_turbo import _near_bf16_midpoint

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_gated_attention_gb300 import build
    build.build()


def _device(spec, case, turbo, mask):
    dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, case.cap,
                     kv_format="turbo4v" if turbo is not None else "bf16")
    dl.load_cache(case.ck, turbo if turbo is not None else case.cv)
    if mask is not None:
        dl.set_mask(torch.from_numpy(np.ascontiguousarray(mask, np.uint8)).cuda())
    return dl


def _check_turbo_rows(spec, case, got_codes, got_scales, oc, os_, ty, what):
    H, Hk, d, R = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.q_len
    off = 2 * H * d + Hk * d
    exact = 0
    for b in range(spec.batch):
        p = int(case.pos[b])
        for r in range(R):
            vr = ty[b, r, off:off + Hk * d].reshape(Hk, d) if ty is not None else None
            for kh in range(Hk):
                if vr is not None and _near_bf16_midpoint(vr[kh]).any():
                    continue
                assert np.array_equal(got_codes[b, kh, p + r], oc[b, kh, p + r]), what
                assert np.array_equal(got_scales[b, kh, p + r], os_[b, kh, p + r]), what
                exact += 1
    return exact


@pytest.mark.parametrize("name", ["batched_mixed_small", "verify_2k_p46"])
def test_turbo_cache_with_a_broadcast_mask(name):
    spec = SMALL[name]
    case = make_case(spec)
    codes, scales = synth.turbo4v_cache(spec, case.cap)
    mask = _mask(spec, 1, 31, "tree")
    dl = _device(spec, case, (codes.copy(), scales.copy()), mask)
    try:
        M, H, d = spec.batch * spec.q_len, spec.num_heads, spec.head_dim
        out = torch.zeros((spec.batch, spec.q_len, spec.hidden), dtype=torch.bfloat16, device="cuda")
        ta = torch.zeros((M, H * d), dtype=torch.float32, device="cuda")
        dl.set_taps(None, ta)
        dl.step(x_to_device(spec, case.x), torch.from_numpy(case.pos.astype(np.int32)).cuda(), out)
        dl.poll()
        k, (gc, gs) = dl.read_cache()
        got_out = out.float().cpu().numpy().astype(np.float64)
        got_ta = ta.cpu().numpy().astype(np.float64).reshape(spec.batch, spec.q_len, H, d)
    finally:
        dl.close()
    kc, oc, os_ = case.ck.copy(), codes.copy(), scales.copy()
    ref, ty, rta = orc.layer_step_ext(spec, case.orc_weights, synth.x_values(spec, case.x), kc,
                                      None, case.pos, turbo=(oc, os_), mask=mask, taps=True)
    ok, rep = refs.close(got_out, ref)
    assert ok, f"{name} out: {rep}"
    ok, rep = refs.close(got_ta, rta)
    assert ok, f"{name} attention: {rep}"
    for b in range(spec.batch):
        p = int(case.pos[b])
        assert_rows_close(k[b, :, p:p + spec.q_len], kc[b, :, p:p + spec.q_len], f"{name} k")
    assert _check_turbo_rows(spec, case, gc, gs, oc, os_, ty, name) > 0


def _block(spec, case, turbo, mask):
    il, pl = synth.block_norm_weights_bf16(spec)
    xv = synth.x_values(spec, case.x)
    il = _clear_of_midpoints(spec, xv, il)
    dl = _device(spec, case, turbo, mask)
    try:
        out = torch.zeros((spec.batch, spec.q_len, spec.hidden), dtype=torch.bfloat16, device="cuda")
        on = torch.zeros_like(out)
        dl.step_block(x_to_device(spec, case.x), torch.from_numpy(case.pos.astype(np.int32)).cuda(),
                      _u16(il), _u16(pl), out, on)
        dl.poll()
        cache = dl.read_cache()
        got = (out.float().cpu().numpy().astype(np.float64),
               on.float().cpu().numpy().astype(np.float64), cache)
    finally:
        dl.close()
    kc = case.ck.copy()
    tv = None if turbo is None else (turbo[0].copy(), turbo[1].copy())
    vc = None if turbo is not None else case.cv.copy()
    ref, rn = orc.block_step(spec, case.orc_weights, xv, il, pl, kc, vc, case.pos, turbo=tv,
                             mask=mask)
    return got, (ref, rn, kc, vc, tv)


def test_block_over_a_turbo_cache():
    spec = SMALL["decode_4b"]
    case = make_case(spec)
    codes, scales = synth.turbo4v_cache(spec, case.cap)
    (out, on, (k, (gc, gs))), (ref, rn, kc, _, (oc, os_)) = _block(spec, case, (codes, scales), None)
    for got, want, what in ((out, ref, "out"), (on, rn, "out_normed")):
        ok, rep = refs.close(got, want)
        assert ok, f"{what}: {rep}"
    p = int(case.pos[0])
    assert_rows_close(k[0, :, p:p + 1], kc[0, :, p:p + 1], "block turbo k")
    # the block's layer input is the normed row, so the V rows are checked on their dequantized values
    for kh in range(spec.num_kv_heads):
        gv = orc.turbo4_dequant_rows(gc[0, kh, p][None], gs[0, kh, p][None])[0]
        wv = orc.turbo4_dequant_rows(oc[0, kh, p][None], os_[0, kh, p][None])[0]
        assert np.linalg.norm(gv - wv) <= 0.2 * np.linalg.norm(wv)
    assert np.sum(gc[0, :, p] == oc[0, :, p]) > 0.9 * gc[0, :, p].size


def test_block_with_a_mask():
    spec = SMALL["batched_mixed_small"]
    case = make_case(spec)
    mask = _mask(spec, 1, 32, "random")
    (out, on, (k, v)), (ref, rn, kc, vc, _) = _block(spec, case, None, mask)
    for got, want, what in ((out, ref, "out"), (on, rn, "out_normed")):
        ok, rep = refs.close(got, want)
        assert ok, f"{what}: {rep}"
    for b in range(spec.batch):
        p = int(case.pos[b])
        assert_rows_close(k[b, :, p:p + spec.q_len], kc[b, :, p:p + spec.q_len], "block mask k")
        assert_rows_close(v[b, :, p:p + spec.q_len], vc[b, :, p:p + spec.q_len], "block mask v")
