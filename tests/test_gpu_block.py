"""The decoder-block step (gattn_layer_step_block) against the oracle's block:
out = x + layer(RMSNorm(x) * input_ln), out_normed = RMSNorm(bf16(out)) * post_ln.

The residual x dominates out, and out is bf16, so each case also runs with x
scaled down by 64: the input norm makes the layer part scale-invariant, and
out's ulp is then small enough to check the layer part closely."""
import numpy as np
import pytest
import torch

import oracle as orc
from qwen3_gated_attention_gb300 import gattn, synth
from qwen3_gated_attention_gb300.device import DeviceLayer, x_to_device
from tests import refs
from tests.cases import make_case
from tests.test_gpu_layer import SMALL, assert_rows_close

pytestmark = pytest.mark.gpu

# the post-norm rides in the o_proj launch up to 16384 output elements
CASES = {n: SMALL[n] for n in ["tiny", "decode_4b", "verify_2k_p46", "batched_mixed_small"]}
CASES["decode_4b_b2r4"] = synth.WORKLOADS["decode_4b"].with_(
    name="decode_4b_b2r4", batch=2, q_len=4, cache_pos=None, length_range=(100, 3000))
POST_LAUNCH = {n: 5 if s.batch * s.q_len * s.hidden <= 16384 else 6 for n, s in CASES.items()}


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_gated_attention_gb300 import build
    build.build()


def _u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _run(case, x, il, pl, with_post=True):
    spec = case.spec
    dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, case.cap)
    try:
        dl.load_cache(case.ck, case.cv)
        out = torch.full((spec.batch, spec.q_len, spec.hidden), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        on = torch.full_like(out, float("nan")) if with_post else None
        pd = torch.from_numpy(np.ascontiguousarray(case.pos, np.int32)).cuda()
        dl.step_block(x_to_device(spec, x), pd, _u16(il), _u16(pl) if with_post else None, out, on)
        dl.poll()
        k, v = dl.read_cache()
        res = dict(out=out.float().cpu().numpy().astype(np.float64), k=k, v=v,
                   launches=gattn.layer_launches_per_step(dl.h))
        if with_post:
            res["on"] = on.float().cpu().numpy().astype(np.float64)
        return res
    finally:
        dl.close()


def _oracle(case, xv, il, pl):
    k2, v2 = case.ck.copy(), case.cv.copy()
    out, on = orc.block_step(case.spec, case.orc_weights, xv, il, pl, k2, v2, case.pos)
    return out, on, k2, v2


def _clear_of_midpoints(spec, xv, il, margin=4e-5, seed=11):
    """A bf16 layer rounds h = RMSNorm(x) * input_ln to bf16, the kernel from
    fp32 arithmetic and the oracle from fp64.  Elements of h within a relative
    `margin` of a rounding midpoint (well above the fp32 error of the norm) may
    round differently; step input_ln of their columns by an ulp or two until
    no such element is left, so both sides feed the layer the same h."""
    if spec.x_dtype != "bf16":
        return il
    rng = np.random.default_rng(seed)
    xs = xv.reshape(-1, spec.hidden)
    inv = 1.0 / np.sqrt(np.mean(xs * xs, axis=1) + spec.rms_eps)
    il = il.copy()
    for _ in range(500):
        w = synth.bf16_bits_to_f32(il).astype(np.float64)
        h = np.abs(xs * inv[:, None] * w[None, :])
        ulp = np.exp2(np.floor(np.log2(np.maximum(h, 1e-30))) - 7)
        t = h / ulp
        near = (np.abs(t - np.floor(t) - 0.5) < margin * t) & (h > 0)
        cols = np.flatnonzero(near.any(axis=0))
        if cols.size == 0:
            return il
        il[cols] = (il[cols].astype(np.int32) + rng.choice([-2, -1, 1, 2], cols.size)).astype(np.uint16)
    raise AssertionError("input_ln could not be moved clear of bf16 midpoints")


def _scaled_input(spec, x, factor):
    """x / factor in the layer's x representation (bf16 bits or fp32)."""
    v = synth.x_values(spec, x) / factor
    return v.astype(np.float32) if spec.x_dtype == "f32" else \
        synth.f32_to_bf16_bits(v.astype(np.float32))


@pytest.mark.parametrize("scale", [1.0, 64.0])
@pytest.mark.parametrize("name", list(CASES))
def test_block_parity(name, scale):
    spec = CASES[name]
    case = make_case(spec)
    il, pl = synth.block_norm_weights_bf16(spec)
    x = _scaled_input(spec, case.x, scale)
    xv = synth.x_values(spec, x)
    il = _clear_of_midpoints(spec, xv, il)
    got = _run(case, x, il, pl)
    out, on, k2, v2 = _oracle(case, xv, il, pl)
    assert got["launches"] == POST_LAUNCH[name]
    ok, rep = refs.close(got["out"], out)
    assert ok, f"out: {rep}"
    ok, rep = refs.close(got["on"], on)
    assert ok, f"out_normed: {rep}"
    if scale > 1.0:
        # the layer part itself, out - x, at bf16 resolution of the small out
        ok, rep = refs.close(got["out"] - xv, out - xv, abs_tol=2e-3, rel_tol=2e-2, l2_tol=2e-2)
        assert ok, f"layer part: {rep}"
    R = spec.q_len
    for b in range(spec.batch):
        p = int(case.pos[b])
        for key, ref in (("k", k2), ("v", v2)):
            assert_rows_close(got[key][b, :, p:p + R], ref[b, :, p:p + R], f"{name} {key}")
            mask = np.ones(ref.shape[1:3], bool)
            mask[:, p:p + R] = False
            assert np.array_equal(got[key][b][mask], ref[b][mask])


def test_block_without_post_norm_matches_block_with_it():
    spec = SMALL["batched_mixed_small"]
    case = make_case(spec)
    il, pl = synth.block_norm_weights_bf16(spec)
    a = _run(case, case.x, il, pl, with_post=True)
    b = _run(case, case.x, il, pl, with_post=False)
    assert a["launches"] == 5 and b["launches"] == 5
    assert np.array_equal(a["out"], b["out"])
