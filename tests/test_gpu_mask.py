"""Attention masks on the GPU against the oracle (DS4Server issue 113:
broadcast and head-specific masks on the verify route)."""
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


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_gated_attention_gb300 import build
    build.build()


def _run(spec, case, mask, head_chunk=True):
    dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, case.cap, head_chunk=head_chunk)
    try:
        dl.load_cache(case.ck, case.cv)
        M, H, d = spec.batch * spec.q_len, spec.num_heads, spec.head_dim
        out = torch.full((spec.batch, spec.q_len, spec.hidden), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        ta = torch.zeros((M, H * d), dtype=torch.float32, device="cuda")
        dl.set_taps(None, ta)
        if mask is not None:
            dl.set_mask(torch.from_numpy(np.ascontiguousarray(mask, np.uint8)).cuda())
        pd = torch.from_numpy(np.ascontiguousarray(case.pos, np.int32)).cuda()
        dl.step(x_to_device(spec, case.x), pd, out)
        dl.poll()
        k, v = dl.read_cache()
        return dict(out=out.float().cpu().numpy().astype(np.float64),
                    attn=ta.cpu().numpy().astype(np.float64).reshape(spec.batch, spec.q_len, H, d),
                    k=k, v=v)
    finally:
        dl.close()


def _oracle(spec, case, mask, head_chunk=True):
    kc, vc = case.ck.copy(), case.cv.copy()
    out, _, ta = orc.layer_step(spec, case.orc_weights, synth.x_values(spec, case.x), kc, vc,
                                case.pos, head_chunk=head_chunk, taps=True, mask=mask)
    return out, ta, kc, vc


def _mask(spec, heads, seed, kind="random"):
    rng = np.random.default_rng(seed)
    pos = spec.positions()
    T = int(pos.max()) + spec.q_len + 3
    if kind == "random":
        m = (rng.random((spec.batch, heads, spec.q_len, T)) < 0.5).astype(np.uint8)
    else:
        # a tree-verify mask: the prefix, plus a random ancestor chain among the new rows
        m = np.zeros((spec.batch, heads, spec.q_len, T), np.uint8)
        for b in range(spec.batch):
            p0 = int(pos[b])
            m[b, :, :, :p0] = 1
            for r in range(spec.q_len):
                m[b, :, r, p0 + r] = 1
                if r:
                    m[b, :, r, p0:p0 + r] = rng.random((heads, r)) < 0.5
    return m


CASES = {"batched_mixed_small": SMALL["batched_mixed_small"],
         "verify_2k_p46": SMALL["verify_2k_p46"], "decode_4b": SMALL["decode_4b"],
         "tiny_r8": synth.WORKLOADS["tiny"].with_(name="tiny_r8", batch=2, q_len=8, cache_pos=None,
                                                  length_range=(30, 200), x_dtype="bf16")}


def _check(name, spec, case, got, out, ta, kc):
    ok, rep = refs.close(got["out"], out)
    assert ok, f"{name} out: {rep}"
    ok, rep = refs.close(got["attn"], ta)
    assert ok, f"{name} attention: {rep}"
    for b in range(spec.batch):
        p = int(case.pos[b])
        assert_rows_close(got["k"][b, :, p:p + spec.q_len], kc[b, :, p:p + spec.q_len], f"{name} k")


@pytest.mark.parametrize("kind", ["random", "tree"])
@pytest.mark.parametrize("name", list(CASES))
def test_broadcast_mask_parity(name, kind):
    spec = CASES[name]
    case = make_case(spec)
    mask = _mask(spec, 1, 11, kind)
    got = _run(spec, case, mask)
    out, ta, kc, vc = _oracle(spec, case, mask)
    _check(name, spec, case, got, out, ta, kc)


@pytest.mark.parametrize("name", ["batched_mixed_small", "verify_2k_p46", "tiny_r8"])
def test_head_specific_mask_parity(name):
    spec = CASES[name]
    case = make_case(spec)
    mask = _mask(spec, spec.num_heads, 12)
    # the head-chunk route refuses a head-specific mask where it applies
    chunked = len(orc.head_chunk_plan(spec.q_len, spec.num_heads, spec.num_kv_heads)) > \
        spec.num_kv_heads
    if chunked:
        with pytest.raises(gattn.GattnError) as ei:
            _run(spec, case, mask, head_chunk=True)
        assert ei.value.status == 2
        with pytest.raises(orc.MaskRouteError):
            _oracle(spec, case, mask, head_chunk=True)
    got = _run(spec, case, mask, head_chunk=False)
    out, ta, kc, vc = _oracle(spec, case, mask, head_chunk=False)
    _check(name, spec, case, got, out, ta, kc)


def test_causal_mask_equals_the_unmasked_step_bitwise():
    spec = CASES["batched_mixed_small"]
    case = make_case(spec)
    pos = spec.positions()
    T = int(pos.max()) + spec.q_len
    t = np.arange(T)
    mask = np.zeros((spec.batch, 1, spec.q_len, T), np.uint8)
    for b in range(spec.batch):
        for r in range(spec.q_len):
            mask[b, 0, r] = t <= pos[b] + r
    a = _run(spec, case, mask)
    b = _run(spec, case, None)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["attn"], b["attn"])


def test_fully_masked_rows_are_zero():
    spec = CASES["tiny_r8"]
    case = make_case(spec)
    mask = _mask(spec, 1, 13)
    mask[0, :, 2] = 0
    mask[1, :, 5] = 0
    got = _run(spec, case, mask)
    assert np.all(got["attn"][0, 2] == 0) and np.all(got["attn"][1, 5] == 0)
    out, ta, kc, vc = _oracle(spec, case, mask)
    _check("tiny_r8", spec, case, got, out, ta, kc)



@pytest.mark.parametrize("name", ["batched_mixed_small", "tiny_r8"])
def test_mask_rows_shorter_than_the_attended_span(name):
    """Mask rows of fewer positions than cache_pos + R (DS4Server issue 113,
    masks sliced per head chunk): positions past a row are not attended.  The
    row length here sits inside the shortest sequence's span, so every
    sequence loses its tail.  Against the oracle's short-row entry, and
    bitwise equal to the same mask padded with zeros."""
    spec = CASES[name]
    case = make_case(spec)
    pos = spec.positions()
    T = int(pos.min()) + 1
    mask = _mask(spec, 1, 15, "tree")[..., :T].copy()
    mask[..., 0] = 1                      # every row keeps one visible position
    got = _run(spec, case, mask)
    kc, vc = case.ck.copy(), case.cv.copy()
    out, _, ta = orc.layer_step_ext(spec, case.orc_weights, synth.x_values(spec, case.x), kc, vc,
                                    case.pos, mask=mask, taps=True)
    _check(name, spec, case, got, out, ta, kc)
    padded = np.zeros(mask.shape[:3] + (int(pos.max()) + spec.q_len,), np.uint8)
    padded[..., :T] = mask
    full = _run(spec, case, padded)
    assert np.array_equal(got["out"], full["out"]) and np.array_equal(got["attn"], full["attn"])
