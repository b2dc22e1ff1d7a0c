"""The Bf16KTurbo4V cache on the GPU against the oracle: the standalone
quantizer bit for bit, and the layer step (output, attention tap, appended K
rows, appended V codes and scales, untouched slots)."""
import numpy as np
import pytest
import torch

import oracle as orc
from qwen3_gated_attention_gb300 import gattn, synth
from qwen3_gated_attention_gb300.device import DeviceLayer, x_to_device
from qwen3_gated_attention_gb300.synth import f32_to_bf16_bits
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


# ------------------------------------------------------------ quantizer

def _rows(d, n, seed):
    rng = np.random.default_rng(seed)
    parts = [rng.standard_normal((n, d)),
             rng.standard_t(3, size=(n, d)) * np.exp(rng.uniform(-8, 8, size=(n, 1))),
             rng.standard_normal((n, d)) * (rng.random((n, d)) < 0.05),
             np.zeros((2, d)), np.full((2, d), 3e4)]
    return f32_to_bf16_bits(np.concatenate(parts).astype(np.float32))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_quantizer_is_bit_exact(d):
    v = _rows(d, 700, d)
    codes, scales = orc.turbo4_quantize_rows(v)
    vd = torch.from_numpy(v.view(np.int16)).cuda()
    cd = torch.full((v.shape[0], d // 2), 0xAA, dtype=torch.uint8, device="cuda")
    sd = torch.full((v.shape[0], d // 16), 0xAA, dtype=torch.uint8, device="cuda")
    gattn.turbo4_quantize_device(vd.data_ptr(), v.shape[0], d, cd.data_ptr(), sd.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    gc, gs = cd.cpu().numpy(), sd.cpu().numpy()
    assert np.array_equal(gs, scales), np.argwhere(gs != scales)[:5]
    assert np.array_equal(gc, codes), np.argwhere(gc != codes)[:5]


# ------------------------------------------------------------ layer step

CASES = {n: SMALL[n] for n in ["tiny", "decode_4b", "verify_2k_p46", "batched_mixed_small"]}
CASES["d128_r4"] = [s for n, s in SMALL.items() if s.head_dim == 128][0] \
    if any(s.head_dim == 128 for s in SMALL.values()) else None
CASES = {k: v for k, v in CASES.items() if v is not None}


def _near_bf16_midpoint(v, rel=4e-6):
    """Elements of float64 v within `rel` of a bf16 rounding midpoint (where the
    kernel's fp32 projection may round to the other neighbour)."""
    a = np.abs(v)
    ulp = np.exp2(np.floor(np.log2(np.maximum(a, 1e-30))) - 7)
    t = a / ulp
    return (np.abs(t - np.floor(t) - 0.5) < rel * t) & (a > 0)


def _run_turbo(spec, case, codes, scales, head_chunk=True):
    dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, case.cap, kv_format="turbo4v",
                     head_chunk=head_chunk)
    try:
        dl.load_cache(case.ck, (codes, scales))
        M, H, d = spec.batch * spec.q_len, spec.num_heads, spec.head_dim
        out = torch.full((spec.batch, spec.q_len, spec.hidden), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        ta = torch.zeros((M, H * d), dtype=torch.float32, device="cuda")
        dl.set_taps(None, ta)
        pd = torch.from_numpy(np.ascontiguousarray(case.pos, np.int32)).cuda()
        dl.step(x_to_device(spec, case.x), pd, out)
        dl.poll()
        k, (c2, s2) = dl.read_cache()
        return dict(out=out.float().cpu().numpy().astype(np.float64),
                    attn=ta.cpu().numpy().astype(np.float64).reshape(spec.batch, spec.q_len, H, d),
                    k=k, codes=c2, scales=s2, launches=gattn.layer_launches_per_step(dl.h))
    finally:
        dl.close()


@pytest.mark.parametrize("name", list(CASES))
def test_turbo_layer_parity(name):
    spec = CASES[name]
    case = make_case(spec)
    codes, scales = synth.turbo4v_cache(spec, case.cap)
    got = _run_turbo(spec, case, codes.copy(), scales.copy())
    kc, oc, os_ = case.ck.copy(), codes.copy(), scales.copy()
    out, ty, ta = orc.layer_step_turbo4v(spec, case.orc_weights, synth.x_values(spec, case.x), kc,
                                         oc, os_, case.pos, taps=True)
    assert got["launches"] in (4, 5)
    ok, rep = refs.close(got["out"], out)
    assert ok, f"out: {rep}"
    ok, rep = refs.close(got["attn"], ta)
    assert ok, f"attention: {rep}"
    H, Hk, d, R = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.q_len
    off = 2 * H * d + Hk * d
    exempt = 0
    for b in range(spec.batch):
        p = int(case.pos[b])
        assert_rows_close(got["k"][b, :, p:p + R], kc[b, :, p:p + R], f"{name} k")
        for r in range(R):
            vr = ty[b, r, off:off + Hk * d].reshape(Hk, d)
            for kh in range(Hk):
                gc, gs = got["codes"][b, kh, p + r], got["scales"][b, kh, p + r]
                wc, ws = oc[b, kh, p + r], os_[b, kh, p + r]
                if _near_bf16_midpoint(vr[kh]).any():
                    # the bf16 input itself may differ by an ulp: the row must
                    # still be a faithful quantization of the oracle's row
                    exempt += 1
                    gv = orc.turbo4_dequant_rows(gc[None], gs[None])[0]
                    wv = orc.turbo4_dequant_rows(wc[None], ws[None])[0]
                    assert np.linalg.norm(gv - wv) <= 0.2 * np.linalg.norm(wv)
                    continue
                assert np.array_equal(gc, wc), (name, b, kh, r)
                assert np.array_equal(gs, ws), (name, b, kh, r)
        # every slot outside the appended rows is untouched (stale canaries included)
        mask = np.ones(oc.shape[1:3], bool)
        mask[:, p:p + R] = False
        assert np.array_equal(got["codes"][b][mask], codes[b][mask])
        assert np.array_equal(got["scales"][b][mask], scales[b][mask])
        kmask = np.ones(kc.shape[1:3], bool)
        kmask[:, p:p + R] = False
        assert np.array_equal(got["k"][b][kmask], case.ck[b][kmask])
    # about a third of d = 256 rows hold an element that close to a midpoint;
    # the rest (at least one row per case) must match bit for bit
    assert exempt < spec.batch * R * Hk


def test_turbo_head_chunk_on_and_off_agree_bitwise():
    spec = CASES["verify_2k_p46"]
    case = make_case(spec)
    codes, scales = synth.turbo4v_cache(spec, case.cap)
    a = _run_turbo(spec, case, codes.copy(), scales.copy(), head_chunk=True)
    b = _run_turbo(spec, case, codes.copy(), scales.copy(), head_chunk=False)
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["scales"], b["scales"])



# ------------------------------------------------- symmetric Turbo4 cache

def _run_sym(spec, case, kplanes, vplanes, head_chunk=True):
    dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, case.cap, kv_format="turbo4",
                     head_chunk=head_chunk)
    try:
        dl.load_cache(kplanes, vplanes)
        M, H, d = spec.batch * spec.q_len, spec.num_heads, spec.head_dim
        out = torch.full((spec.batch, spec.q_len, spec.hidden), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        ta = torch.zeros((M, H * d), dtype=torch.float32, device="cuda")
        dl.set_taps(None, ta)
        pd = torch.from_numpy(np.ascontiguousarray(case.pos, np.int32)).cuda()
        dl.step(x_to_device(spec, case.x), pd, out)
        dl.poll()
        (kc, ks), (vc, vs) = dl.read_cache()
        return dict(out=out.float().cpu().numpy().astype(np.float64),
                    attn=ta.cpu().numpy().astype(np.float64).reshape(spec.batch, spec.q_len, H, d),
                    kc=kc, ks=ks, vc=vc, vs=vs)
    finally:
        dl.close()


@pytest.mark.parametrize("name", list(CASES))
def test_symmetric_turbo_layer_parity(name):
    spec = CASES[name]
    case = make_case(spec)
    vcodes, vscales = synth.turbo4v_cache(spec, case.cap)
    kcodes, kscales = synth.turbo4v_cache(spec, case.cap, plane="k")
    got = _run_sym(spec, case, (kcodes.copy(), kscales.copy()), (vcodes.copy(), vscales.copy()))
    okc, oks, ovc, ovs = kcodes.copy(), kscales.copy(), vcodes.copy(), vscales.copy()
    out, ty, ta = orc.layer_step_ext(spec, case.orc_weights, synth.x_values(spec, case.x), None,
                                     None, case.pos, turbo=(ovc, ovs), turbo_k=(okc, oks),
                                     taps=True)
    ok, rep = refs.close(got["out"], out)
    assert ok, f"out: {rep}"
    ok, rep = refs.close(got["attn"], ta)
    assert ok, f"attention: {rep}"
    H, Hk, d, R = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.q_len
    rd = orc.rotary_dims(d, spec.partial_rotary_factor)
    kn_w = synth.bf16_bits_to_f32(case.kn).astype(np.float64)
    eps, theta = float(np.float32(spec.rms_eps)), float(np.float32(spec.rope_theta))
    exact = rows = 0
    for b in range(spec.batch):
        p = int(case.pos[b])
        for r in range(R):
            for kh in range(Hk):
                kraw = ty[b, r, 2 * H * d + kh * d:2 * H * d + (kh + 1) * d]
                k64 = orc.rope(orc.rms_norm(kraw, kn_w, eps), rd, p + r, theta)
                v64 = ty[b, r, 2 * H * d + Hk * d + kh * d:2 * H * d + Hk * d + (kh + 1) * d]
                for g, w, val in (((got["kc"], got["ks"]), (okc, oks), k64),
                                  ((got["vc"], got["vs"]), (ovc, ovs), v64)):
                    rows += 1
                    gc, gs = g[0][b, kh, p + r], g[1][b, kh, p + r]
                    wc, ws = w[0][b, kh, p + r], w[1][b, kh, p + r]
                    if _near_bf16_midpoint(val).any():
                        gv = orc.turbo4_dequant_rows(gc[None], gs[None])[0]
                        wv = orc.turbo4_dequant_rows(wc[None], ws[None])[0]
                        assert np.linalg.norm(gv - wv) <= 0.2 * np.linalg.norm(wv)
                        continue
                    assert np.array_equal(gc, wc) and np.array_equal(gs, ws), (name, b, kh, r)
                    exact += 1
        for g, before in ((got["kc"], kcodes), (got["ks"], kscales), (got["vc"], vcodes),
                          (got["vs"], vscales)):
            mask = np.ones(g.shape[1:3], bool)
            mask[:, p:p + R] = False
            assert np.array_equal(g[b][mask], before[b][mask])
    assert exact > 0, rows
