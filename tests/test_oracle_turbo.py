"""Pins of the oracle's Turbo4 V-cache format (the Bf16KTurbo4V cache of the
Atlas qwen3_5 forward page: MetalKvDtype, LayerKvCache), each against
something other than the oracle itself: torch's float8_e4m3fn for the E4M3
codec, numerical integration for the Lloyd-Max optimality conditions, a dense
Hadamard matrix (scipy) for the rotation, the quantizer's distortion bound for
the round trip, and a numpy attention over the dequantized rows for the layer
step's wiring."""
import numpy as np
import pytest
import torch

import oracle as orc
from qwen3_gated_attention_gb300 import synth
from qwen3_gated_attention_gb300.synth import bf16_bits_to_f32, f32_to_bf16_bits

scipy_linalg = pytest.importorskip("scipy.linalg")
scipy_integrate = pytest.importorskip("scipy.integrate")
scipy_stats = pytest.importorskip("scipy.stats")


# ------------------------------------------------------------------ E4M3

def _torch_e4m3_bytes(x):
    t = torch.tensor(np.asarray(x, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _torch_e4m3_values(b):
    return torch.tensor(np.asarray(b, np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def test_e4m3_decode_matches_torch():
    b = np.arange(256, dtype=np.uint8)
    ref = _torch_e4m3_values(b).astype(np.float64)
    got = np.array([orc.e4m3_to_double(int(i)) for i in b])
    nan = (b & 0x7F) == 0x7F
    assert np.all(np.isnan(got[nan])) and np.all(np.isnan(ref[nan]))
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_encode_matches_torch_cast():
    """Nearest value, ties to even, inside the finite range: every E4M3 value,
    every midpoint between neighbours (the ties), points just off them, and
    random values over the whole range including the subnormals."""
    vals = _torch_e4m3_values(np.arange(256, dtype=np.uint8)).astype(np.float64)
    pos = np.unique(vals[np.isfinite(vals) & (vals >= 0)])
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.default_rng(3)
    xs = np.concatenate([pos, mids, mids * (1 + 1e-6), mids * (1 - 1e-6),
                         rng.uniform(0, 448, 4000), np.exp(rng.uniform(np.log(1e-4), np.log(448), 4000))])
    xs = np.concatenate([xs, -xs]).astype(np.float32)
    xs = xs[np.abs(xs) <= 448]
    got = np.array([orc.e4m3_from_float(float(x)) for x in xs], np.uint8)
    ref = _torch_e4m3_bytes(xs)
    # +0 and -0 may differ in sign only
    same = (got == ref) | ((got & 0x7F) == 0) & ((ref & 0x7F) == 0)
    assert same.all(), xs[~same][:5]


def test_e4m3_encode_saturates():
    assert orc.e4m3_from_float(448.0) == 0x7E
    for x in (449.0, 500.0, 1e6, float("inf")):
        assert orc.e4m3_from_float(x) == 0x7E
        assert orc.e4m3_from_float(-x) == 0xFE
    assert orc.e4m3_from_float(float("nan")) == 0x7F


# ------------------------------------------------------------- codebook

def test_lloyd_max_codebook_is_optimal():
    """Centroid condition (each level is the mean of N(0, 1) over its cell,
    cells bounded by the midpoints) by adaptive quadrature; for a log-concave
    density these conditions fix the quantizer uniquely."""
    c = orc.turbo4_codebook()
    assert np.all(np.diff(c) > 0)
    assert np.array_equal(c, -c[::-1])                 # exactly symmetric
    t = np.concatenate([[-np.inf], (c[1:] + c[:-1]) / 2, [np.inf]])
    pdf = scipy_stats.norm.pdf
    for j in range(16):
        m0 = scipy_integrate.quad(pdf, t[j], t[j + 1], epsabs=1e-15, epsrel=1e-13)[0]
        m1 = scipy_integrate.quad(lambda x: x * pdf(x), t[j], t[j + 1], epsabs=1e-15,
                                  epsrel=1e-13)[0]
        assert abs(m1 / m0 - c[j]) < 1e-9, (j, m1 / m0, c[j])


def _distortion(c):
    t = np.concatenate([[-np.inf], (c[1:] + c[:-1]) / 2, [np.inf]])
    return sum(scipy_integrate.quad(lambda x, cj=cj: (x - cj) ** 2 * scipy_stats.norm.pdf(x),
                                    t[j], t[j + 1], epsabs=1e-15)[0] for j, cj in enumerate(c))


def test_codebook_tables_f32():
    c = orc.turbo4_codebook()
    lv, th = orc.turbo4_tables_f32()
    assert np.array_equal(lv, c.astype(np.float32))
    assert np.array_equal(th, ((c[1:] + c[:-1]) / 2).astype(np.float32))
    assert th[7] == 0.0


# ------------------------------------------------------------ quantizer

def _rows(d, n, seed, kind="normal"):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        v = rng.standard_normal((n, d))
    elif kind == "heavy":
        v = rng.standard_t(3, size=(n, d)) * np.exp(rng.uniform(-6, 6, size=(n, 1)))
    elif kind == "sparse":
        v = rng.standard_normal((n, d)) * (rng.random((n, d)) < 0.05)
    return f32_to_bf16_bits(v.astype(np.float32))


@pytest.mark.parametrize("kind", ["normal", "heavy", "sparse"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_quantizer_decisions_against_dense_hadamard(d, kind):
    """Rotation by the dense Sylvester Hadamard matrix in float64; per group of
    16: the nearest level of y / rms(y) (where fp32 rounding cannot decide
    otherwise), the E4M3 scale of ||y|| / ||c(idx)||, nibble j of byte j/2."""
    v = _rows(d, 300, d + len(kind), kind)
    codes, scales = orc.turbo4_quantize_rows(v)
    H = scipy_linalg.hadamard(d).astype(np.float64)
    y = bf16_bits_to_f32(v).astype(np.float64) @ H.T / np.sqrt(d)
    c = orc.turbo4_codebook()
    t = (c[1:] + c[:-1]) / 2
    idx = np.empty((v.shape[0], d), np.int64)
    idx[:, 0::2] = codes & 15
    idx[:, 1::2] = codes >> 4
    checked = 0
    for g in range(d // 16):
        yg = y[:, 16 * g:16 * (g + 1)]
        ss = np.sum(yg * yg, axis=1)
        nz = ss > 0
        u = yg[nz] / np.sqrt(ss[nz] / 16)[:, None]
        want = np.searchsorted(t, u, side="left")       # thresholds strictly below u
        margin = np.min(np.abs(u[..., None] - t), axis=-1)
        sure = margin > 1e-5 * np.maximum(1.0, np.abs(u))
        assert np.array_equal(idx[nz, 16 * g:16 * (g + 1)][sure], want[sure])
        checked += int(sure.sum())
        # zero groups: codes 0, scale 0
        assert np.all(idx[~nz, 16 * g:16 * (g + 1)] == 0) and np.all(scales[~nz, g] == 0)
        # the scale: E4M3 of the matched-norm ratio for the codes chosen
        cn = np.sqrt(np.sum(c[idx[nz, 16 * g:16 * (g + 1)]] ** 2, axis=1))
        s = np.sqrt(ss[nz]) / cn
        ref = _torch_e4m3_bytes(np.minimum(s, 448.0))
        vals = _torch_e4m3_values(np.arange(256, dtype=np.uint8)).astype(np.float64)
        fin = np.sort(np.unique(vals[np.isfinite(vals) & (vals >= 0)]))
        mids = (fin[1:] + fin[:-1]) / 2
        near_tie = np.min(np.abs(s[:, None] - mids), axis=1) < 1e-5 * s
        got = scales[nz, g]
        assert np.array_equal(got[~near_tie], ref[~near_tie])
    assert checked > 0.99 * v.shape[0] * d * 0.9


def test_quantizer_zero_and_saturating_rows():
    d = 64
    v = np.zeros((3, d), np.uint16)
    v[1] = f32_to_bf16_bits(np.full(d, 3e4, np.float32))       # scale past 448
    v[2, 5] = f32_to_bf16_bits(np.array([1.0], np.float32))[0]  # one nonzero
    codes, scales = orc.turbo4_quantize_rows(v)
    assert np.all(codes[0] == 0) and np.all(scales[0] == 0)
    assert scales[1].max() == 0x7E                               # saturated, not NaN
    r = orc.turbo4_dequant_rows(codes, scales)
    assert np.all(np.isfinite(r))


def test_round_trip_error_within_the_codebook_distortion():
    """dequant(quantize(v)) for N(0, 1) rows: the relative squared error is
    below the Lloyd-Max distortion D of N(0, 1) (each group is normalized by
    its own RMS and its scale matched to its norm, which only helps) and
    above D / 2; dropping the inverse rotation makes it ~2."""
    D = _distortion(orc.turbo4_codebook())
    assert abs(D - 0.0095) < 2e-4
    for d in (64, 256):
        v = _rows(d, 1500, 7 * d)
        vf = bf16_bits_to_f32(v).astype(np.float64)
        codes, scales = orc.turbo4_quantize_rows(v)
        err = lambda r: float(np.mean(np.sum((r - vf) ** 2, 1) / np.sum(vf ** 2, 1)))
        e = err(orc.turbo4_dequant_rows(codes, scales))
        assert D / 2 < e < D, (d, e, D)
        assert err(orc.turbo4_dequant_rows(codes, scales, mutate="turbo_no_iwht")) > 1.0


def test_dequant_is_the_inverse_rotation_of_the_scaled_levels():
    d = 128
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 256, size=(20, d // 2), dtype=np.uint8)
    scales = rng.integers(0x28, 0x48, size=(20, d // 16), dtype=np.uint8)
    c = orc.turbo4_codebook()
    idx = np.empty((20, d), np.int64)
    idx[:, 0::2] = codes & 15
    idx[:, 1::2] = codes >> 4
    s = _torch_e4m3_values(scales).astype(np.float64)
    yhat = c[idx] * np.repeat(s, 16, axis=1)
    H = scipy_linalg.hadamard(d).astype(np.float64)
    want = yhat @ H.T / np.sqrt(d)
    assert np.allclose(orc.turbo4_dequant_rows(codes, scales), want, rtol=0, atol=1e-12)


# ------------------------------------------------------------ layer step

def _turbo_case(spec):
    from tests.cases import make_case
    case = make_case(spec)
    codes, scales = synth.turbo4v_cache(spec, case.cap)
    return case, codes, scales


def _numpy_attention(spec, ty, kc, vd, pos):
    """q = RoPE(RMSNorm(query)) from the projection tap, then causal GQA
    softmax attention over bf16 K rows and float64 V rows."""
    B, R = ty.shape[:2]
    H, Hk, d = spec.num_heads, spec.num_kv_heads, spec.head_dim
    gqa = H // Hk
    rd = orc.rotary_dims(d, spec.partial_rotary_factor)
    qn_w = bf16_bits_to_f32(synth.norm_weights_bf16(spec)[0]).astype(np.float64)
    out = np.zeros((B, R, H, d))
    for b in range(B):
        p0 = int(pos[b])
        for h in range(H):
            kh = h // gqa
            K = bf16_bits_to_f32(kc[b, kh]).astype(np.float64)
            for r in range(R):
                qf = ty[b, r, h * 2 * d:h * 2 * d + d]
                q = orc.rope(orc.rms_norm(qf, qn_w, float(np.float32(spec.rms_eps))), rd, p0 + r,
                             float(np.float32(spec.rope_theta)))
                last = p0 + r
                sc = K[:last + 1] @ q / np.sqrt(d)
                p = np.exp(sc - sc.max())
                p /= p.sum()
                out[b, r, h] = p @ vd[b, kh, :last + 1]
    return out


@pytest.mark.parametrize("name", ["tiny", "batched"])
def test_turbo_layer_step_wiring(name):
    """The Turbo4 layer step appends the quantized bf16 V rows and attends the
    dequantized V rows: its attention tap equals a numpy attention over the
    cache it leaves behind, and its new code rows are the quantizer's output
    on the bf16 values of its own v projection."""
    spec = synth.WORKLOADS["tiny"]
    if name == "batched":
        spec = spec.with_(batch=3, q_len=2, cache_pos=None, length_range=(20, 300), x_dtype="bf16")
    case, codes, scales = _turbo_case(spec)
    x = synth.x_values(spec, case.x)
    kc = case.ck.copy()
    out, ty, ta = orc.layer_step_turbo4v(spec, case.orc_weights, x, kc, codes, scales, case.pos,
                                         taps=True)
    H, Hk, d, R = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.q_len
    off = 2 * H * d + Hk * d
    for b in range(spec.batch):
        p0 = int(case.pos[b])
        for r in range(R):
            # bf16 rounding of the float64 tap, as the oracle rounds (nearest-even)
            vrow = np.array([[orc.bf16_from_double(float(t)) for t in row]
                             for row in ty[b, r, off:off + Hk * d].reshape(Hk, d)], np.uint16)
            cq, sq = orc.turbo4_quantize_rows(vrow)
            assert np.array_equal(codes[b, :, p0 + r], cq)
            assert np.array_equal(scales[b, :, p0 + r], sq)
    vd = orc.turbo4_dequant_rows(codes, scales)
    want = _numpy_attention(spec, ty, kc, vd, case.pos)
    assert np.allclose(ta, want, rtol=1e-10, atol=1e-12)
    # the mutation that skips the inverse rotation is visible in the same comparison
    c2, s2, k2 = *synth.turbo4v_cache(spec, case.cap), case.ck.copy()
    _, _, ta2 = orc.layer_step_turbo4v(spec, case.orc_weights, x, k2, c2, s2, case.pos,
                                       mutate="turbo_no_iwht", taps=True)
    assert not np.allclose(ta2, want, rtol=1e-3, atol=1e-3)


def test_turbo_layer_step_ignores_stale_slots():
    """Slots past cache_pos + R hold NaN scales (0x7F): nothing reads them."""
    spec = synth.WORKLOADS["tiny"].with_(batch=2, q_len=2, cache_pos=None, length_range=(20, 60))
    case, codes, scales = _turbo_case(spec)
    out = orc.layer_step_turbo4v(spec, case.orc_weights, synth.x_values(spec, case.x),
                                 case.ck.copy(), codes, scales, case.pos)
    assert np.all(np.isfinite(out))


def test_turbo_layer_step_with_a_mask_matches_numpy():
    """A Turbo4 V cache and a broadcast mask together: the attention tap is the
    numpy attention over the dequantized rows with the mask's positions."""
    spec = synth.WORKLOADS["tiny"].with_(batch=2, q_len=3, cache_pos=None, length_range=(20, 90),
                                         x_dtype="bf16")
    case, codes, scales = _turbo_case(spec)
    rng = np.random.default_rng(21)
    T = int(case.pos.max()) + spec.q_len
    mask = (rng.random((spec.batch, 1, spec.q_len, T)) < 0.6).astype(np.uint8)
    kc = case.ck.copy()
    out, ty, ta = orc.layer_step_ext(spec, case.orc_weights, synth.x_values(spec, case.x), kc, None,
                                     case.pos, turbo=(codes, scales), mask=mask, taps=True)
    vd = orc.turbo4_dequant_rows(codes, scales)
    B, R = spec.batch, spec.q_len
    H, Hk, d = spec.num_heads, spec.num_kv_heads, spec.head_dim
    rd = orc.rotary_dims(d, spec.partial_rotary_factor)
    qn_w = bf16_bits_to_f32(synth.norm_weights_bf16(spec)[0]).astype(np.float64)
    for b in range(B):
        p0 = int(case.pos[b])
        for h in range(H):
            K = bf16_bits_to_f32(kc[b, h // (H // Hk), :p0 + R]).astype(np.float64)
            for r in range(R):
                q = orc.rope(orc.rms_norm(ty[b, r, h * 2 * d:h * 2 * d + d], qn_w,
                                          float(np.float32(spec.rms_eps))), rd, p0 + r,
                             float(np.float32(spec.rope_theta)))
                keep = mask[b, 0, r, :p0 + R] != 0
                if not keep.any():
                    assert np.all(ta[b, r, h] == 0)
                    continue
                s = np.where(keep, K @ q / np.sqrt(d), -np.inf)
                p = np.exp(s - s.max())
                want = (p / p.sum()) @ vd[b, h // (H // Hk), :p0 + R]
                assert np.allclose(ta[b, r, h], want, rtol=1e-10, atol=1e-12)


def test_block_over_a_turbo_cache_reduces_to_the_turbo_layer():
    """input_ln = 1 on bf16 rows of unit RMS: the block's layer part is the
    Turbo4 layer step on x itself (rounding h to bf16 gives back x)."""
    from tests.test_oracle_pins import _unit_rms_bf16_rows
    spec = synth.WORKLOADS["tiny"].with_(batch=2, q_len=2, cache_pos=None, length_range=(20, 90),
                                         x_dtype="bf16")
    case, codes, scales = _turbo_case(spec)
    x = _unit_rms_bf16_rows(spec.batch, spec.q_len, spec.hidden, 4)
    ones = np.full(spec.hidden, 0x3F80, np.uint16)
    k1, c1, s1 = case.ck.copy(), codes.copy(), scales.copy()
    out, _ = orc.block_step(spec, case.orc_weights, x, ones, None, k1, None, case.pos,
                            turbo=(c1, s1))
    k2, c2, s2 = case.ck.copy(), codes.copy(), scales.copy()
    ref = orc.layer_step_ext(spec, case.orc_weights, x, k2, None, case.pos, turbo=(c2, s2))
    assert np.allclose(out - x, ref, rtol=1e-12, atol=1e-14)
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2) and np.array_equal(k1, k2)


def test_symmetric_turbo_layer_step_wiring():
    """The symmetric Turbo4 cache ([atlas-mod] MetalKvDtype::Turbo4): the new K
    rows are the quantizer's output on the bf16 normed, rotated key, the new V
    rows on the bf16 value, and the attention tap is a numpy attention over
    the dequantized K and V rows."""
    spec = synth.WORKLOADS["tiny"].with_(batch=2, q_len=2, cache_pos=None, length_range=(20, 90),
                                         x_dtype="bf16")
    case, vcodes, vscales = _turbo_case(spec)
    kcodes, kscales = synth.turbo4v_cache(spec, case.cap, plane="k")
    out, ty, ta = orc.layer_step_ext(spec, case.orc_weights, synth.x_values(spec, case.x), None,
                                     None, case.pos, turbo=(vcodes, vscales),
                                     turbo_k=(kcodes, kscales), taps=True)
    B, R = spec.batch, spec.q_len
    H, Hk, d = spec.num_heads, spec.num_kv_heads, spec.head_dim
    rd = orc.rotary_dims(d, spec.partial_rotary_factor)
    qn_w, kn_w = (bf16_bits_to_f32(w).astype(np.float64) for w in synth.norm_weights_bf16(spec))
    eps, theta = float(np.float32(spec.rms_eps)), float(np.float32(spec.rope_theta))
    for b in range(B):
        p0 = int(case.pos[b])
        for r in range(R):
            for kh in range(Hk):
                k = orc.rope(orc.rms_norm(ty[b, r, 2 * H * d + kh * d:2 * H * d + (kh + 1) * d], kn_w,
                                          eps), rd, p0 + r, theta)
                kb = np.array([[orc.bf16_from_double(float(t)) for t in k]], np.uint16)
                cq, sq = orc.turbo4_quantize_rows(kb)
                assert np.array_equal(kcodes[b, kh, p0 + r], cq[0])
                assert np.array_equal(kscales[b, kh, p0 + r], sq[0])
    kd = orc.turbo4_dequant_rows(kcodes, kscales)
    vd = orc.turbo4_dequant_rows(vcodes, vscales)
    gqa = H // Hk
    for b in range(B):
        p0 = int(case.pos[b])
        for h in range(H):
            for r in range(R):
                q = orc.rope(orc.rms_norm(ty[b, r, h * 2 * d:h * 2 * d + d], qn_w, eps), rd, p0 + r,
                             theta)
                s = kd[b, h // gqa, :p0 + r + 1] @ q / np.sqrt(d)
                p = np.exp(s - s.max())
                want = (p / p.sum()) @ vd[b, h // gqa, :p0 + r + 1]
                assert np.allclose(ta[b, r, h], want, rtol=1e-10, atol=1e-12)
