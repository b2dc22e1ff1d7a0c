"""Pins for the float64 CPU oracle: each check ties a part of the oracle to
something other than itself -- library routines, closed forms, invariants,
special cases and brute force -- and the mutation checks show that a plausible
mistake in any step fails the same comparison the GPU parity tests apply."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as orc
from qwen3_gated_attention_gb300 import synth
from qwen3_gated_attention_gb300.synth import bf16_bits_to_f32, f32_to_bf16_bits
from tests import refs

BITS = (2, 3, 4, 5, 6, 8)


# --------------------------------------------------------------------- bf16

def test_bf16_rounding_matches_torch_on_float32_values():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
                        np.array([0.0, -0.0, 1.0, 3.4e38, -3.4e38, 1e-40, -1e-40, 2.0 ** -133,
                                  2.0 ** -134, 1.5 * 2.0 ** -133], np.float32)]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_from_double(float(a)) for a in v], np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rounding_of_float64_values_near_ties():
    """float64 values within a hair of a bf16 tie, where a float32 step in
    between would round twice: the oracle rounds once, like the round-to-odd
    reference the torch pins use."""
    rng = np.random.default_rng(11)
    v = rng.standard_normal(3000) * 10.0 ** rng.integers(-20, 20, 3000)
    base = np.array([orc.bf16_to_double(orc.bf16_from_double(float(a))) for a in v])
    base = base[base != 0]
    half_ulp = np.ldexp(1.0, np.frexp(base)[1] - 9)      # bf16 keeps 8 significant bits
    x = np.concatenate([base + half_ulp * (1 + 2.0 ** -30), base + half_ulp * (1 - 2.0 ** -30),
                        base + half_ulp, base - half_ulp * (1 + 2.0 ** -40)])
    got = np.array([orc.bf16_to_double(orc.bf16_from_double(float(a))) for a in x])
    ref = refs.to_bf16_values(torch.from_numpy(x)).numpy()
    assert np.array_equal(got, ref)
    twice = torch.from_numpy(x).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.any(twice != ref)          # the cases do separate one rounding from two


def test_bf16_ties_to_even_and_specials():
    assert orc.bf16_from_double(1.0) == 0x3F80
    assert orc.bf16_from_double(1.0 + 2.0 ** -8) == 0x3F80          # tie -> even
    assert orc.bf16_from_double(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie -> even
    assert orc.bf16_from_double(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert orc.bf16_from_double(float("inf")) == 0x7F80
    assert orc.bf16_from_double(-float("inf")) == 0xFF80
    assert orc.bf16_from_double(2.0 ** 128) == 0x7F80
    assert orc.bf16_from_double(2.0 ** -133) == 0x0001
    assert orc.bf16_from_double(float("nan")) & 0x7F80 == 0x7F80
    for h in (0x0001, 0x3F80, 0xC2F7, 0x7F7F, 0x8000):
        assert orc.bf16_from_double(orc.bf16_to_double(h)) == h


# ---------------------------------------------------------- packing, dequant

@pytest.mark.parametrize("bits", BITS)
def test_every_code_at_every_position_roundtrips(bits):
    K = 128
    N = (1 << bits) + 3
    codes = np.zeros((N, K), np.int64)
    for n in range(N):
        codes[n] = (np.arange(K) + n) % (1 << bits)
    packed = refs.encode_codes(codes, bits)
    assert np.array_equal(orc.unpack_codes(packed, N, K, bits), codes)
    assert np.array_equal(refs.decode_codes(packed, K, bits), codes)


@pytest.mark.parametrize("bits,group", [(2, 32), (3, 32), (4, 64), (5, 64), (6, 128), (8, 64),
                                        (4, 128), (8, 32)])
def test_quantizer_error_bound_and_dequant_closed_form(bits, group):
    rng = np.random.default_rng(bits * 1000 + group)
    N, K = 24, 256
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32).astype(np.float64)
    w[3, :group] = 0.125          # constant group: scale 0, code 0, bias exact
    packed, scales, biases = orc.quantize_affine(w, bits, group)
    codes = refs.decode_codes(packed, K, bits)
    assert codes.max() <= (1 << bits) - 1
    s = np.repeat(bf16_bits_to_f32(scales).astype(np.float64), group, axis=1)
    b = np.repeat(bf16_bits_to_f32(biases).astype(np.float64), group, axis=1)
    W = orc.dequantize(packed, scales, biases, N, K, bits, group)
    assert np.array_equal(W, s * codes + b)                 # w = scale * q + bias, exactly
    wmin = np.repeat(w.reshape(N, -1, group).min(2), group, axis=1)
    wmax = np.repeat(w.reshape(N, -1, group).max(2), group, axis=1)
    bound = s / 2 + 2.0 ** -8 * (np.abs(wmin) + np.abs(wmax)) + 1e-12
    assert np.all(np.abs(W - w) <= bound)
    assert np.all(W[3, :group] == 0.125)


@pytest.mark.parametrize("bits,group", [(4, 64), (8, 64), (6, 128), (3, 32)])
def test_qmatvec_equals_dense_matvec(bits, group):
    rng = np.random.default_rng(7)
    N, K = 40, 256
    w = rng.standard_normal((N, K)) * 0.02
    packed, scales, biases = orc.quantize_affine(w, bits, group)
    x = rng.standard_normal((3, K))
    y = orc.qmatvec(packed, scales, biases, N, K, bits, group, x)
    Wn = refs.dequant_np(packed, scales, biases, K, bits, group)
    np.testing.assert_allclose(y, x @ Wn.T, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ norm, rotary

def test_rms_norm_matches_torch_and_invariants():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(256) * 3.0
    w = 1 + 0.1 * rng.standard_normal(256)
    eps = float(np.float32(1e-6))
    y = orc.rms_norm(x, w, eps)
    ref = F.rms_norm(torch.from_numpy(x), (256,), torch.from_numpy(w), eps).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-15)
    one = orc.rms_norm(x, np.ones(256), 0.0)
    assert abs(math.sqrt(np.mean(one ** 2)) - 1.0) < 1e-13
    np.testing.assert_allclose(orc.rms_norm(7.5 * x, w, 0.0), orc.rms_norm(x, w, 0.0), rtol=1e-13)


def test_rotary_dims_from_partial_factor():
    assert orc.rotary_dims(256, 0.25) == 64
    assert orc.rotary_dims(64, float(np.float32(0.25))) == 16
    assert orc.rotary_dims(256, 1.0) == 256
    assert orc.rotary_dims(100, 0.33) == 33          # truncates


def test_rope_identity_at_zero_and_untouched_tail():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(256)
    assert np.array_equal(orc.rope(x, 64, 0.0, 1e7), x)
    y = orc.rope(x, 64, 1234.0, 1e7)
    assert np.array_equal(y[64:], x[64:])
    assert not np.allclose(y[:64], x[:64])
    pairs_x = x[:32] ** 2 + x[32:64] ** 2
    pairs_y = y[:32] ** 2 + y[32:64] ** 2
    np.testing.assert_allclose(pairs_y, pairs_x, rtol=1e-12)


def test_rope_matches_complex_exponential_form():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 256))
    pos = np.array([0, 1, 2, 46, 4095, 32767, 100000], np.float64)
    got = np.stack([orc.rope(x[i], 64, pos[i], 1e7) for i in range(7)])
    ref = refs.rope_complex(torch.from_numpy(x), 64, torch.from_numpy(pos), 1e7).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-9)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    a = orc.rope(q, 16, 5.0, 1e7) @ orc.rope(k, 16, 2.0, 1e7)
    b = orc.rope(q, 16, 130.0, 1e7) @ orc.rope(k, 16, 127.0, 1e7)
    assert abs(a - b) < 1e-10


# ---------------------------------------------------------- head-chunk plan

def _plan_rederived(q_len, H, Hk, enabled):
    """Per-head chunk labels from the eligibility sentence, built head by head."""
    gqa = H // Hk
    eligible = enabled and q_len * gqa > 32 and q_len <= 32
    per = max(1, min(gqa, 32 // q_len)) if eligible else gqa
    labels = [(h // gqa, (h % gqa) // per) for h in range(H)]
    chunks = []
    for h in range(H):
        if h == 0 or labels[h] != labels[h - 1]:
            chunks.append([h, 0])
        chunks[-1][1] += 1
    return [tuple(c) for c in chunks]


def test_head_chunk_plan_brute_force():
    n = 0
    for q_len in range(1, 34):
        for gqa in range(1, 65):
            for Hk in (1, 2, 3):
                for enabled in (True, False):
                    H = gqa * Hk
                    got = orc.head_chunk_plan(q_len, H, Hk, enabled)
                    assert got == _plan_rederived(q_len, H, Hk, enabled), (q_len, gqa, Hk, enabled)
                    n += 1
    assert n == 33 * 64 * 3 * 2


def test_head_chunk_plan_shipped_verify_case():
    # 24 query heads over 2 KV heads, four rows: 48 > 32 -> chunks of 8 and a remainder of 4
    assert orc.head_chunk_plan(4, 24, 2) == [(0, 8), (8, 4), (12, 8), (20, 4)]
    assert orc.head_chunk_plan(4, 24, 2, enabled=False) == [(0, 12), (12, 12)]
    assert orc.head_chunk_plan(1, 16, 4) == [(0, 4), (4, 4), (8, 4), (12, 4)]   # 4 <= 32: off
    assert orc.head_chunk_plan(33, 24, 2) == [(0, 12), (12, 12)]                  # q_len > 32


# ------------------------------------------------------------------- SDPA

def _rand_cache(rng, Hk, cap, d):
    k = f32_to_bf16_bits(rng.standard_normal((Hk, cap, d)).astype(np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((Hk, cap, d)).astype(np.float32))
    return k, v


@pytest.mark.parametrize("H,Hk,R,pos0", [(4, 2, 1, 0), (4, 2, 1, 31), (24, 2, 4, 46), (8, 8, 3, 10),
                                         (6, 1, 4, 5)])
def test_sdpa_matches_torch_gqa_causal(H, Hk, R, pos0):
    rng = np.random.default_rng(H * 100 + R)
    d, cap = 32, 64
    k, v = _rand_cache(rng, Hk, cap, d)
    q = rng.standard_normal((H, R, d))
    got = orc.sdpa(q, k, v, H, 0, pos0)
    L = pos0 + R
    Kt = torch.from_numpy(bf16_bits_to_f32(k[:, :L]).astype(np.float64))[None]
    Vt = torch.from_numpy(bf16_bits_to_f32(v[:, :L]).astype(np.float64))[None]
    mask = torch.arange(L)[None, :] <= (pos0 + torch.arange(R))[:, None]
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[None], Kt, Vt, attn_mask=mask,
                                         enable_gqa=True)[0].numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_sdpa_special_cases():
    rng = np.random.default_rng(9)
    d, cap, H, Hk = 16, 32, 4, 2
    k, v = _rand_cache(rng, Hk, cap, d)
    q = rng.standard_normal((H, 1, d))
    # one visible position: the output is that V row
    out = orc.sdpa(q, k, v, H, 0, 0)
    for h in range(H):
        assert np.array_equal(out[h, 0], bf16_bits_to_f32(v[h // 2, 0]).astype(np.float64))
    # all keys equal: uniform weights, the mean of the visible V rows
    k2 = np.repeat(k[:, :1], cap, axis=1)
    out = orc.sdpa(q, k2, v, H, 0, 9)
    for h in range(H):
        want = bf16_bits_to_f32(v[h // 2, :10]).astype(np.float64).mean(0)
        np.testing.assert_allclose(out[h, 0], want, rtol=1e-13, atol=1e-14)
    # identical query heads in a group give identical outputs
    q2 = np.repeat(q[:1], H, axis=0)
    out = orc.sdpa(q2, k, v, H, 0, 20)
    assert np.array_equal(out[0], out[1]) and np.array_equal(out[2], out[3])


# ------------------------------------------------------------------ layer

def _oracle_case(spec, B=None):
    if B is not None:
        spec = spec.with_(batch=B)
    wf = synth.weights_f32(spec)
    packed, scales, biases = [], [], []
    for i, w in enumerate(wf):
        p, s, b = orc.quantize_affine(w.astype(np.float64), spec.bits[i], spec.group[i])
        packed.append(p), scales.append(s), biases.append(b)
    qn, kn = synth.norm_weights_bf16(spec)
    W = orc.OracleWeights(packed, scales, biases, qn, kn, list(spec.bits), list(spec.group))
    x = synth.x_values(spec, synth.layer_input(spec))
    ck, cv = synth.cache(spec, fill=0x3F80)
    return spec, W, x, ck, cv, spec.positions()


def _run_oracle(spec, W, x, ck, cv, pos, **kw):
    ck, cv = ck.copy(), cv.copy()
    out, y, attn = orc.layer_step(spec, W, x, ck, cv, pos, taps=True, **kw)
    R = spec.q_len
    k_rows = np.stack([ck[b, :, pos[b]:pos[b] + R] for b in range(len(pos))])
    v_rows = np.stack([cv[b, :, pos[b]:pos[b] + R] for b in range(len(pos))])
    return dict(out=out, y=y, attn=attn, k_rows=bf16_bits_to_f32(k_rows).astype(np.float64),
                v_rows=bf16_bits_to_f32(v_rows).astype(np.float64)), ck, cv


def _torch_case(spec, W, x, ck, cv, pos):
    Ks = [spec.hidden] * 3 + [spec.num_heads * spec.head_dim]
    Wdeq = [refs.dequant_np(W.packed[i], W.scales[i], W.biases[i], Ks[i], spec.bits[i],
                            spec.group[i]) for i in range(4)]
    out, y, attn, kb, vb = refs.torch_layer(
        spec, Wdeq, bf16_bits_to_f32(W.q_norm).astype(np.float64),
        bf16_bits_to_f32(W.k_norm).astype(np.float64), x,
        bf16_bits_to_f32(ck).astype(np.float64), bf16_bits_to_f32(cv).astype(np.float64), pos)
    return dict(out=out, y=y, attn=attn, k_rows=kb.transpose(0, 2, 1, 3), v_rows=vb.transpose(0, 2, 1, 3))


SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    "verify_small": synth.WORKLOADS["tiny"].with_(name="verify_small", num_heads=12, num_kv_heads=1,
                                                  q_len=4, cache_pos=(46,), x_dtype="bf16"),
    "batched_small": synth.WORKLOADS["tiny"].with_(name="batched_small", batch=3, q_len=2,
                                                   cache_pos=None, length_range=(20, 90),
                                                   bits=(6, 6, 6, 3), group=(128, 128, 128, 32)),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_matches_torch_composition(name):
    case = _oracle_case(SMALL[name])
    spec = case[0]
    got, _, _ = _run_oracle(*case)
    ref = _torch_case(*case)
    for k in ("out", "y", "attn"):
        np.testing.assert_allclose(got[k], ref[k], rtol=1e-8, atol=1e-10, err_msg=k)
    # cache rows: both sides round the float64 rows once to bf16
    for k in ("k_rows", "v_rows"):
        assert np.array_equal(got[k], ref[k]), k
    assert spec.n_q == 2 * spec.num_heads * spec.head_dim     # doubled q_proj
    assert got["y"].shape[-1] == spec.n_q + 2 * spec.n_kv


def _random_geometries(n=12, seed=2024):
    """Seeded layer shapes beyond the named cases: full, half and quarter RoPE,
    gqa 1 to 6 (odd ones included), head dims 64 and 128, every code width,
    mixed q/k/v vs o widths and groups, 1 to 17 rows, one or two sequences at
    random positions.  Both sides get the same shapes; nothing is tuned."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([64, 128]))
        Hk = int(rng.choice([1, 2, 4]))
        gqa = int(rng.choice([1, 2, 3, 6]))
        H = Hk * gqa
        prf = float(rng.choice([0.25, 0.5, 1.0]))
        hidden = int(rng.choice([128, 256, 384]))
        bq, bo = (int(b) for b in rng.choice([2, 3, 4, 5, 6, 8], 2))
        gq, go = (int(g) for g in rng.choice([32, 64, 128], 2))
        if hidden % gq or (H * d) % go:
            continue
        R = int(rng.choice([1, 2, 3, 4, 5, 17]))
        B = int(rng.integers(1, 3))
        out.append(synth.WORKLOADS["tiny"].with_(
            name=f"rand{len(out)}", hidden=hidden, num_heads=H, num_kv_heads=Hk, head_dim=d,
            partial_rotary_factor=prf, bits=(bq, bq, bq, bo), group=(gq, gq, gq, go), batch=B,
            q_len=R, cache_pos=None, length_range=(R + 1, 120), x_dtype=str(rng.choice(["f32", "bf16"])),
            seed=len(out) + 1))
    return out


@pytest.mark.parametrize("spec", _random_geometries(), ids=lambda s: s.name)
def test_layer_matches_torch_composition_on_varied_geometry(spec):
    case = _oracle_case(spec)
    got, _, _ = _run_oracle(*case)
    ref = _torch_case(*case)
    for k in ("out", "y", "attn"):
        np.testing.assert_allclose(got[k], ref[k], rtol=1e-8, atol=1e-10, err_msg=k)
    for k in ("k_rows", "v_rows"):
        assert np.array_equal(got[k], ref[k]), k
    # with the head-chunk route off the oracle gives the same result
    off, _, _ = _run_oracle(*case, head_chunk=False)
    np.testing.assert_allclose(off["out"], got["out"], rtol=1e-12, atol=1e-14)


# mutations below the bf16 precision of the GPU path itself: the torch pin
# catches them, the parity tolerance cannot (and need not)
_SUB_TOLERANCE = {"no_bf16_cache"}
# mutations of the Turbo4 V-cache path (the bf16 layer never runs it): the pins
# in test_oracle_turbo.py catch them
_TURBO_ONLY = {"turbo_no_iwht"}


@pytest.mark.parametrize("mutation", [m for m in orc.MUTATIONS
                                      if m != "none" and m not in _TURBO_ONLY])
def test_every_planted_mistake_fails_the_torch_pin(mutation):
    """Each mutation is a plausible mistake; the library-routine composition
    rejects every one of them at float64 tolerance."""
    bad = []
    for name in ("verify_small", "batched_small"):
        case = _oracle_case(SMALL[name])
        got, _, _ = _run_oracle(*case, mutate=mutation)
        ref = _torch_case(*case)
        bad += [(name, k) for k in ("out", "y", "attn", "k_rows", "v_rows")
                if not np.allclose(got[k], ref[k], rtol=1e-8, atol=1e-10)]
    assert bad, f"mutation {mutation} matches the torch composition"


@pytest.mark.parametrize("mutation", [m for m in orc.MUTATIONS
                                      if m != "none" and m not in _SUB_TOLERANCE | _TURBO_ONLY])
def test_every_planted_mistake_fails_the_parity_comparison(mutation):
    """The comparison the GPU tests use (out, attention tap, projection tap,
    appended cache rows at the parity tolerance) rejects the same mistakes."""
    reps = []
    for name in ("verify_small", "batched_small"):
        case = _oracle_case(SMALL[name])
        ref, _, _ = _run_oracle(*case)
        got, _, _ = _run_oracle(*case, mutate=mutation)
        ok, rep = refs.compare_layer(ref, got)
        reps.append(rep)
        if not ok:
            return
    pytest.fail(f"mutation {mutation} passes the comparison: {reps}")


def test_unmutated_oracle_passes_comparison_against_torch():
    case = _oracle_case(SMALL["verify_small"])
    ok, rep = refs.compare_layer(_torch_case(*case), _run_oracle(*case)[0])
    assert ok, rep


def _with_gate_rows(spec, W, scale_bits, bias_bits):
    """Set every gate row of q_proj to codes 0 with the given bf16 scale/bias."""
    packed = [p.copy() for p in W.packed]
    scales = [s.copy() for s in W.scales]
    biases = [b.copy() for b in W.biases]
    d = spec.head_dim
    for h in range(spec.num_heads):
        rows = slice(h * 2 * d + d, (h + 1) * 2 * d)
        packed[0][rows] = 0
        scales[0][rows] = scale_bits
        biases[0][rows] = bias_bits
    return orc.OracleWeights(packed, scales, biases, W.q_norm, W.k_norm, W.bits, W.group)


def test_gate_limits():
    spec, W, x, ck, cv, pos = _oracle_case(SMALL["verify_small"])
    xp = np.abs(x) + 0.5                            # x > 0 so the gate = sum(x) * bias
    ungated, _, _ = _run_oracle(spec, W, xp, ck, cv, pos, mutate="no_gate")
    # gate rows with bias +1: gate = sum(x) >> 0, sigmoid -> 1: the ungated layer
    big, _, _ = _run_oracle(spec, _with_gate_rows(spec, W, 0, 0x3F80), xp, ck, cv, pos)
    np.testing.assert_allclose(big["out"], ungated["out"], rtol=1e-12, atol=1e-15)
    # gate rows zero: sigmoid(0) = 1/2 exactly
    half, _, _ = _run_oracle(spec, _with_gate_rows(spec, W, 0, 0), xp, ck, cv, pos)
    np.testing.assert_allclose(half["out"], 0.5 * ungated["out"], rtol=1e-12, atol=1e-15)
    # large negative gate: the layer output vanishes
    neg, _, _ = _run_oracle(spec, _with_gate_rows(spec, W, 0, 0xBF80), xp, ck, cv, pos)
    assert np.max(np.abs(neg["out"])) < 1e-30


def test_zero_query_rows_give_uniform_attention():
    spec, W, x, ck, cv, pos = _oracle_case(SMALL["tiny"])
    d = spec.head_dim
    packed = [p.copy() for p in W.packed]
    scales = [s.copy() for s in W.scales]
    biases = [b.copy() for b in W.biases]
    for h in range(spec.num_heads):
        rows = slice(h * 2 * d, h * 2 * d + d)
        packed[0][rows], scales[0][rows], biases[0][rows] = 0, 0, 0
    W0 = orc.OracleWeights(packed, scales, biases, W.q_norm, W.k_norm, W.bits, W.group)
    got, ck2, cv2 = _run_oracle(spec, W0, x, ck, cv, pos)
    p = int(pos[0])
    for h in range(spec.num_heads):
        kh = h // spec.gqa
        want = bf16_bits_to_f32(cv2[0, kh, :p + 1]).astype(np.float64).mean(0)
        np.testing.assert_allclose(got["attn"][0, 0, h], want, rtol=1e-12, atol=1e-14)


def test_one_verify_step_equals_row_by_row_steps_and_batch_equals_solo():
    spec, W, x, ck, cv, pos = _oracle_case(SMALL["batched_small"])
    full, ckf, cvf = _run_oracle(spec, W, x, ck, cv, pos)
    # row by row: q_len 1 at cache_pos + r
    ck1, cv1 = ck.copy(), cv.copy()
    s1 = spec.with_(q_len=1)
    for r in range(spec.q_len):
        out = orc.layer_step(s1, W, np.ascontiguousarray(x[:, r:r + 1]), ck1, cv1, pos + r)
        np.testing.assert_allclose(out[:, 0], full["out"][:, r], rtol=1e-12, atol=1e-15)
    assert np.array_equal(ck1, ckf) and np.array_equal(cv1, cvf)
    # sequence by sequence
    for b in range(spec.batch):
        sb = spec.with_(batch=1)
        kb, vb = ck[b:b + 1].copy(), cv[b:b + 1].copy()
        out = orc.layer_step(sb, W, np.ascontiguousarray(x[b:b + 1]), kb, vb, pos[b:b + 1])
        assert np.array_equal(out[0], full["out"][b])
        assert np.array_equal(kb[0], ckf[b])


def test_head_chunk_route_agrees_with_unchunked():
    spec, W, x, ck, cv, pos = _oracle_case(SMALL["verify_small"])
    assert len(orc.head_chunk_plan(spec.q_len, spec.num_heads, spec.num_kv_heads)) == 2
    on, _, _ = _run_oracle(spec, W, x, ck, cv, pos, head_chunk=True)
    off, _, _ = _run_oracle(spec, W, x, ck, cv, pos, head_chunk=False)
    for k in on:
        assert np.array_equal(on[k], off[k])


def test_capacity_overflow_is_rejected_without_writes():
    spec, W, x, ck, cv, pos = _oracle_case(SMALL["tiny"])
    cap = ck.shape[2]
    bad = np.array([cap - spec.q_len + 1], np.int32)
    ck2, cv2 = ck.copy(), cv.copy()
    with pytest.raises(ValueError):
        orc.layer_step(spec, W, x, ck2, cv2, bad)
    assert np.array_equal(ck2, ck) and np.array_equal(cv2, cv)


# ------------------------------------------------ decoder block (norm + residual)

def _block(spec, x, scale=1.0, input_ln=None, post_ln=None, with_post=True):
    from tests.cases import make_case
    case = make_case(spec)
    il, pl = synth.block_norm_weights_bf16(spec)
    il = il if input_ln is None else input_ln
    pl = pl if post_ln is None else post_ln
    k2, v2 = case.ck.copy(), case.cv.copy()
    out, on = orc.block_step(spec, case.orc_weights, x * scale, il, pl if with_post else None,
                             k2, v2, case.pos)
    return case, out, on, k2, v2


def test_block_layer_part_is_invariant_to_the_input_scale():
    """h = RMSNorm(x) * input_ln does not depend on the scale of x (up to eps),
    so out - x does not either; a block that skipped the input norm would
    scale its layer part by c (the q/k norms undo it, v and o_proj do not)."""
    spec = synth.WORKLOADS["tiny"]
    x = synth.x_values(spec, synth.layer_input(spec))
    _, o1, _, k1, v1 = _block(spec, x, 1.0)
    _, o4, _, k4, v4 = _block(spec, x, 4.0)
    ok, rep = refs.close(o4 - 4.0 * x, o1 - x, abs_tol=1e-5, rel_tol=1e-5, l2_tol=1e-5)
    assert ok, rep
    bad = np.abs((o4 - 4.0 * x) - 4.0 * (o1 - x)).max()
    assert bad > 1e-3      # the check above has power: scaled layer parts differ


def _unit_rms_bf16_rows(B, R, hidden, seed):
    """Rows whose every element is a bf16 number and whose mean square is
    exactly 1: groups of five (+-2, +-0.5 x 4; squares summing to 5) with the
    rest +-1, in random places and signs."""
    rng = np.random.default_rng(seed)
    x = np.empty((B, R, hidden))
    for b in range(B):
        for r in range(R):
            g = rng.integers(0, hidden // 5 + 1)
            row = np.array([2.0] * g + [0.5] * (4 * g) + [1.0] * (hidden - 5 * g))
            x[b, r] = rng.permutation(row) * rng.choice([-1.0, 1.0], hidden)
    assert np.all(np.mean(x * x, axis=-1) == 1.0)
    return x


@pytest.mark.parametrize("x_dtype", ["f32", "bf16"])
def test_block_reduces_to_the_layer_on_unit_rms_rows(x_dtype):
    """input_ln = 1 and rows of unit RMS: h = x up to eps, so out - x is the
    layer.  For a bf16 layer the rows are bf16 numbers, where rounding h to
    bf16 gives back x exactly (eps moves it by far less than half an ulp)."""
    spec = synth.WORKLOADS["tiny"].with_(batch=3, q_len=2, cache_pos=None,
                                         length_range=(20, 300), x_dtype=x_dtype)
    if x_dtype == "f32":
        x = synth.x_values(spec, synth.layer_input(spec))
        x = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True))
    else:
        x = _unit_rms_bf16_rows(spec.batch, spec.q_len, spec.hidden, 7)
    ones = np.full(spec.hidden, 0x3F80, np.uint16)
    case, out, _, k2, v2 = _block(spec, x, input_ln=ones)
    k3, v3 = case.ck.copy(), case.cv.copy()
    ref = orc.layer_step(spec, case.orc_weights, x, k3, v3, case.pos)
    ok, rep = refs.close(out - x, ref, abs_tol=1e-6, rel_tol=1e-5, l2_tol=1e-5)
    assert ok, rep


def test_block_post_norm_rows_have_unit_rms():
    """post_ln = 1: every row of RMSNorm(bf16(out)) has RMS 1 (up to eps)."""
    spec = synth.WORKLOADS["tiny"]
    x = synth.x_values(spec, synth.layer_input(spec))
    ones = np.full(spec.hidden, 0x3F80, np.uint16)
    _, out, on, _, _ = _block(spec, x, post_ln=ones)
    rms = np.sqrt(np.mean(on * on, axis=-1))
    assert np.allclose(rms, 1.0, atol=1e-5)
    # it normalizes the stored bf16 row, not the exact sum
    rb = np.vectorize(lambda v: orc.bf16_to_double(orc.bf16_from_double(v)))(out)
    exp = rb / np.sqrt(np.mean(rb * rb, axis=-1, keepdims=True) + spec.rms_eps)
    assert np.allclose(on, exp, rtol=0, atol=1e-12)


@pytest.mark.parametrize("spec", [SMALL["tiny"], SMALL["batched_small"],
                                  SMALL["verify_small"]] + _random_geometries()[:4],
                         ids=lambda s: s.name)
def test_block_matches_torch_composition(spec):
    """The decoder-block oracle against library routines: h = F.rms_norm(x,
    input_ln) (rounded once to bf16 for a bf16 layer), the torch layer on h,
    out = x + layer, out_normed = F.rms_norm(bf16(out), post_ln)."""
    _, W, x, ck, cv, pos = _oracle_case(spec)
    il, pl = synth.block_norm_weights_bf16(spec)
    out, on = orc.block_step(spec, W, x, il, pl, ck.copy(), cv.copy(), pos)
    eps = float(np.float32(spec.rms_eps))
    ilw = torch.from_numpy(bf16_bits_to_f32(il).astype(np.float64))
    plw = torch.from_numpy(bf16_bits_to_f32(pl).astype(np.float64))
    h = F.rms_norm(torch.from_numpy(x), (spec.hidden,), ilw, eps)
    if spec.x_dtype == "bf16":
        h = refs.to_bf16_values(h)
    ref = _torch_case(spec, W, h.numpy(), ck, cv, pos)
    want = x + ref["out"]
    np.testing.assert_allclose(out, want, rtol=1e-10, atol=1e-12)
    want_n = F.rms_norm(refs.to_bf16_values(torch.from_numpy(want)), (spec.hidden,), plw, eps).numpy()
    np.testing.assert_allclose(on, want_n, rtol=1e-9, atol=1e-11)
