"""Pins of the oracle's attention masks (DS4Server issue 113: broadcast and
head-specific masks handed to each head chunk of the verify route): a numpy
attention over the same cache decides what every masked row must be."""
import numpy as np
import pytest

import oracle as orc
from qwen3_gated_attention_gb300 import synth
from qwen3_gated_attention_gb300.synth import bf16_bits_to_f32
from tests.cases import make_case


def _spec(R=4, B=2, H=None, Hk=None):
    s = synth.WORKLOADS["tiny"].with_(batch=B, q_len=R, cache_pos=None, length_range=(20, 90),
                                      x_dtype="bf16")
    if H is not None:
        s = s.with_(num_heads=H, num_kv_heads=Hk)
    return s


def _run(spec, mask=None, head_chunk=True):
    case = make_case(spec)
    kc, vc = case.ck.copy(), case.cv.copy()
    out, ty, ta = orc.layer_step(spec, case.orc_weights, synth.x_values(spec, case.x), kc, vc,
                                 case.pos, head_chunk=head_chunk, taps=True, mask=mask)
    return case, out, ty, ta, kc, vc


def _numpy_attention(spec, case, ty, kc, vc, mask):
    """q = RoPE(RMSNorm(query)) from the projection tap; softmax over the
    positions the mask keeps (t < cache_pos + R); a row with none is zero."""
    B, R = ty.shape[:2]
    H, Hk, d = spec.num_heads, spec.num_kv_heads, spec.head_dim
    gqa = H // Hk
    rd = orc.rotary_dims(d, spec.partial_rotary_factor)
    qn_w = bf16_bits_to_f32(case.qn).astype(np.float64)
    out = np.zeros((B, R, H, d))
    for b in range(B):
        p0 = int(case.pos[b])
        L = p0 + R
        for h in range(H):
            K = bf16_bits_to_f32(kc[b, h // gqa, :L]).astype(np.float64)
            V = bf16_bits_to_f32(vc[b, h // gqa, :L]).astype(np.float64)
            for r in range(R):
                q = orc.rope(orc.rms_norm(ty[b, r, h * 2 * d:h * 2 * d + d], qn_w,
                                          float(np.float32(spec.rms_eps))),
                             rd, p0 + r, float(np.float32(spec.rope_theta)))
                keep = mask[b, h if mask.shape[1] > 1 else 0, r, :L] != 0
                if not keep.any():
                    continue
                s = (K @ q) / np.sqrt(d)
                s = np.where(keep, s, -np.inf)
                p = np.exp(s - s.max())
                out[b, r, h] = (p / p.sum()) @ V
    return out


def _random_mask(spec, heads, seed, density=0.6):
    rng = np.random.default_rng(seed)
    T = int(spec.positions().max()) + spec.q_len + 5           # a wider row stride than needed
    return (rng.random((spec.batch, heads, spec.q_len, T)) < density).astype(np.uint8)


@pytest.mark.parametrize("heads", ["broadcast", "per_head"])
def test_masked_attention_matches_numpy(heads):
    spec = _spec()
    hm = 1 if heads == "broadcast" else spec.num_heads
    mask = _random_mask(spec, hm, 3)
    case, out, ty, ta, kc, vc = _run(spec, mask, head_chunk=False)
    want = _numpy_attention(spec, case, ty, kc, vc, mask)
    assert np.allclose(ta, want, rtol=1e-10, atol=1e-12)


def test_causal_mask_reproduces_the_unmasked_step_bit_for_bit():
    spec = _spec()
    pos = spec.positions()
    T = int(pos.max()) + spec.q_len
    t = np.arange(T)
    mask = np.zeros((spec.batch, 1, spec.q_len, T), np.uint8)
    for b in range(spec.batch):
        for r in range(spec.q_len):
            mask[b, 0, r] = t <= pos[b] + r
    _, out_m, _, ta_m, _, _ = _run(spec, mask)
    _, out_c, _, ta_c, _, _ = _run(spec, None)
    assert np.array_equal(ta_m, ta_c) and np.array_equal(out_m, out_c)


def test_single_visible_position_returns_that_value_row_and_empty_rows_are_zero():
    spec = _spec(R=3)
    pos = spec.positions()
    T = int(pos.max()) + spec.q_len
    mask = np.zeros((spec.batch, 1, spec.q_len, T), np.uint8)
    pick = [[3, 0, None], [7, None, 5]]                      # None: a fully masked row
    for b in range(spec.batch):
        for r in range(spec.q_len):
            if pick[b][r] is not None:
                mask[b, 0, r, pick[b][r]] = 1
    case, out, ty, ta, kc, vc = _run(spec, mask)
    gqa = spec.num_heads // spec.num_kv_heads
    for b in range(spec.batch):
        for r in range(spec.q_len):
            for h in range(spec.num_heads):
                if pick[b][r] is None:
                    assert np.all(ta[b, r, h] == 0.0)
                else:
                    v = bf16_bits_to_f32(vc[b, h // gqa, pick[b][r]]).astype(np.float64)
                    assert np.allclose(ta[b, r, h], v, rtol=0, atol=1e-15)


def test_head_specific_mask_is_refused_by_the_head_chunk_route():
    """R * gqa > 32 makes the verify head-chunk plan apply: a mask over all H
    heads does not fit a head chunk, a broadcast mask does (and the route only
    changes the partition, so its result equals the unchunked one)."""
    spec = _spec(R=8, B=1, H=8, Hk=1)                        # R * gqa = 64 > 32
    plan = orc.head_chunk_plan(spec.q_len, spec.num_heads, spec.num_kv_heads, True)
    assert len(plan) > spec.num_kv_heads                     # the route chunks the heads
    per_head = _random_mask(spec, spec.num_heads, 5)
    with pytest.raises(orc.MaskRouteError):
        _run(spec, per_head, head_chunk=True)
    case, out, ty, ta, kc, vc = _run(spec, per_head, head_chunk=False)
    assert np.allclose(ta, _numpy_attention(spec, case, ty, kc, vc, per_head), rtol=1e-10, atol=1e-12)
    bc = _random_mask(spec, 1, 6)
    _, out_on, _, ta_on, _, _ = _run(spec, bc, head_chunk=True)
    _, out_off, _, ta_off, _, _ = _run(spec, bc, head_chunk=False)
    assert np.allclose(ta_on, ta_off, rtol=1e-12, atol=1e-14)


def test_each_head_of_a_head_specific_mask_sees_its_own_positions():
    spec = _spec(R=1, B=1)
    T = int(spec.positions().max()) + 1
    mask = np.zeros((1, spec.num_heads, 1, T), np.uint8)
    for h in range(spec.num_heads):
        mask[0, h, 0, 2 * h + 1] = 1
    case, out, ty, ta, kc, vc = _run(spec, mask)
    gqa = spec.num_heads // spec.num_kv_heads
    for h in range(spec.num_heads):
        v = bf16_bits_to_f32(vc[0, h // gqa, 2 * h + 1]).astype(np.float64)
        assert np.allclose(ta[0, 0, h], v, rtol=0, atol=1e-15)


@pytest.mark.parametrize("kv", ["bf16", "turbo4v"])
def test_short_mask_rows_equal_zero_padded_rows(kv):
    """Rows shorter than cache_pos + R (the library's mask of `positions`
    bytes per row): the positions past a row are not attended, which is the
    same as the full-length mask with those positions zeroed; a row that
    keeps nothing within its length is a zero row."""
    spec = _spec(R=3, B=2)
    case = make_case(spec)
    x = synth.x_values(spec, case.x)
    full = _random_mask(spec, 1, 21, density=0.7)
    T = int(case.pos.min()) + 1                     # shorter than every sequence's span
    short = np.ascontiguousarray(full[..., :T])
    padded = full.copy()
    padded[..., T:] = 0
    padded[0, 0, 1, :] = 0                          # a row with nothing left ...
    short[0, 0, 1, :] = 0
    turbo = synth.turbo4v_cache(spec, case.cap) if kv == "turbo4v" else None

    def run(mask):
        kc, vc = case.ck.copy(), case.cv.copy()
        tv = None if turbo is None else (turbo[0].copy(), turbo[1].copy())
        return orc.layer_step_ext(spec, case.orc_weights, x, kc, None if tv else vc, case.pos,
                                  turbo=tv, mask=mask, taps=True)

    a_out, _, a_attn = run(short)
    b_out, _, b_attn = run(padded)
    assert np.array_equal(a_out, b_out) and np.array_equal(a_attn, b_attn)
    assert np.all(a_attn[0, 1] == 0.0)              # ... attends nothing
    assert np.any(a_attn[1] != 0.0)
