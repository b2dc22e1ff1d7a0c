"""Parity of the CUDA library (through the C ABI) with the float64 oracle.

Tolerances (stated for the layer's bf16 output and the fp32 taps):
element-wise |gpu - oracle| <= 2e-2 + 1e-2 |oracle| and ||gpu - oracle|| /
||oracle|| <= 1e-2; appended cache rows within 1 bf16 ulp (near-zero elements:
within one ulp plus 1e-5 of the row RMS, the fp32 accumulation error of the
projection); every other cache byte unchanged; codes and dequantized weights
bit-exact."""
import numpy as np
import pytest
import torch

import oracle as orc
from qwen3_gated_attention_gb300 import gattn, synth
from qwen3_gated_attention_gb300.device import DeviceLayer, x_to_device
from qwen3_gated_attention_gb300.synth import bf16_bits_to_f32
from tests import refs
from tests.cases import bf16_ulp_distance, make_case, oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_gated_attention_gb300 import build
    build.build()
    torch.cuda.init()


def gpu_run(case, head_chunk=True, layout="bhtd", taps=True, pos=None, x=None, q_len=None,
            batch=None, dl=None, keep=False):
    spec = case.spec
    own = dl is None
    if own:
        dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, case.cap,
                         head_chunk=head_chunk, layout=layout)
        dl.load_cache(case.ck, case.cv)
    B = batch or spec.batch
    R = q_len or spec.q_len
    xx = case.x if x is None else x
    pp = case.pos if pos is None else pos
    H, Hk, d, Hd = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.hidden
    Ny = 2 * H * d + 2 * Hk * d
    ty = torch.full((B * R, Ny), float("nan"), device="cuda") if taps else None
    ta = torch.full((B * R, H * d), float("nan"), device="cuda") if taps else None
    dl.set_taps(ty, ta)
    out = torch.full((B, R, Hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    xd = x_to_device(spec, xx)
    pd = torch.from_numpy(np.ascontiguousarray(pp, np.int32)).cuda()
    dl.step(xd, pd, out, batch=B, q_len=R)
    dl.poll()
    k, v = dl.read_cache()
    res = dict(out=out.float().cpu().numpy().astype(np.float64), k=k, v=v,
               launches=gattn.layer_launches_per_step(dl.h),
               kernels=gattn.layer_step_kernels(dl.h))
    if taps:
        res["y"] = ty.cpu().numpy().astype(np.float64).reshape(B, R, Ny)
        res["attn"] = ta.cpu().numpy().astype(np.float64).reshape(B, R, H, d)
    if own and not keep:
        dl.close()
    elif keep:
        res["dl"] = dl
    return res


def assert_rows_close(rows_g, rows_r, what):
    """Appended bf16 cache rows: within one bf16 ulp; near-zero elements, where
    the fp32 dot product over K terms may move a tiny value by more than its own
    ulp, within one ulp plus 1e-5 of the row's RMS (fp32 accumulation error)."""
    ulp = bf16_ulp_distance(rows_g, rows_r)
    if ulp.max() <= 1:
        return
    vg = bf16_bits_to_f32(rows_g).astype(np.float64)
    vr = bf16_bits_to_f32(rows_r).astype(np.float64)
    rms = np.sqrt(np.mean(vr ** 2, axis=-1, keepdims=True))
    ulp_r = np.abs(vr) * 2.0 ** -7 + 1e-38
    bad = np.abs(vg - vr) > ulp_r + 1e-5 * rms
    worst = np.unravel_index(np.argmax(ulp), ulp.shape)
    assert not bad.any(), (f"{what} rows differ by {ulp.max()} ulp at {worst}: "
                           f"{vg[worst]} vs {vr[worst]}")


def check_parity(case, got, ref, batches=None, what=""):
    spec = case.spec
    R = spec.q_len
    idx = list(range(spec.batch)) if batches is None else list(batches)
    g = dict(out=got["out"][idx], y=got["y"][idx], attn=got["attn"][idx])
    ok, rep = refs.compare_layer(ref, g, keys=("out", "attn", "y"))
    assert ok, f"{what}: {rep}"
    pos = case.pos[idx]
    gk, gv = got["k"][idx], got["v"][idx]
    for name, gc, rc, before in (("k", gk, ref["k"], case.ck[idx]), ("v", gv, ref["v"], case.cv[idx])):
        for j in range(len(idx)):
            p = int(pos[j])
            assert_rows_close(gc[j, :, p:p + R], rc[j, :, p:p + R], f"{what}: {name}")
            mask = np.ones(gc.shape[1:3], bool)
            mask[:, p:p + R] = False
            assert np.array_equal(gc[j][mask], before[j][mask]), f"{what}: {name} cache bytes changed"
    return rep


SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    "decode_4b": synth.WORKLOADS["decode_4b"],
    "verify_2k_p46": synth.WORKLOADS["verify_2k_p46"],
    "verify_2k_p2048": synth.WORKLOADS["verify_2k_p2048"],
    # several sequences with ragged lengths, mixed 6-/3-bit widths, head_dim 64
    "batched_mixed_small": synth.WORKLOADS["tiny"].with_(
        name="batched_mixed_small", batch=3, q_len=2, cache_pos=None, length_range=(20, 300),
        bits=(6, 6, 6, 3), group=(128, 128, 128, 32), x_dtype="bf16"),
    # head_dim 128, 5-bit q/k/v and 2-bit o, four rows, gqa 6
    "d128_b5_b2": synth.LayerSpec(
        name="d128_b5_b2", hidden=512, num_heads=12, num_kv_heads=2, head_dim=128,
        partial_rotary_factor=0.5, rope_theta=1e6, rms_eps=1e-6, bits=(5, 5, 5, 2),
        group=(32, 32, 32, 64), batch=2, q_len=4, x_dtype="f32", length_range=(70, 200)),
    # eight sequences of one row each, 8-bit, 4 query heads per KV head
    "batch8_decode": synth.WORKLOADS["decode_4b"].with_(
        name="batch8_decode", hidden=1024, num_heads=8, num_kv_heads=2, batch=8, cache_pos=None,
        length_range=(1, 700)),
}

# Head layouts the configuration check admits beyond the workloads: k and v
# blocks of the concatenated q|k|v rows that start inside a 128-row block
# (num_kv_heads * head_dim not a multiple of 128), one query head per KV head
# (gqa 1, MHA), and full or half rotation at head_dim 256 (partial_rotary_factor
# 1.0 and 0.5; mlxd #99 admits any factor in (0, 1]).
ADMITTED = {
    "h6_hk3_d64": synth.WORKLOADS["tiny"].with_(
        name="h6_hk3_d64", hidden=384, num_heads=6, num_kv_heads=3, batch=2, q_len=1,
        cache_pos=None, length_range=(20, 200), x_dtype="bf16"),
    "h2_hk1_d64": synth.WORKLOADS["tiny"].with_(
        name="h2_hk1_d64", hidden=256, num_heads=2, num_kv_heads=1, bits=(8,) * 4, group=(32,) * 4,
        q_len=3, cache_pos=(100,), x_dtype="bf16"),
    "mha_h4_d128": synth.LayerSpec(
        name="mha_h4_d128", hidden=512, num_heads=4, num_kv_heads=4, head_dim=128,
        partial_rotary_factor=0.5, rope_theta=1e6, rms_eps=1e-6, bits=(4,) * 4, group=(64,) * 4,
        batch=2, q_len=2, x_dtype="bf16", length_range=(10, 300)),
    "prf1_d256": synth.WORKLOADS["decode_4b"].with_(
        name="prf1_d256", hidden=1024, num_heads=4, num_kv_heads=2, partial_rotary_factor=1.0,
        bits=(4,) * 4, group=(128,) * 4, cache_pos=(500,)),
    "prf05_d256": synth.WORKLOADS["decode_4b"].with_(
        name="prf05_d256", hidden=1024, num_heads=4, num_kv_heads=2, partial_rotary_factor=0.5,
        bits=(4,) * 4, group=(64,) * 4, q_len=4, cache_pos=(300,)),
}


@pytest.mark.parametrize("name", list(ADMITTED))
def test_admitted_head_layouts_parity(name):
    case = make_case(ADMITTED[name])
    ref = oracle_run(case)
    for chunk in (True, False):
        got = gpu_run(case, head_chunk=chunk)
        rep = check_parity(case, got, ref, what=f"{name} chunk={chunk}")
        print(name, chunk, rep)


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_parity(name):
    case = make_case(SMALL[name])
    got = gpu_run(case)
    # the q|k|v kernel converts x itself when its tables fit, else x prep runs first
    assert got["kernels"][-4:] == ["proj_qkv", "attn", "merge", "proj_o"]
    assert got["launches"] == len(got["kernels"])
    ref = oracle_run(case)
    rep = check_parity(case, got, ref, what=name)
    print(name, rep)


# Wider verify / short prefill rows: q_len 8, 16 and 32 on the verify layer
# (gqa 12), where the head-chunk plan cuts each KV group into 4, 2 and 1 head(s)
# per chunk; a 32-row step spans several 64-row attention row blocks unchunked.
WIDE = {
    "verify_r8": synth.WORKLOADS["verify_2k_p46"].with_(name="verify_r8", q_len=8, cache_pos=(300,)),
    "verify_r16_b2": synth.WORKLOADS["verify_2k_p46"].with_(
        name="verify_r16_b2", q_len=16, batch=2, cache_pos=None, length_range=(40, 700)),
    "verify_r32": synth.WORKLOADS["verify_2k_p46"].with_(name="verify_r32", q_len=32,
                                                        cache_pos=(1000,)),
}


@pytest.mark.parametrize("name", list(WIDE))
def test_wide_verify_rows(name):
    case = make_case(WIDE[name])
    ref = oracle_run(case)
    runs = {}
    for chunk in (True, False):
        got = runs[chunk] = gpu_run(case, head_chunk=chunk)
        rep = check_parity(case, got, ref, what=f"{name} chunk={chunk}")
        print(name, chunk, rep)
    # the head-chunk route changes only the head partition: bit for bit equal
    assert np.array_equal(runs[True]["attn"], runs[False]["attn"])
    assert np.array_equal(runs[True]["out"], runs[False]["out"])


@pytest.mark.parametrize("name", ["verify_2k_p46", "verify_2k_p2048", "d128_b5_b2"])
def test_head_chunk_route_agrees_with_unchunked(name):
    case = make_case(SMALL[name])
    assert len(gattn.head_chunk_plan(case.spec.q_len, case.spec.num_heads,
                                     case.spec.num_kv_heads)) > case.spec.num_kv_heads or name == "d128_b5_b2"
    on = gpu_run(case, head_chunk=True)
    off = gpu_run(case, head_chunk=False)
    ref = oracle_run(case)
    check_parity(case, on, ref, what="chunked")
    check_parity(case, off, ref, what="unchunked")
    # the two routes differ only in how heads are grouped into segments: every
    # segment is cut at the same tokens and a row's arithmetic does not depend
    # on the other rows of its segment, so the results are equal bit for bit
    # (DS4Server issue 113 closing comment: all results match the raw bits)
    assert np.array_equal(on["attn"], off["attn"])
    assert np.array_equal(on["out"], off["out"])
    assert np.array_equal(on["y"], off["y"])
    assert np.array_equal(on["k"], off["k"]) and np.array_equal(on["v"], off["v"])


def test_token_major_cache_layout():
    case = make_case(SMALL["batched_mixed_small"])
    a = gpu_run(case, layout="bhtd")
    b = gpu_run(case, layout="btd")
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["k"], b["k"]) and np.array_equal(a["v"], b["v"])


def test_stale_nan_cache_slots_do_not_leak():
    spec = SMALL["batched_mixed_small"]
    a = gpu_run(make_case(spec, fill=0x3F80))
    b = gpu_run(make_case(spec, fill=0x7FC1))        # NaN past each sequence's end
    assert np.all(np.isfinite(b["out"]))
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["attn"], b["attn"])


def test_verify_step_equals_row_by_row_steps():
    """Four one-row steps on one layer (each reads the rows the previous ones
    appended) equal one four-row step, and every step leaves the layer's
    counters ready for the next."""
    spec = SMALL["verify_2k_p46"]
    case = make_case(spec)
    full = gpu_run(case)
    s1 = spec.with_(q_len=1)
    dl = DeviceLayer(s1, case.lib_packed, case.qn, case.kn, case.cap, max_q_len=1)
    dl.load_cache(case.ck, case.cv)
    case1 = make_case(s1, capacity=case.cap)
    rows = []
    for r in range(spec.q_len):
        res = gpu_run(case1, x=np.ascontiguousarray(case.x[:, r:r + 1]), pos=case.pos + r, dl=dl,
                      q_len=1)
        rows.append(res)
    dl.close()
    assert np.array_equal(rows[-1]["k"], full["k"]) and np.array_equal(rows[-1]["v"], full["v"])
    for r in range(spec.q_len):
        ok, rep = refs.close(rows[r]["out"][:, 0], full["out"][:, r])
        assert ok, rep


def test_batch_equals_solo_calls():
    spec = SMALL["batch8_decode"]
    case = make_case(spec)
    full = gpu_run(case)
    for b in (0, 3, 7):
        sb = spec.with_(batch=1)
        cb = make_case(sb, capacity=case.cap, with_cache=False)
        cb.ck, cb.cv = case.ck[b:b + 1], case.cv[b:b + 1]
        cb.pos, cb.x = case.pos[b:b + 1], case.x[b:b + 1]
        solo = gpu_run(cb)
        ok, rep = refs.close(solo["out"][0], full["out"][b])
        assert ok, rep
        assert np.array_equal(solo["k"][0], full["k"][b])


def test_capacity_overflow_is_reported_and_skipped():
    spec = SMALL["batched_mixed_small"]
    case = make_case(spec)
    good = gpu_run(case)
    bad_pos = case.pos.copy()
    bad_pos[1] = case.cap - spec.q_len + 1          # would write past the capacity
    dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, case.cap)
    dl.load_cache(case.ck, case.cv)
    out = torch.full((spec.batch, spec.q_len, spec.hidden), 7.0, dtype=torch.bfloat16, device="cuda")
    dl.step(x_to_device(spec, case.x), torch.from_numpy(bad_pos).cuda(), out)
    code = gattn.layer_poll_status_code(dl.h, torch.cuda.current_stream().cuda_stream)
    assert code == 4                                  # GATTN_E_DEVICE_RANGE
    k, v = dl.read_cache()
    dl.close()
    o = out.float().cpu().numpy()
    assert np.all(o[1] == 0.0)
    assert np.array_equal(k[1], case.ck[1]) and np.array_equal(v[1], case.cv[1])
    for b in (0, 2):
        ok, rep = refs.close(o[b], good["out"][b])
        assert ok, rep
        assert np.array_equal(k[b], good["k"][b])


@pytest.mark.parametrize("name", ["tiny", "decode_4b", "batched_mixed_small", "d128_b5_b2",
                                  "h6_hk3_d64", "h2_hk1_d64"])
def test_dequant_from_tile_layout_is_bit_exact(name):
    """Both dequant entry points (the allocating one and the static-scratch
    one) against the oracle; the two d64 layouts start their v rows inside a
    128-row block."""
    spec = SMALL.get(name) or ADMITTED[name]
    case = make_case(spec, with_cache=False)
    dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, 64)
    Ks = [spec.hidden] * 3 + [spec.num_heads * spec.head_dim]
    Ns = [spec.n_q, spec.n_kv, spec.n_kv, spec.hidden]
    for p in range(4):
        w = torch.empty((Ns[p], Ks[p]), dtype=torch.float32, device="cuda")
        gattn.layer_dequant_device(dl.h, p, w.data_ptr())
        W = case.orc_weights
        ref = orc.dequantize(W.packed[p], W.scales[p], W.biases[p], Ns[p], Ks[p], spec.bits[p],
                             spec.group[p]).astype(np.float32)
        assert np.array_equal(w.cpu().numpy(), ref), f"projection {p}"
        if Ns[p] * Ks[p] <= (1 << 20):
            ws = torch.full_like(w, float("nan"))
            gattn.layer_dequant_device_static(dl.h, p, ws.data_ptr())
            torch.cuda.synchronize()
            assert np.array_equal(ws.cpu().numpy(), ref), f"projection {p} (static scratch)"
    dl.close()


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 6, 8])
def test_unpack_codes_device_is_bit_exact(bits):
    rng = np.random.default_rng(bits)
    N, K = 37, 256
    w = rng.standard_normal((N, K)).astype(np.float32)
    packed, _, _ = gattn.pack_affine_host(w, bits, 32)
    pd = torch.from_numpy(packed.view(np.int32)).cuda()
    codes = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    gattn.unpack_codes_device(pd.data_ptr(), N, K, bits, codes.data_ptr())
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), orc.unpack_codes(packed, N, K, bits))
