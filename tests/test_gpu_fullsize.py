"""Full-size parity of the two largest workloads, in the launch configuration
the bench uses: the 9B-class batched decode (32 sequences, lengths
U{512..8192}) and the long-context mixed-width verify (8 sequences, cache
length 32768, 6-bit g128 q/k/v and 3-bit g32 o_proj).

The oracle computes sampled sequences one by one (every sequence is
independent given the shared weights): the shortest and longest sequence and
two more.  Every sequence is checked for cache integrity (bytes outside the
new rows unchanged) and finite outputs."""
import numpy as np
import pytest
import torch

from qwen3_gated_attention_gb300 import synth
from tests.cases import make_case, oracle_run
from tests.test_gpu_layer import check_parity, gpu_run

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_gated_attention_gb300 import build
    build.build()


def _run(name, sample):
    spec = synth.WORKLOADS[name]
    case = make_case(spec, fill=0x7FC1)            # NaN in every slot past a sequence's end
    got = gpu_run(case)
    assert np.all(np.isfinite(got["out"]))
    R = spec.q_len
    for b in range(spec.batch):
        p = int(case.pos[b])
        for gc, before in ((got["k"], case.ck), (got["v"], case.cv)):
            assert np.array_equal(gc[b, :, :p], before[b, :, :p])
            assert np.array_equal(gc[b, :, p + R:], before[b, :, p + R:])
    idx = sorted(set(sample(case.pos)))
    ref = oracle_run(case, batches=idx)
    rep = check_parity(case, got, ref, batches=idx, what=name)
    print(name, idx, rep)


def test_batched_9b_decode_full_size():
    _run("batched_9b", lambda pos: [int(np.argmin(pos)), int(np.argmax(pos)), 7, 19])


def test_long_verify_mixed_widths_full_size():
    _run("long_verify_mixed", lambda pos: [0, 5])


def test_batched_9b_turbo4v_full_size():
    """The 9B-class batched decode over a Bf16K-Turbo4V cache at full size:
    every sequence keeps its cache outside the new rows (NaN-scale canaries
    past each end included); sampled sequences against the oracle (output,
    attention, K rows, V codes and scales bit for bit where the bf16 V row
    cannot round differently)."""
    import oracle as orc
    from tests import refs
    from tests.test_gpu_layer import assert_rows_close
    from tests.test_gpu_turbo import _near_bf16_midpoint, _run_turbo

    spec = synth.WORKLOADS["batched_9b"]
    case = make_case(spec)
    codes, scales = synth.turbo4v_cache(spec, case.cap)
    got = _run_turbo(spec, case, codes.copy(), scales.copy())
    assert np.all(np.isfinite(got["out"]))
    R = spec.q_len
    for b in range(spec.batch):
        p = int(case.pos[b])
        for g, before in ((got["codes"], codes), (got["scales"], scales), (got["k"], case.ck)):
            assert np.array_equal(g[b, :, :p], before[b, :, :p])
            assert np.array_equal(g[b, :, p + R:], before[b, :, p + R:])
    idx = sorted({int(np.argmin(case.pos)), int(np.argmax(case.pos)), 7, 19})
    sub = spec.with_(batch=len(idx))
    kc = np.ascontiguousarray(case.ck[idx]).copy()
    oc = np.ascontiguousarray(codes[idx]).copy()
    os_ = np.ascontiguousarray(scales[idx]).copy()
    xs = np.ascontiguousarray(synth.x_values(spec, case.x)[idx])
    out, ty, ta = orc.layer_step_turbo4v(sub, case.orc_weights, xs, kc, oc, os_,
                                         np.ascontiguousarray(case.pos[idx]), taps=True)
    ok, rep = refs.close(got["out"][idx], out)
    assert ok, f"out: {rep}"
    ok, rep = refs.close(got["attn"][idx], ta)
    assert ok, f"attention: {rep}"
    H, Hk, d = spec.num_heads, spec.num_kv_heads, spec.head_dim
    off = 2 * H * d + Hk * d
    exact = 0
    for j, b in enumerate(idx):
        p = int(case.pos[b])
        assert_rows_close(got["k"][b, :, p:p + R], kc[j, :, p:p + R], "batched_9b turbo k")
        for r in range(R):
            vr = ty[j, r, off:off + Hk * d].reshape(Hk, d)
            for kh in range(Hk):
                if _near_bf16_midpoint(vr[kh]).any():
                    continue
                assert np.array_equal(got["codes"][b, kh, p + r], oc[j, kh, p + r])
                assert np.array_equal(got["scales"][b, kh, p + r], os_[j, kh, p + r])
                exact += 1
    assert exact > 0
    print("batched_9b turbo4v", idx, rep, "exact V rows", exact)


def test_wide_verify_r32_full_size():
    """The 2K-context verify at 32 new rows (the head-chunk route's widest
    case: one head per chunk) at full size."""
    _run("verify_2k_r32", lambda pos: [0])
