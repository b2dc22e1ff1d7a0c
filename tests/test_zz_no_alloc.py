"""The allocation-free dequant entry point (gattn_layer_dequant_device_static).

Callers that cannot allocate device memory at the point of the call (graph
capture in global mode, a framework-owned memory pool, latency-sensitive
paths) use this entry point instead of gattn_layer_dequant_device.  These
tests call it through the C ABI and check it against the allocating entry
point bit for bit (the tolerance every dequant test here uses), on calls made
back to back: the fixed staging array keeps the previous call's contents, so a
second call must not depend on them.  Collected last on purpose, so that a run
stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle as orc
from qwen3_gated_attention_gb300 import gattn, synth
from qwen3_gated_attention_gb300.device import DeviceLayer
from tests.cases import make_case

pytestmark = pytest.mark.gpu

SPECS = {
    "tiny": synth.WORKLOADS["tiny"],
    # 5-bit q/k/v, 2-bit o, head_dim 128 (the o projection spans several row blocks)
    "d128_b5_b2": synth.LayerSpec(
        name="d128_b5_b2", hidden=512, num_heads=12, num_kv_heads=2, head_dim=128,
        partial_rotary_factor=0.5, rope_theta=1e6, rms_eps=1e-6, bits=(5, 5, 5, 2),
        group=(32, 32, 32, 64), batch=2, q_len=4, x_dtype="f32", length_range=(70, 200)),
    # one KV head of head_dim 64: the q rows fill two 128-row blocks, k takes the
    # first half of the third and v starts 64 rows into it, so the copy out of
    # the staging array begins inside a row block
    "h2_hk1_d64": synth.WORKLOADS["tiny"].with_(
        name="h2_hk1_d64", hidden=256, num_heads=2, num_kv_heads=1, bits=(8,) * 4,
        group=(32,) * 4, x_dtype="bf16"),
}


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_gated_attention_gb300 import build
    build.build()


def _layer(spec):
    wf = synth.weights_f32(spec)
    packed = [gattn.pack_affine_host(w, spec.bits[i], spec.group[i]) for i, w in enumerate(wf)]
    qn, kn = synth.norm_weights_bf16(spec)
    return DeviceLayer(spec, packed, qn, kn, 64)


def _shape(spec, p):
    Ns = [spec.n_q, spec.n_kv, spec.n_kv, spec.hidden]
    Ks = [spec.hidden] * 3 + [spec.num_heads * spec.head_dim]
    return Ns[p], Ks[p]


@pytest.mark.parametrize("name", list(SPECS))
def test_static_dequant_matches_allocating_entry_point(name):
    spec = SPECS[name]
    dl = _layer(spec)
    orc_w = make_case(spec, with_cache=False).orc_weights if name == "h2_hk1_d64" else None
    stream = torch.cuda.current_stream().cuda_stream
    try:
        # two passes over all projections, back to back on one stream: every
        # call reuses the staging array left behind by a different projection
        for _ in range(2):
            for p in (0, 3, 1, 2):
                N, K = _shape(spec, p)
                ref = torch.empty((N, K), dtype=torch.float32, device="cuda")
                got = torch.full((N, K), float("nan"), dtype=torch.float32, device="cuda")
                gattn.layer_dequant_device(dl.h, p, ref.data_ptr(), stream)
                gattn.layer_dequant_device_static(dl.h, p, got.data_ptr(), stream)
                torch.cuda.synchronize()
                assert torch.equal(got, ref), f"projection {p}"
                if name == "h2_hk1_d64":
                    W = orc_w
                    want = orc.dequantize(W.packed[p], W.scales[p], W.biases[p], N, K,
                                          spec.bits[p], spec.group[p]).astype(np.float32)
                    assert np.array_equal(got.cpu().numpy(), want), f"projection {p} vs oracle"
    finally:
        dl.close()


def test_static_dequant_rejects_projections_beyond_its_limit():
    spec = synth.WORKLOADS["decode_4b"]      # q_proj: 8192 x 2560 floats > 4 Mi
    dl = _layer(spec)
    try:
        out = torch.empty((spec.n_q, spec.hidden), dtype=torch.float32, device="cuda")
        with pytest.raises(gattn.GattnError) as ei:
            gattn.layer_dequant_device_static(dl.h, 0, out.data_ptr())
        assert ei.value.status == 2
        assert "static scratch" in str(ei.value)
    finally:
        dl.close()
