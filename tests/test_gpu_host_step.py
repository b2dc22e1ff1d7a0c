"""gattn_layer_step_host: the step from host buffers (x and cache_pos copied in
by the library, out copied back) gives bit for bit the output and cache rows of
gattn_layer_step on the same inputs, across consecutive steps whose cache
positions change (each step reads the positions its own call copied), and
matches the oracle."""
import numpy as np
import pytest
import torch

from qwen3_gated_attention_gb300 import gattn
from qwen3_gated_attention_gb300.device import DeviceLayer, x_to_device
from tests.cases import make_case, oracle_run
from tests.test_gpu_layer import SMALL, check_parity, gpu_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_gated_attention_gb300 import build
    build.build()


def _x_host(spec, x):
    xd = x_to_device(spec, x)
    raw = xd.view(torch.int16) if xd.dtype == torch.bfloat16 else xd
    return xd, raw.cpu().pin_memory()


@pytest.mark.parametrize("name", ["decode_4b", "verify_2k_p46", "batched_mixed_small"])
def test_host_step_equals_device_step(name):
    # room past the spec's cache for the two further steps
    case = make_case(SMALL[name], capacity=SMALL[name].capacity() + 64)
    spec = case.spec
    shape = (spec.batch, spec.q_len, spec.hidden)
    a = DeviceLayer(case.spec, case.lib_packed, case.qn, case.kn, case.cap)
    b = DeviceLayer(case.spec, case.lib_packed, case.qn, case.kn, case.cap)
    try:
        a.load_cache(case.ck, case.cv)
        b.load_cache(case.ck, case.cv)
        xd, xh = _x_host(spec, case.x)
        s = torch.cuda.current_stream().cuda_stream
        for step in range(3):
            # consecutive steps: positions move on, each step's rows are appended
            pos = np.ascontiguousarray(case.pos + step * spec.q_len, np.int32)
            pd = torch.from_numpy(pos).cuda()
            ph = torch.from_numpy(pos).pin_memory()
            out_d = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
            out_h = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
            a.step(xd, pd, out_d)
            gattn.layer_step_host(b.h, xh.data_ptr(), b.kv, ph.data_ptr(), spec.batch, spec.q_len,
                                  out_h.data_ptr(), s)
            torch.cuda.synchronize()
            assert torch.equal(out_d.cpu().view(torch.int16), out_h.view(torch.int16)), step
            if step == 0:
                first = out_h.clone()
        gattn.layer_poll_status(a.h, s)
        gattn.layer_poll_status(b.h, s)
        ka, va = a.read_cache()
        kb, vb = b.read_cache()
        assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    finally:
        a.close()
        b.close()
    # the first step is the parity-tested single step, bit for bit
    fresh = gpu_run(case)
    check_parity(case, fresh, oracle_run(case), what=f"{name} host step")
    assert np.array_equal(first.float().numpy().astype(np.float64), fresh["out"])


def test_host_step_arguments():
    case = make_case(SMALL["tiny"])
    spec = case.spec
    dl = DeviceLayer(case.spec, case.lib_packed, case.qn, case.kn, case.cap)
    try:
        xd, xh = _x_host(spec, case.x)
        ph = torch.from_numpy(np.ascontiguousarray(case.pos, np.int32)).pin_memory()
        out_h = torch.empty((spec.batch, spec.q_len, spec.hidden), dtype=torch.bfloat16).pin_memory()
        with pytest.raises(gattn.GattnError):
            gattn.layer_step_host(dl.h, None, dl.kv, ph.data_ptr(), spec.batch, spec.q_len,
                                  out_h.data_ptr(), 0)
        with pytest.raises(gattn.GattnError):
            gattn.layer_step_host(dl.h, xh.data_ptr(), dl.kv, ph.data_ptr(), 0, spec.q_len,
                                  out_h.data_ptr(), 0)
    finally:
        dl.close()
