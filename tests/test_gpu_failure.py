"""A bounded device wait that runs out: reported, survived, and followed by an
exact step.

The projection kernels bound every wait they make (a weight stage landing in
shared memory, a ring slot coming free, partial sums arriving from the other
CTAs of a cluster).  Through a test hook of the C ABI the q|k|v projection's
CTA 0 skips the copy of its last weight stage, under a wait limit of a few
milliseconds: that wait gives up, the kernel finishes its launch without the
stage, and the layer's status word carries the timeout bit.  Nothing here
traps, faults or spins without a bound: the host sees the failure through
gattn_layer_poll_status, the context stays usable, and the next step (hook
off, same cache positions, so the rows the failed step appended are written
again) matches the oracle on the same handle and on a fresh one."""
import time

import numpy as np
import pytest
import torch

from qwen3_gated_attention_gb300 import gattn
from qwen3_gated_attention_gb300.device import DeviceLayer, x_to_device
from tests.cases import make_case, oracle_run
from tests.test_gpu_layer import SMALL, check_parity, gpu_run

pytestmark = pytest.mark.gpu

GATTN_E_DEVICE_TIMEOUT = 6
LIMIT_NS = 3_000_000             # 3 ms


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_gated_attention_gb300 import build
    build.build()


def _failed_step(dl, case):
    spec = case.spec
    out = torch.zeros((spec.batch, spec.q_len, spec.hidden), dtype=torch.bfloat16, device="cuda")
    xd = x_to_device(spec, case.x)
    pd = torch.from_numpy(np.ascontiguousarray(case.pos, np.int32)).cuda()
    torch.cuda.synchronize()
    gattn.layer_set_test_wait(dl.h, LIMIT_NS, True)
    t0 = time.perf_counter()
    dl.step(xd, pd, out)
    code = gattn.layer_poll_status_code(dl.h, torch.cuda.current_stream().cuda_stream)
    elapsed = time.perf_counter() - t0
    gattn.layer_set_test_wait(dl.h, 0, False)
    return code, elapsed


@pytest.mark.parametrize("name", ["decode_4b", "verify_2k_p46"])
def test_a_wait_that_runs_out_is_reported_and_the_next_step_is_exact(name):
    case = make_case(SMALL[name])
    ref = oracle_run(case)
    dl = DeviceLayer(case.spec, case.lib_packed, case.qn, case.kn, case.cap)
    try:
        dl.load_cache(case.ck, case.cv)
        code, elapsed = _failed_step(dl, case)
        assert code == GATTN_E_DEVICE_TIMEOUT, gattn.STATUS_NAMES.get(code, code)
        # the launch waited out the limit and then returned (well under the 2 s default)
        assert LIMIT_NS * 1e-9 <= elapsed < 1.0, elapsed
        # the status word was read and cleared: a clean step reports nothing
        got = gpu_run(case, dl=dl, keep=True)
        check_parity(case, got, ref, what=f"{name}: same handle after the timeout")
    finally:
        dl.close()
    fresh = gpu_run(case)
    check_parity(case, fresh, ref, what=f"{name}: fresh handle after the timeout")


def test_wait_limit_arguments():
    case = make_case(SMALL["tiny"])
    dl = DeviceLayer(case.spec, case.lib_packed, case.qn, case.kn, case.cap)
    try:
        with pytest.raises(gattn.GattnError):
            gattn.layer_set_test_wait(dl.h, -1, False)
        # a generous limit with nothing withheld changes no result
        dl.load_cache(case.ck, case.cv)
        gattn.layer_set_test_wait(dl.h, 500_000_000, False)
        got = gpu_run(case, dl=dl, keep=True)
        check_parity(case, got, oracle_run(case), what="tiny: 0.5 s limit")
    finally:
        dl.close()
