"""Steps captured in a CUDA graph and replayed equal the same steps run eagerly,
bit for bit: three consecutive steps (each reading the rows the previous ones
appended) over bf16 and Bf16KTurbo4V caches, and the decoder-block
step.  The step makes no allocation, host synchronization or host-side
decision from device data, so its capture replays the same work."""
import numpy as np
import pytest
import torch

from qwen3_gated_attention_gb300 import gattn, synth
from qwen3_gated_attention_gb300.device import DeviceLayer, x_to_device
from tests.cases import make_case
from tests.test_gpu_block import _u16
from tests.test_gpu_layer import SMALL

pytestmark = pytest.mark.gpu

STEPS = 3


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_gated_attention_gb300 import build
    build.build()


def _run(spec, case, turbo, block, graph):
    B, R, Hd = spec.batch, spec.q_len, spec.hidden
    dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, case.cap,
                     kv_format="turbo4v" if turbo is not None else "bf16")
    try:
        dl.load_cache(case.ck, turbo if turbo is not None else case.cv)
        xs = [x_to_device(spec, synth.layer_input(spec, step=i)) for i in range(STEPS)]
        ps = [torch.from_numpy((case.pos + i * R).astype(np.int32)).cuda() for i in range(STEPS)]
        nan = float("nan")
        outs = [torch.full((B, R, Hd), nan, dtype=torch.bfloat16, device="cuda") for _ in range(STEPS)]
        normed = [torch.full((B, R, Hd), nan, dtype=torch.bfloat16, device="cuda")
                  for _ in range(STEPS)]
        il, pl = synth.block_norm_weights_bf16(spec)
        ild, pld = _u16(il), _u16(pl)
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()

        def enqueue():
            for i in range(STEPS):
                if block:
                    dl.step_block(xs[i], ps[i], ild, pld, outs[i], normed[i],
                                  stream=stream.cuda_stream)
                else:
                    dl.step(xs[i], ps[i], outs[i], stream=stream.cuda_stream)

        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                g.capture_begin()
                enqueue()
                g.capture_end()
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                g.replay()
        else:
            with torch.cuda.stream(stream):
                enqueue()
        stream.synchronize()
        gattn.layer_poll_status(dl.h, stream.cuda_stream)
        cache = dl.read_cache()
        res = [o.view(torch.int16).cpu().numpy() for o in outs]
        if block:
            res += [o.view(torch.int16).cpu().numpy() for o in normed]
        return res, cache
    finally:
        dl.close()


CASES = [("batched_mixed_small", False, False),
         ("verify_2k_p46", False, False),
         ("verify_2k_p46", True, False),
         ("decode_4b", False, True)]


@pytest.mark.parametrize("name,turbo,block", CASES,
                         ids=["-".join(map(str, c)) for c in CASES])
def test_graph_replay_equals_eager_steps(name, turbo, block):
    spec = SMALL[name]
    case = make_case(spec, capacity=spec.capacity() + 64)
    tv = synth.turbo4v_cache(spec, case.cap) if turbo else None
    eager, ec = _run(spec, case, tv, block, graph=False)
    replay, gc = _run(spec, case, tv, block, graph=True)
    for i, (a, b) in enumerate(zip(eager, replay)):
        assert np.array_equal(a, b), f"output {i}"
    ek, ev = ec
    gk, gv = gc
    assert np.array_equal(ek, gk)
    if turbo:
        assert np.array_equal(ev[0], gv[0]) and np.array_equal(ev[1], gv[1])
    else:
        assert np.array_equal(ev, gv)
    # the three steps appended three blocks of rows
    for b in range(spec.batch):
        p = int(case.pos[b])
        assert not np.array_equal(gk[b, :, p:p + STEPS * spec.q_len], case.ck[b, :, p:p + STEPS * spec.q_len])
