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
