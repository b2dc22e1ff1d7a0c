"""Guard bands and resume on the GPU.

Every buffer the step writes (out, out_normed, the taps, the K/V cache or its
Turbo4 planes) sits inside a larger allocation whose bands before and after it
hold a sentinel pattern; after the step each band is unchanged bit for bit and
the results equal those of the same step on exactly sized buffers.  A second
test checks that the only state carried between steps is the caller's cache:
a step taken on a fresh layer handle over a cache that an earlier handle wrote
equals the same step taken on the earlier handle."""
import types

import numpy as np
import pytest
import torch

from qwen3_gated_attention_gb300 import gattn, synth
from qwen3_gated_attention_gb300.device import DeviceLayer, x_to_device
from tests.cases import make_case
from tests.test_gpu_block import _u16
from tests.test_gpu_layer import SMALL

pytestmark = pytest.mark.gpu

GUARD = 4096                 # elements on either side (8 KiB of bf16: keeps 16-byte alignment)
S16, S32, S8 = 0x7FA5, 0x7FC0A5A5, 0xA5


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from qwen3_gated_attention_gb300 import build
    build.build()


class Guarded:
    """A view of n elements with GUARD sentinel elements before and after it."""

    def __init__(self, shape, kind):
        n = int(np.prod(shape))
        if kind == "bf16":
            raw = torch.full((n + 2 * GUARD,), S16, dtype=torch.int16, device="cuda")
            self.buf, self.view = raw, raw[GUARD:GUARD + n].view(torch.bfloat16).view(shape)
        elif kind == "f32":
            raw = torch.full((n + 2 * GUARD,), S32, dtype=torch.int32, device="cuda")
            self.buf, self.view = raw, raw[GUARD:GUARD + n].view(torch.float32).view(shape)
        else:
            raw = torch.full((n + 2 * GUARD,), S8, dtype=torch.uint8, device="cuda")
            self.buf, self.view = raw, raw[GUARD:GUARD + n].view(shape)
        self.n = n
        self.sent = {"bf16": S16, "f32": S32, "u8": S8}[kind]

    def bands_intact(self):
        b = self.buf.cpu().numpy()
        return bool(np.all(b[:GUARD] == b.dtype.type(self.sent)) and
                    np.all(b[GUARD + self.n:] == b.dtype.type(self.sent)))


def _bits(t):
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy()
    if t.dtype == torch.float32:
        return t.contiguous().view(torch.int32).cpu().numpy()
    return t.cpu().numpy()


def _planes(spec, cap, kv_format):
    """Host cache contents for the format: {name: array}."""
    case = make_case(spec, capacity=cap)
    if kv_format == "bf16":
        return case, {"k": case.ck, "v": case.cv}
    vc, vs = synth.turbo4v_cache(spec, cap)
    if kv_format == "turbo4v":
        return case, {"k": case.ck, "vc": vc, "vs": vs}
    kc, ks = synth.turbo4v_cache(spec, cap, plane="k")
    return case, {"kc": kc, "ks": ks, "vc": vc, "vs": vs}


def _register(h, spec, cap, kv_format, bufs):
    Hk, d, B = spec.num_kv_heads, spec.head_dim, spec.batch
    kst = (d, cap * d, Hk * cap * d)
    cst, sst = (cap * d // 2, Hk * cap * d // 2), (cap * d // 16, Hk * cap * d // 16)
    p = {k: v.view.data_ptr() for k, v in bufs.items()}
    if kv_format == "bf16":
        return gattn.kv_register(h, p["k"], p["v"], B, cap, *kst)
    if kv_format == "turbo4v":
        return gattn.kv_register_turbo4v(h, p["k"], p["vc"], p["vs"], B, cap, kst, cst, sst)
    return gattn.kv_register_turbo4(h, p["kc"], p["ks"], p["vc"], p["vs"], B, cap, cst, sst)


def _exact_run(case, host, kv_format, block):
    """The same step on a DeviceLayer's exactly sized buffers."""
    spec = case.spec
    dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, case.cap, kv_format=kv_format)
    try:
        if kv_format == "bf16":
            dl.load_cache(host["k"], host["v"])
        elif kv_format == "turbo4v":
            dl.load_cache(host["k"], (host["vc"], host["vs"]))
        else:
            dl.load_cache((host["kc"], host["ks"]), (host["vc"], host["vs"]))
        res = _step(dl.h, dl.kv, case, block)
        if kv_format == "bf16":
            k, v = dl.read_cache()
            cache = {"k": k, "v": v}
        elif kv_format == "turbo4v":
            k, (vc, vs) = dl.read_cache()
            cache = {"k": k, "vc": vc, "vs": vs}
        else:
            (kc, ks), (vc, vs) = dl.read_cache()
            cache = {"kc": kc, "ks": ks, "vc": vc, "vs": vs}
        return res, cache
    finally:
        dl.close()


def _step(h, kv, case, block, guarded=False):
    spec = case.spec
    B, R, H, Hk, d, Hd = (spec.batch, spec.q_len, spec.num_heads, spec.num_kv_heads,
                          spec.head_dim, spec.hidden)
    mk = (lambda shape, kind: Guarded(shape, kind)) if guarded else \
        (lambda shape, kind: _Plain(shape, kind))
    out = mk((B, R, Hd), "bf16")
    res = {"out": out}
    stream = torch.cuda.current_stream().cuda_stream
    xd = x_to_device(spec, case.x)
    pd = torch.from_numpy(case.pos.astype(np.int32)).cuda()
    if block:
        il, pl = synth.block_norm_weights_bf16(spec)
        on = mk((B, R, Hd), "bf16")
        res["out_normed"] = on
        gattn.layer_set_taps(h, None, None)
        gattn.layer_step_block(h, xd.data_ptr(), kv, pd.data_ptr(), B, R, _u16(il).data_ptr(),
                               _u16(pl).data_ptr(), out.view.data_ptr(), on.view.data_ptr(), stream)
    else:
        ty = mk((B * R, 2 * H * d + 2 * Hk * d), "f32")
        ta = mk((B * R, H * d), "f32")
        res["ty"], res["ta"] = ty, ta
        gattn.layer_set_taps(h, ty.view.data_ptr(), ta.view.data_ptr())
        gattn.layer_step(h, xd.data_ptr(), kv, pd.data_ptr(), B, R, out.view.data_ptr(), stream)
    gattn.layer_poll_status(h, stream)
    torch.cuda.synchronize()
    return res


class _Plain:
    """An exactly sized buffer holding the same sentinel as a Guarded view."""

    def __init__(self, shape, kind):
        n = int(np.prod(shape))
        if kind == "bf16":
            self.view = torch.full((n,), S16, dtype=torch.int16, device="cuda").view(
                torch.bfloat16).view(shape)
        elif kind == "f32":
            self.view = torch.full((n,), S32, dtype=torch.int32, device="cuda").view(
                torch.float32).view(shape)
        else:
            self.view = torch.full((n,), S8, dtype=torch.uint8, device="cuda").view(shape)


GUARD_CASES = [("batched_mixed_small", "bf16", False),
               ("verify_2k_p46", "bf16", False),
               ("verify_2k_p46", "turbo4v", False),
               ("batched_mixed_small", "turbo4", False),
               ("decode_4b", "bf16", True)]


@pytest.mark.parametrize("name,kv_format,block", GUARD_CASES,
                         ids=["-".join(map(str, c)) for c in GUARD_CASES])
def test_writes_stay_inside_their_buffers(name, kv_format, block):
    spec = SMALL[name]
    case, host = _planes(spec, SMALL[name].capacity(), kv_format)
    want, want_cache = _exact_run(case, host, kv_format, block)
    Hk, d, B, cap = spec.num_kv_heads, spec.head_dim, spec.batch, case.cap
    bufs = {}
    for k, a in host.items():
        if k in ("k", "v"):
            g = Guarded((B, Hk, cap, d), "bf16")
            g.view.copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16))
        else:
            g = Guarded(a.shape, "u8")
            g.view.copy_(torch.from_numpy(np.ascontiguousarray(a, np.uint8)))
        bufs[k] = g
    h = gattn.layer_create(_cfg(spec))
    kv = 0
    try:
        dl_w = _weights(h, case)
        kv = _register(h, spec, cap, kv_format, bufs)
        got = _step(h, kv, case, block, guarded=True)
    finally:
        if kv:
            gattn.kv_destroy(kv)
        gattn.layer_destroy(h)
    del dl_w
    for what, g in list(got.items()) + list(bufs.items()):
        assert g.bands_intact(), f"{what}: a write landed outside the buffer"
    for what in got:
        assert np.array_equal(_bits(got[what].view), _bits(want[what].view)), what
    for what, g in bufs.items():
        gb = _bits(g.view)
        assert np.array_equal(gb.view(want_cache[what].dtype), want_cache[what]), what


def _cfg(spec):
    return gattn.make_cfg(spec.hidden, spec.num_heads, spec.num_kv_heads, spec.head_dim,
                          spec.partial_rotary_factor, spec.rope_theta, spec.rms_eps,
                          tuple(spec.bits), tuple(spec.group), x_dtype=spec.x_dtype,
                          max_batch=spec.batch, max_q_len=spec.q_len, head_chunk=True)


def _weights(h, case):
    """Upload the packed weights and norm vectors; returns the tensors to keep alive."""
    w = [(torch.from_numpy(np.ascontiguousarray(p, np.uint32).view(np.int32)).cuda(),
          torch.from_numpy(np.ascontiguousarray(s, np.uint16).view(np.int16)).cuda(),
          torch.from_numpy(np.ascontiguousarray(b, np.uint16).view(np.int16)).cuda())
         for p, s, b in case.lib_packed]
    qn, kn = _u16(case.qn), _u16(case.kn)
    gattn.layer_set_weights(h, [(p.data_ptr(), s.data_ptr(), b.data_ptr()) for p, s, b in w],
                            qn.data_ptr(), kn.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return w, qn, kn


@pytest.mark.parametrize("kv_format", ["bf16", "turbo4v"])
def test_a_fresh_handle_resumes_from_the_cache(kv_format):
    """Two verify steps on one handle; the second again on a new handle over
    the cache the first step left: same output, same cache, bit for bit."""
    spec = SMALL["verify_2k_p46"]
    R = spec.q_len
    case, host = _planes(spec, spec.capacity() + 64, kv_format)
    x2 = synth.layer_input(spec, step=1)
    step2 = types.SimpleNamespace(spec=spec, x=x2, pos=case.pos + R)

    def fresh():
        dl = DeviceLayer(spec, case.lib_packed, case.qn, case.kn, case.cap, kv_format=kv_format)
        return dl

    def load(dl, cache):
        if kv_format == "bf16":
            dl.load_cache(cache["k"], cache["v"])
        else:
            dl.load_cache(cache["k"], (cache["vc"], cache["vs"]))

    def read(dl):
        if kv_format == "bf16":
            k, v = dl.read_cache()
            return {"k": k, "v": v}
        k, (vc, vs) = dl.read_cache()
        return {"k": k, "vc": vc, "vs": vs}

    dl = fresh()
    try:
        load(dl, host)
        _step(dl.h, dl.kv, case, False)
        after1 = read(dl)
        cont = _step(dl.h, dl.kv, step2, False)
        cont_cache = read(dl)
    finally:
        dl.close()
    dl = fresh()
    try:
        load(dl, after1)
        resumed = _step(dl.h, dl.kv, step2, False)
        resumed_cache = read(dl)
    finally:
        dl.close()
    for what in cont:
        assert np.array_equal(_bits(cont[what].view), _bits(resumed[what].view)), what
    for what in cont_cache:
        assert np.array_equal(cont_cache[what], resumed_cache[what]), what
    # the second step appended its rows after the first step's
    for b in range(spec.batch):
        p = int(case.pos[b])
        key = "k"
        assert not np.array_equal(after1[key][b, :, p + R:p + 2 * R], cont_cache[key][b, :, p + R:p + 2 * R])
