"""Device-memory plumbing around the C ABI: torch owns the buffers (weights in the
interchange layout, bf16 caches, inputs, outputs); every computation goes
through ``gattn.layer_step`` and friends."""
from __future__ import annotations

import numpy as np
import torch

from . import gattn


def _dev_u16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).to(device)


def _dev_u32(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint32).view(np.int32)).to(device)


def cache_strides(layout: str, batch: int, Hk: int, cap: int, d: int):
    """(shape, stride_token, stride_head, stride_batch) in elements."""
    if layout == "bhtd":          # [B][Hk][cap][d]
        return (batch, Hk, cap, d), d, cap * d, Hk * cap * d
    if layout == "btd":           # token-major [B][cap][Hk*d]
        return (batch, cap, Hk, d), Hk * d, d, cap * Hk * d
    raise ValueError(layout)


class DeviceLayer:
    """One layer handle with its weights set and one registered cache: bf16 K/V,
    or (kv_format="turbo4v") bf16 K with Turbo4 V code and E4M3 scale planes
    [B][Hk][cap][d/2] and [B][Hk][cap][d/16] uint8, or (kv_format="turbo4")
    such planes for K and V both."""

    def __init__(self, spec, packed, q_norm, k_norm, capacity, *, batch=None, max_batch=None,
                 max_q_len=None, head_chunk=True, layout="bhtd", device="cuda:0",
                 kv_format="bf16"):
        self.spec = spec
        self.device = torch.device(device)
        self.batch = batch or spec.batch
        self.layout = layout
        self.capacity = capacity
        self.kv_format = kv_format
        self.cfg = gattn.make_cfg(spec.hidden, spec.num_heads, spec.num_kv_heads, spec.head_dim,
                                  spec.partial_rotary_factor, spec.rope_theta, spec.rms_eps,
                                  tuple(spec.bits), tuple(spec.group), x_dtype=spec.x_dtype,
                                  max_batch=max_batch or self.batch,
                                  max_q_len=max_q_len or spec.q_len, head_chunk=head_chunk)
        self.h = gattn.layer_create(self.cfg)
        self.kv = 0
        try:
            self._w = [(_dev_u32(p, self.device), _dev_u16(s, self.device), _dev_u16(b, self.device))
                       for p, s, b in packed]
            self._qn = _dev_u16(q_norm, self.device)
            self._kn = _dev_u16(k_norm, self.device)
            stream = torch.cuda.current_stream(self.device).cuda_stream
            gattn.layer_set_weights(self.h, [(p.data_ptr(), s.data_ptr(), b.data_ptr())
                                             for p, s, b in self._w],
                                    self._qn.data_ptr(), self._kn.data_ptr(), stream)
            Hk, d = spec.num_kv_heads, spec.head_dim
            shape, st, sh, sb = cache_strides(layout, self.batch, Hk, capacity, d)
            self.k = torch.zeros(shape, dtype=torch.bfloat16, device=self.device)
            if kv_format == "turbo4":
                assert layout == "bhtd"
                B = self.batch
                pl = lambda w: torch.zeros((B, Hk, capacity, w), dtype=torch.uint8, device=self.device)
                self.kc, self.ks = pl(d // 2), pl(d // 16)
                self.vc, self.vs = pl(d // 2), pl(d // 16)
                self.kv = gattn.kv_register_turbo4(
                    self.h, self.kc.data_ptr(), self.ks.data_ptr(), self.vc.data_ptr(),
                    self.vs.data_ptr(), B, capacity, (capacity * d // 2, Hk * capacity * d // 2),
                    (capacity * d // 16, Hk * capacity * d // 16))
            elif kv_format == "turbo4v":
                assert layout == "bhtd"
                B = self.batch
                self.vc = torch.zeros((B, Hk, capacity, d // 2), dtype=torch.uint8, device=self.device)
                self.vs = torch.zeros((B, Hk, capacity, d // 16), dtype=torch.uint8,
                                      device=self.device)
                self.kv = gattn.kv_register_turbo4v(
                    self.h, self.k.data_ptr(), self.vc.data_ptr(), self.vs.data_ptr(), B, capacity,
                    (st, sh, sb), (capacity * d // 2, Hk * capacity * d // 2),
                    (capacity * d // 16, Hk * capacity * d // 16))
            else:
                self.v = torch.zeros(shape, dtype=torch.bfloat16, device=self.device)
                self.kv = gattn.kv_register(self.h, self.k.data_ptr(), self.v.data_ptr(),
                                            self.batch, capacity, st, sh, sb)
        except Exception:
            self.close()
            raise

    # caches are exchanged with the host as [B][Hk][cap][d] bf16 bit patterns
    def load_cache(self, k_bits: np.ndarray, v_bits, batches=None):
        """v_bits: bf16 bits [B][Hk][cap][d], or (codes, scales) for a turbo4v cache."""
        idx = list(range(self.batch)) if batches is None else list(batches)
        if self.kv_format == "turbo4":
            (kc, ks), (vc, vs) = k_bits, v_bits
            for j, b in enumerate(idx):
                for dst, src in ((self.kc, kc), (self.ks, ks), (self.vc, vc), (self.vs, vs)):
                    dst[b].copy_(torch.from_numpy(np.ascontiguousarray(src[j], np.uint8)))
            return
        if self.kv_format == "turbo4v":
            codes, scales = v_bits
            for j, b in enumerate(idx):
                self.vc[b].copy_(torch.from_numpy(np.ascontiguousarray(codes[j], np.uint8)))
                self.vs[b].copy_(torch.from_numpy(np.ascontiguousarray(scales[j], np.uint8)))
            pairs = ((self.k, k_bits),)
        else:
            pairs = ((self.k, k_bits), (self.v, v_bits))
        for dst, src in pairs:
            for j, b in enumerate(idx):
                t = _dev_u16(src[j], self.device).view(torch.bfloat16)      # [Hk][cap][d]
                if self.layout == "bhtd":
                    dst[b].copy_(t)
                else:
                    dst[b].copy_(t.transpose(0, 1))

    def read_cache(self, batches=None):
        """(K bits, V bits), or (K bits, (codes, scales)) for a turbo4v cache."""
        idx = list(range(self.batch)) if batches is None else list(batches)
        if self.kv_format == "turbo4":
            g = lambda t: np.stack([t[b].cpu().numpy() for b in idx])
            return (g(self.kc), g(self.ks)), (g(self.vc), g(self.vs))
        if self.kv_format == "turbo4v":
            k = np.stack([self.k[b].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
                          for b in idx])
            return k, (np.stack([self.vc[b].cpu().numpy() for b in idx]),
                       np.stack([self.vs[b].cpu().numpy() for b in idx]))
        outs = []
        for src in (self.k, self.v):
            parts = []
            for b in idx:
                t = src[b] if self.layout == "bhtd" else src[b].transpose(0, 1)
                parts.append(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
            outs.append(np.stack(parts))
        return outs[0], outs[1]

    def step(self, x: torch.Tensor, cache_pos: torch.Tensor, out: torch.Tensor, batch=None,
             q_len=None, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        gattn.layer_step(self.h, x.data_ptr(), self.kv, cache_pos.data_ptr(), batch or self.batch,
                         q_len or self.spec.q_len, out.data_ptr(), s)

    def step_block(self, x: torch.Tensor, cache_pos: torch.Tensor, input_ln: torch.Tensor,
                   post_ln: torch.Tensor | None, out: torch.Tensor,
                   out_normed: torch.Tensor | None = None, batch=None, q_len=None, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        gattn.layer_step_block(self.h, x.data_ptr(), self.kv, cache_pos.data_ptr(),
                               batch or self.batch, q_len or self.spec.q_len, input_ln.data_ptr(),
                               post_ln.data_ptr() if post_ln is not None else None, out.data_ptr(),
                               out_normed.data_ptr() if out_normed is not None else None, s)

    def set_taps(self, y: torch.Tensor | None, attn: torch.Tensor | None):
        gattn.layer_set_taps(self.h, y.data_ptr() if y is not None else None,
                             attn.data_ptr() if attn is not None else None)

    def set_mask(self, mask: torch.Tensor | None):
        """mask: uint8 [B][1 or H][R][T] on the device (None clears it)."""
        if mask is None:
            gattn.layer_set_mask(self.h, None)
            return
        assert mask.dtype == torch.uint8 and mask.dim() == 4 and mask.is_contiguous()
        self._mask = mask
        gattn.layer_set_mask(self.h, mask.data_ptr(), mask.shape[1], mask.shape[3],
                             (mask.stride(2), mask.stride(1), mask.stride(0)))

    def poll(self):
        gattn.layer_poll_status(self.h, torch.cuda.current_stream(self.device).cuda_stream)

    def close(self):
        if getattr(self, "kv", 0):
            gattn.kv_destroy(self.kv)
            self.kv = 0
        if getattr(self, "h", 0):
            gattn.layer_destroy(self.h)
            self.h = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def x_to_device(spec, x: np.ndarray, device="cuda:0") -> torch.Tensor:
    if spec.x_dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)
    return _dev_u16(x, device).view(torch.bfloat16)


def bf16_tensor_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
