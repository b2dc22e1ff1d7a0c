"""Test helpers that pin the oracle from outside it.

* ``decode_codes`` -- vectorised decoder of the packed row bitstream (numpy
  ``unpackbits``), written independently of the oracle's word/shift decoder.
* ``encode_codes`` -- Python big-integer encoder of the same bitstream.
* ``torch_layer`` -- the layer composed from library routines in float64
  (``torch.matmul``, ``F.rms_norm``, complex-exponential rotary,
  ``F.scaled_dot_product_attention`` with GQA, ``torch.sigmoid``).
* ``compare_layer`` -- the comparison every parity test applies.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

from qwen3_gated_attention_gb300.synth import bf16_bits_to_f32


def encode_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes [N][K] -> packed uint32 [N][K*bits/32]: code j at bits [j*bits, (j+1)*bits)."""
    N, K = codes.shape
    words = K * bits // 32
    out = np.zeros((N, words), np.uint32)
    for n in range(N):
        v = 0
        for j, c in enumerate(codes[n].tolist()):
            v |= int(c) << (j * bits)
        for w in range(words):
            out[n, w] = (v >> (32 * w)) & 0xFFFFFFFF
    return out


def decode_codes(packed: np.ndarray, K: int, bits: int) -> np.ndarray:
    N = packed.shape[0]
    raw = np.ascontiguousarray(packed, np.dtype("<u4")).view(np.uint8).reshape(N, -1)
    bitv = np.unpackbits(raw, axis=1, bitorder="little")[:, :K * bits].reshape(N, K, bits)
    weights = (1 << np.arange(bits)).astype(np.int64)
    return (bitv.astype(np.int64) * weights).sum(axis=2)


def dequant_np(packed, scales, biases, K, bits, group) -> np.ndarray:
    q = decode_codes(packed, K, bits).astype(np.float64)
    s = np.repeat(bf16_bits_to_f32(scales).astype(np.float64), group, axis=1)
    b = np.repeat(bf16_bits_to_f32(biases).astype(np.float64), group, axis=1)
    return s * q + b


def rope_complex(x: torch.Tensor, rd: int, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """Rotary as complex multiplication: z_i = x_i + i x_{i+rd/2} times e^{i pos theta^(-2i/rd)};
    x [..., d] float64, pos broadcastable to x[..., 0]."""
    half = rd // 2
    i = torch.arange(half, dtype=torch.float64)
    freq = torch.exp(-torch.log(torch.tensor(theta, dtype=torch.float64)) * 2.0 * i / rd)
    ang = pos[..., None].to(torch.float64) * freq
    z = torch.complex(x[..., :half], x[..., half:rd]) * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([z.real, z.imag, x[..., rd:]], dim=-1)


def to_bf16_values(t: torch.Tensor) -> torch.Tensor:
    """float64 values rounded once to bf16 (nearest, ties to even).  torch takes
    float64 to bfloat16 through float32, which can round twice; a float32
    intermediate rounded to odd (truncated toward zero, last bit set when
    inexact) keeps enough bits for the final float32 -> bfloat16 rounding to be
    the correct single rounding (round-to-odd, Boldo and Melquiond)."""
    x = t.detach().cpu().numpy().astype(np.float64)
    f = x.astype(np.float32)
    over = np.abs(f.astype(np.float64)) > np.abs(x)
    f = np.where(over, np.nextafter(f, np.float32(0)), f).astype(np.float32)
    inexact = f.astype(np.float64) != x
    f = (f.view(np.uint32) | inexact.astype(np.uint32)).view(np.float32)
    return torch.from_numpy(f).to(torch.bfloat16).to(torch.float64)


def torch_layer(spec, Wdeq, qn_w, kn_w, x, cache_k, cache_v, cache_pos):
    """Layer step from library routines, float64.  Wdeq: dequantized [q, k, v, o]
    float64 numpy; qn_w/kn_w float64; x [B][R][Hd]; caches [B][Hk][cap][d] float64
    (values).  Returns (out, y, attn, new_k_rows, new_v_rows)."""
    H, Hk, d, Hd = spec.num_heads, spec.num_kv_heads, spec.head_dim, spec.hidden
    rd = int(d * float(np.float32(spec.partial_rotary_factor)))
    eps = float(np.float32(spec.rms_eps))
    theta = float(np.float32(spec.rope_theta))
    X = torch.from_numpy(np.asarray(x, np.float64))
    B, R, _ = X.shape
    Wq, Wk, Wv, Wo = (torch.from_numpy(w) for w in Wdeq)
    q_full = X @ Wq.T
    k = X @ Wk.T
    v = X @ Wv.T
    y = torch.cat([q_full, k, v], dim=-1)
    qf = q_full.view(B, R, H, 2 * d)
    query, gate = qf[..., :d], qf[..., d:]
    pos = torch.from_numpy(np.asarray(cache_pos, np.int64))[:, None] + torch.arange(R)[None, :]
    qn = F.rms_norm(query, (d,), torch.from_numpy(qn_w), eps)
    kn = F.rms_norm(k.view(B, R, Hk, d), (d,), torch.from_numpy(kn_w), eps)
    qn = rope_complex(qn, rd, pos[:, :, None], theta)
    kn = rope_complex(kn, rd, pos[:, :, None], theta)
    kb, vb = to_bf16_values(kn), to_bf16_values(v.view(B, R, Hk, d))
    Kc = torch.from_numpy(np.array(cache_k, np.float64))
    Vc = torch.from_numpy(np.array(cache_v, np.float64))
    attn = torch.zeros(B, R, H, d, dtype=torch.float64)
    for b in range(B):
        p0 = int(cache_pos[b])
        Kc[b, :, p0:p0 + R] = kb[b].transpose(0, 1)
        Vc[b, :, p0:p0 + R] = vb[b].transpose(0, 1)
        L = p0 + R
        t = torch.arange(L)
        mask = t[None, :] <= (p0 + torch.arange(R))[:, None]          # [R][L]
        o = F.scaled_dot_product_attention(qn[b].transpose(0, 1)[None], Kc[b, :, :L][None],
                                           Vc[b, :, :L][None], attn_mask=mask, enable_gqa=True)
        attn[b] = o[0].transpose(0, 1)
    ga = attn * torch.sigmoid(gate)
    out = ga.reshape(B, R, H * d) @ Wo.T
    return (out.numpy(), y.numpy(), attn.numpy(), kb.numpy(), vb.numpy())


# ------------------------------------------------------------- comparisons

ABS_TOL = 2e-2      # element-wise |g - o| <= ABS_TOL + REL_TOL * |o|
REL_TOL = 1e-2
L2_TOL = 1e-2       # ||g - o|| / ||o|| (derived: bf16 operands and output, ~3e-3 expected)


def close(got, ref, abs_tol=ABS_TOL, rel_tol=REL_TOL, l2_tol=L2_TOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if got.shape != ref.shape:
        return False, f"shape {got.shape} != {ref.shape}"
    if not np.all(np.isfinite(got)):
        return False, "non-finite values"
    err = np.abs(got - ref)
    elem_ok = bool(np.all(err <= abs_tol + rel_tol * np.abs(ref)))
    nref = np.linalg.norm(ref)
    l2 = float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(np.linalg.norm(got))
    ok = elem_ok and l2 <= l2_tol
    return ok, f"max_abs={err.max():.3e} l2_rel={l2:.3e} elem_ok={elem_ok}"


def compare_layer(ref: dict, got: dict, keys=("out", "attn", "y", "k_rows", "v_rows")):
    """ref/got: dicts of arrays.  Returns (all_ok, report)."""
    ok_all, rep = True, []
    for k in keys:
        if k not in ref or k not in got:
            continue
        ok, msg = close(got[k], ref[k])
        ok_all &= ok
        rep.append(f"{k}: {msg}")
    return ok_all, "; ".join(rep)
