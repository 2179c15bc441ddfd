"""Library-routine restatements used to pin the oracle (test code only).

Every function here reaches its result through library routines (torch's
float8/bfloat16 casts, einsum, softmax, logsumexp, topk, numpy indexing) and
none of the oracle's code, so agreement with the oracle on special cases pins
the oracle to something other than itself.
"""
from __future__ import annotations

import numpy as np
import torch


def e4m3_to_f64(codes) -> torch.Tensor:
    t = torch.as_tensor(np.ascontiguousarray(codes)).to(torch.uint8)
    return t.view(torch.float8_e4m3fn).to(torch.float64)


def bf16_to_f64(bits) -> torch.Tensor:
    t = torch.as_tensor(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float64)


def dequant_records(records, Dn: int, Dr: int, sb: int) -> torch.Tensor:
    """[n, rec] uint8 records -> [n, Dn+Dr] float64 via library casts."""
    rec = np.ascontiguousarray(records)
    n = rec.shape[0]
    nblk = (Dn + sb - 1) // sb
    nope = e4m3_to_f64(rec[:, :Dn])
    rope = bf16_to_f64(rec[:, Dn:Dn + 2 * Dr].copy().view(np.uint16))
    scales = torch.as_tensor(rec[:, Dn + 2 * Dr:Dn + 2 * Dr + 4 * nblk].copy().view(np.float32)).to(torch.float64)
    per_dim = scales.repeat_interleave(sb, dim=1)[:, :Dn]
    return torch.cat([nope * per_dim, rope], dim=1).reshape(n, Dn + Dr)


def softmax_attention_with_sink(q_bf16_bits, sink, scale, X):
    """q [H,D] bf16 bits, sink [H], X [n,D] float64 -> (o [H,D], lse [H]).
    The sink is an extra logit with a zero value vector: the textbook softmax
    over [sink, z_1..z_n] applied to [0, x_1..x_n]."""
    q = bf16_to_f64(q_bf16_bits)
    z = scale * (q @ X.T)                                   # [H, n]
    s = torch.as_tensor(np.asarray(sink, dtype=np.float32)).to(torch.float64)[:, None]
    logits = torch.cat([s, z], dim=1)
    p = torch.softmax(logits, dim=1)[:, 1:]
    o = p @ X
    lse = torch.logsumexp(logits, dim=1)
    return o, lse


def make_records(rng: np.random.Generator, n: int, Dn: int, Dr: int, sb: int, spread: float = 1.0):
    """n random records in the layout [Dn e4m3 | Dr bf16 | nblk f32 scales]."""
    nblk = (Dn + sb - 1) // sb
    rec_bytes = Dn + 2 * Dr + 4 * nblk
    x = torch.as_tensor(rng.standard_normal((n, Dn + Dr)) * spread, dtype=torch.float32)
    codes, scales = [], []
    for i in range(nblk):
        xb = x[:, i * sb:min(Dn, (i + 1) * sb)]
        amax = xb.abs().amax(dim=1, keepdim=True)
        s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        codes.append((xb / s).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8))
        scales.append(s)
    rec = torch.cat([torch.cat(codes, 1),
                     x[:, Dn:].to(torch.bfloat16).contiguous().view(torch.uint8),
                     torch.cat(scales, 1).contiguous().view(torch.uint8)], dim=1)
    assert rec.shape[1] == rec_bytes
    return rec.numpy().copy()


def random_bf16_bits(rng: np.random.Generator, shape) -> np.ndarray:
    x = torch.as_tensor(rng.standard_normal(shape), dtype=torch.float32).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16).copy()
