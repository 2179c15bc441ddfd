"""The attention's arithmetic precision, chosen on measured error.

"DSV4 Audit" §B1 proposes feeding the FP8 nope codes to the FMHA directly and
quantising q to FP8 (FP8 x FP8 MMAs), and leaves the rope dims' precision to a
cosine check. The attention here instead dequantises the nope codes in shared
memory to BF16 (code x block multiplier, rounded once) and runs QK and PV as
BF16 MMAs. This file records why, on the headline workloads' shapes and
distributions: each variant is emulated exactly at its rounding points (E4M3 /
BF16 round-to-nearest-even through torch's casts; everything else in fp64,
standing in for the tensor core's fp32 accumulation) and compared with the
oracle under the attention gate (per-head cosine >= 0.999 and per-head max
relative error <= 2e-2):

* BF16 latent, BF16 P (the built kernel): passes with a wide margin;
* q in E4M3 (one scale per head and 128-dim block): fails the max relative
  error gate at every candidate count (the 3-bit mantissa moves each score by
  a few per cent of its spread);
* P in E4M3 (with the block multiplier folded in, one scale per head):
  fails it too;
* q as the sum of two E4M3 terms (hi + residual) passes, as accurately as
  BF16, but the keys' per-128-dim fp32 multipliers then need one accumulator
  per block for QK (5 x 64 TMEM columns per 64-candidate chunk beside the
  256-column output), which the tensor memory does not hold.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

SCALE = 1.0 / math.sqrt(512)
BLOCKS = [slice(0, 128), slice(128, 256), slice(256, 384), slice(384, 448)]
GATE_COS, GATE_REL = 0.999, 2e-2


def _cast(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).float().to(dtype).double().numpy()


def _decode(rec):
    codes = torch.from_numpy(rec[:, :448].copy()).view(torch.float8_e4m3fn).double().numpy()
    rope = torch.from_numpy(rec[:, 448:576].copy()).view(torch.bfloat16).double().numpy()
    mult = rec[:, 576:592].copy().view(np.float32).astype(np.float64)
    return codes, rope, mult


def _e4m3_scaled(x, axis=1):
    """x rounded to E4M3 with one scale per slice along ``axis`` (amax / 448)."""
    s = np.abs(x).max(axis=axis, keepdims=True) / 448.0
    s[s == 0] = 1.0
    return _cast(x / s, torch.float8_e4m3fn) * s


def _emulate(q, sink, rec, q_fp8=False, q_two_terms=False, p_fp8=False):
    """Sink-merged attention of one query over ``rec`` with the variant's
    rounding points; q [H,512] float64, sink [H] float64."""
    codes, rope, mult = _decode(rec)
    nope = np.concatenate([codes[:, b] * mult[:, i:i + 1] for i, b in enumerate(BLOCKS)], axis=1)
    x_bf16 = _cast(np.concatenate([nope, rope], axis=1), torch.bfloat16)
    if q_fp8:
        s = q[:, 448:] @ rope.T
        for i, b in enumerate(BLOCKS):
            qb = _e4m3_scaled(q[:, b])
            if q_two_terms:
                qb = qb + _e4m3_scaled(q[:, b] - qb)
            s = s + (qb @ codes[:, b].T) * mult[:, i][None, :]
        s = SCALE * s
    else:
        s = SCALE * (q @ x_bf16.T)
    mx = np.maximum(s.max(axis=1), sink)
    p = np.exp(s - mx[:, None])
    denom = p.sum(axis=1) + np.exp(sink - mx)
    if p_fp8:
        o = np.empty((q.shape[0], 512))
        for i, b in enumerate(BLOCKS):
            o[:, b] = _e4m3_scaled(p * mult[:, i][None, :]) @ codes[:, b]
        o[:, 448:] = _cast(p, torch.bfloat16) @ rope
    else:
        o = _cast(p, torch.bfloat16) @ x_bf16
    return o / denom[:, None]


def _errors(o, ref):
    cos = (o * ref).sum(1) / np.linalg.norm(o, axis=1) / np.linalg.norm(ref, axis=1)
    rel = np.abs(o - ref).max(1) / np.abs(ref).max(1)
    return float(cos.min()), float(rel.max())


VARIANTS = {
    "bf16 latent, bf16 P (built)": {},
    "q e4m3": dict(q_fp8=True),
    "P e4m3": dict(p_fp8=True),
    "q e4m3 hi+lo": dict(q_fp8=True, q_two_terms=True),
}


@pytest.fixture(scope="module")
def study():
    """Worst per-head cosine and max relative error of every variant over two
    seeded queries at 640 candidates (top-512 + SWA 128) and 2176 (top-2048 +
    SWA 128), latents, q and sink drawn as in the benchmark workloads."""
    g = torch.Generator().manual_seed(7)
    worst = {k: [1.0, 0.0] for k in VARIANTS}
    for n in (640, 2176):
        for _ in range(2):
            rec = synth.random_records(n, g, "cpu").numpy()
            q = torch.randn((128, 512), generator=g).to(torch.bfloat16)
            sink = torch.randn(128, generator=g).float().numpy()
            ref, _ = oracle.attention_row(q.view(torch.int16).numpy().view(np.uint16), sink, SCALE, rec)
            for name, kw in VARIANTS.items():
                c, r = _errors(_emulate(q.double().numpy(), sink.astype(np.float64), rec, **kw), ref)
                worst[name][0] = min(worst[name][0], c)
                worst[name][1] = max(worst[name][1], r)
    for name, (c, r) in worst.items():
        print(f"{name:30s} min cos {c:.6f}  max rel {r:.4f}")
    return worst


def test_built_precision_passes_the_gate_with_margin(study):
    c, r = study["bf16 latent, bf16 P (built)"]
    assert c >= GATE_COS and r <= GATE_REL / 3


def test_single_fp8_q_or_p_fails_the_gate(study):
    assert study["q e4m3"][1] > GATE_REL
    assert study["P e4m3"][1] > GATE_REL


def test_two_term_fp8_q_is_as_accurate_as_bf16(study):
    c, r = study["q e4m3 hi+lo"]
    assert c >= GATE_COS and r <= GATE_REL / 3
