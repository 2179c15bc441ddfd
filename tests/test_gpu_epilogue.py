"""GPU parity of the attention's output epilogue ("DSV4 Audit" §A4 inverse
RoPE at the query position; "ROADMAP -- Stage E" §E6 E2M1 output with a
per-128-element amax), through the C ABI's _ex entry points.

Both the split path (the combine kernel forms the output: the 1K and 32K
workloads) and the single-split path (the attention kernel forms it: HCA with
64 queries) are covered; the HCA queries sit near position 2^20, where the
rotation angles reach 10^6 rad.

* Inverse RoPE, BF16 output: the same attention gates as the plain call
  against the oracle's output turned back by the oracle's inverse RoPE; the
  nope dims and the LSE are bit-identical to the plain call; the rope dims
  equal the plain call's output turned back in fp64 to within the two BF16
  roundings.
* E2M1 output: the multipliers and codes equal the oracle's quantisation of
  the same call's BF16 output (same epilogue), except where a value lies
  within BF16 rounding of an E2M1 rounding boundary; dequantised, the output
  agrees with the oracle's fp64 output quantised by the oracle as closely as
  the 4-bit format allows.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import check_attention, lse_bounds_for_rows, oracle_cache

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1
SCALE = 1.0 / math.sqrt(512)
THETA = 10000.0
CASES = {"csa_b1_ctx1k_k64": [0], "csa_b8_ctx16k32k_k512": [0, 5], "hca_b64_ctx1m": [0, 37, 63],
         "csa_b2t4_ctx20k_k128": [0, 3, 5, 7]}
# a small multi-token workload: 4 tokens a sequence, each with its own position (and rotation)
CUSTOM = {"csa_b2t4_ctx20k_k128": synth.custom("csa", B=2, T=4, ncap=5000, k=128, ctx=20000,
                                              name="csa_b2t4_ctx20k_k128")}
# E2M1 rounding boundaries (midpoints between neighbouring magnitudes)
BOUNDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
E2M1 = np.array([oracle.e2m1_value(c) for c in range(16)])

_cache = {}


def _setup(csd, name):
    if name not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        x = synth.generate(CUSTOM.get(name, name), seed=3, device="cuda")
        comp = csd.cache_desc(x.comp, x.wl.ncap, x.seq_stride)
        if x.wl.kind == "csa":
            lg = csd.csa_indexer_logits(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q_pos, x.n_comp,
                                        x.wl.m)
            idx, cnt = csd.csa_topk(lg, x.q_pos, x.n_comp, x.wl.m, x.wl.k)
        else:
            idx = cnt = None
        _cache[name] = (x, comp, idx, cnt)
    return _cache[name]


def _attend(csd, name, **epi):
    x, comp, idx, cnt = _setup(csd, name)
    if x.wl.kind == "csa":
        return csd.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, x.wl.W, idx, cnt, x.q_pos, **epi)
    return csd.hca_sink_attention_decode(x.q, x.sink, SCALE, comp, x.n_comp, x.ring, x.wl.W, x.q_pos, x.wl.m, **epi)


def _oracle(name, rows):
    x, _, idx, cnt = _cache[name]
    if x.wl.kind == "csa":
        oo, ol = oracle.csa_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x),
                                      x.ring.cpu().numpy(), x.wl.W, idx.cpu(), cnt.cpu(), x.q_pos.cpu(),
                                      threads=THREADS, rows=rows)
        gi, gc = idx.cpu().numpy().reshape(-1, x.wl.k), cnt.cpu().numpy().reshape(-1)
        sel = lambda r: gi[r][:gc[r]]
    else:
        oo, ol = oracle.hca_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x),
                                      x.n_comp.cpu(), x.ring.cpu().numpy(), x.wl.W, x.q_pos.cpu(), x.wl.m,
                                      threads=THREADS, rows=rows)
        qp, nc = x.q_pos.cpu().numpy().reshape(-1), x.n_comp.cpu().numpy()
        sel = lambda r: np.arange(min(qp[r] // x.wl.m, nc[r // x.wl.T], x.wl.ncap))
    oo = oo.reshape(-1, 128, 512)[rows]
    ol = ol.reshape(-1, 128)[rows]
    pos = x.q_pos.cpu().numpy().reshape(-1)[rows]
    return oo, ol, pos, lse_bounds_for_rows(x, rows, sel, SCALE)


def _unpack(packed):
    p = packed.cpu().numpy()
    codes = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    codes[..., 0::2] = p & 15
    codes[..., 1::2] = p >> 4
    return codes


@pytest.mark.parametrize("name,theta", [(n, THETA) for n in CASES] + [("csa_b8_ctx16k32k_k512", 1.0e6)])
def test_inverse_rope_bf16(cuda_lib, name, theta):
    csd = cuda_lib
    rows = CASES[name]
    plain, lse0 = _attend(csd, name)
    out, lse = _attend(csd, name, inverse_rope=True, rope_theta=theta)
    torch.cuda.synchronize()
    assert csd.csa_read_device_error() == 0
    assert torch.equal(out[..., :448], plain[..., :448]) and torch.equal(lse, lse0)
    B, T = out.shape[:2]
    # the rotation itself: the plain output turned back in fp64
    pos_all = _cache[name][0].q_pos.cpu().numpy().reshape(-1)
    want = oracle.inverse_rope(plain.float().cpu().numpy().reshape(B * T, 128, 512), pos_all, theta)
    got = out.float().cpu().numpy().reshape(B * T, 128, 512)
    mag = np.abs(plain.float().cpu().numpy().reshape(B * T, 128, 512)[..., 448:])
    pair_mag = np.repeat(np.hypot(mag[..., 0::2], mag[..., 1::2]), 2, axis=-1)
    assert np.all(np.abs(got[..., 448:] - want[..., 448:]) <= 2 ** -7 * pair_mag + 1e-30)
    # against the oracle's output turned back by the oracle
    oo, ol, pos, tol = _oracle(name, rows)
    ref = oracle.inverse_rope(oo, pos, theta)
    stats = check_attention(got[rows], lse.cpu().numpy().reshape(-1, 128)[rows], ref, ol, f"{name} inverse rope", tol)
    print(f"{name} inverse rope (theta {theta:g}): min cos {stats[0]:.6f}  max rel {stats[1]:.3g}")


def _near_bound(v, rel):
    a = np.abs(v)
    return np.any(np.abs(a[..., None] - BOUNDS) <= rel * np.maximum(a[..., None], BOUNDS), axis=-1)


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_fp4_output(cuda_lib, name, rope):
    csd = cuda_lib
    rows = CASES[name]
    epi = dict(inverse_rope=rope, rope_theta=THETA)
    bf16, lse0 = _attend(csd, name, **epi)
    (packed, scales), lse = _attend(csd, name, fp4_out=True, **epi)
    torch.cuda.synchronize()
    assert csd.csa_read_device_error() == 0
    assert torch.equal(lse, lse0)
    B, T = bf16.shape[:2]
    codes = _unpack(packed).reshape(B * T, 128, 512)
    s_gpu = scales.cpu().numpy().astype(np.float64).reshape(B * T, 128, 4)
    # the quantiser: the oracle's E2M1 quantisation of this call's BF16 output
    v = bf16.float().cpu().numpy().astype(np.float64).reshape(B * T, 128, 512)
    oc, os_ = oracle.e2m1_quantize(v, 128)
    np.testing.assert_allclose(s_gpu, os_, rtol=2 ** -8, atol=0)
    ratio = v / np.repeat(os_, 128, axis=-1)
    differ = codes != oc
    # a code may differ only next to a rounding boundary (BF16 rounding of the value and of the amax), by one step
    assert not np.any(differ & ~_near_bound(ratio, 2 ** -7)), f"{int((differ & ~_near_bound(ratio, 2 ** -7)).sum())}"
    mi, mo = codes[differ] & 7, oc[differ] & 7
    adjacent = ((np.abs(mi.astype(int) - mo) == 1) & ((codes[differ] & 8) == (oc[differ] & 8))) | ((mi == 0) & (mo == 0))
    assert np.all(adjacent)
    # dequantised, against the oracle's exact (fp64) output: as close as the
    # oracle's own E2M1 quantisation of that output, per head, up to what the
    # attention's own error (cos >= 0.999 gate) can move a 4-bit code
    oo, _, pos, _ = _oracle(name, rows)
    ref = oracle.inverse_rope(oo, pos, THETA) if rope else oo
    rc, rs = oracle.e2m1_quantize(ref, 128)
    deq_ref = E2M1[rc] * np.repeat(rs, 128, axis=-1)
    deq = E2M1[codes[rows]] * np.repeat(s_gpu[rows], 128, axis=-1)
    cos = lambda a, b: (a * b).sum(-1) / np.linalg.norm(a, axis=-1) / np.linalg.norm(b, axis=-1)
    cos_gpu, cos_fmt = cos(deq, ref), cos(deq_ref, ref)
    print(f"{name} fp4 rope={rope}: {int(differ.sum())} codes at boundaries of {differ.size}; "
          f"min cos to the exact output {cos_gpu.min():.5f} (oracle-quantised {cos_fmt.min():.5f}); "
          f"largest per-head shortfall {float((cos_fmt - cos_gpu).max()):.2e}")
    assert np.all(cos_gpu >= cos_fmt - 1e-3)


@pytest.mark.parametrize("name", ["csa_b8_ctx16k32k_k512", "csa_b2t4_ctx20k_k128"])
def test_decode_step_with_epilogue_equals_separate_calls(cuda_lib, name):
    csd = cuda_lib
    x, comp, idx, cnt = _setup(csd, name)
    wl = x.wl
    epi = dict(inverse_rope=True, rope_theta=THETA, fp4_out=True)
    (p1, s1), l1 = _attend(csd, name, **epi)
    sidx, scnt = torch.empty_like(idx), torch.empty_like(cnt)
    (p2, s2), l2 = csd.csa_decode_step(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q, x.sink, SCALE,
                                       comp, x.ring, wl.W, x.q_pos, x.n_comp, wl.m, wl.k, topk_idx=sidx,
                                       topk_cnt=scnt, **epi)
    torch.cuda.synchronize()
    assert csd.csa_read_device_error() == 0
    assert torch.equal(sidx, idx) and torch.equal(scnt, cnt)
    assert torch.equal(p1, p2) and torch.equal(s1, s2) and torch.equal(l1, l2)
