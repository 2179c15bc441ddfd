"""The allocation-free attention entry point (csa_sink_attention_decode_noalloc).

It serves callers that cannot allocate device memory on the decode path (a
runtime whose memory is reserved by its own pool, a plugin whose framework owns
allocation, latency-critical code that cannot take cudaMalloc's implicit
synchronisation): the split partials live in the library's static device
scratch instead of a caller workspace. The kernels and the split count are
those of the workspace entry point, so the results must be bit-identical to
it, whatever the scratch held before: calls alternate between two workloads
with different split counts (each call starts from the other's leftovers), in
both orders relative to the workspace calls. One output is also checked
against the oracle. This file is collected last on purpose.
"""
import math
import os

import pytest
import torch

import oracle
import synth
from _parity import check_attention, lse_bounds_for_rows, oracle_cache

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(512)
THREADS = os.cpu_count() or 1


def _selection(csd, x):
    lg = csd.csa_indexer_logits(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q_pos, x.n_comp, x.wl.m)
    return csd.csa_topk(lg, x.q_pos, x.n_comp, x.wl.m, x.wl.k)


def test_noalloc_matches_workspace_entry_point_twice(cuda_lib):
    csd = cuda_lib
    cases = []
    for name in ("csa_b8_ctx16k32k_k512", "csa_b1_ctx1k_k64"):
        x = synth.generate(name, seed=0, device="cuda")
        idx, cnt = _selection(csd, x)
        comp = csd.cache_desc(x.comp, x.wl.ncap, x.seq_stride)
        assert csd.csa_workspace_bytes(csd.OP_ATTENTION, x.wl.B, x.wl.T, x.wl.ncap, x.wl.k) > 0  # splits in use
        cases.append((name, x, idx, cnt, comp))

    def noalloc(c):
        _, x, idx, cnt, comp = c
        return csd.csa_sink_attention_decode_noalloc(x.q, x.sink, SCALE, comp, x.ring, x.wl.W, idx, cnt, x.q_pos)

    def with_ws(c):
        _, x, idx, cnt, comp = c
        return csd.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, x.wl.W, idx, cnt, x.q_pos)

    # noalloc first (two calls in a row), then the workspace calls
    first = [noalloc(c) for c in cases]
    ref = [with_ws(c) for c in cases]
    # workspace calls first, then noalloc again in the opposite workload order
    ref2 = [with_ws(c) for c in reversed(cases)][::-1]
    second = [noalloc(c) for c in reversed(cases)][::-1]
    torch.cuda.synchronize()
    assert csd.csa_read_device_error() == 0
    for (name, *_), (o1, l1), (o0, l0), (o2, l2), (o3, l3) in zip(cases, first, ref, ref2, second):
        assert torch.equal(o0, o2) and torch.equal(l0, l2), f"{name}: workspace calls differ"
        assert torch.equal(o1, o0) and torch.equal(l1, l0), f"{name}: noalloc (before) differs from the workspace call"
        assert torch.equal(o3, o0) and torch.equal(l3, l0), f"{name}: noalloc (after) differs from the workspace call"

    # the allocation-free output against the oracle on a few rows
    name, x, idx, cnt, comp = cases[0]
    out, lse = second[0]
    rows = [0, 3, 7]
    k = x.wl.k
    oo, ol = oracle.csa_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x),
                                  x.ring.cpu().numpy(), x.wl.W, idx.cpu(), cnt.cpu(), x.q_pos.cpu(), threads=THREADS,
                                  rows=rows)
    gi, gc = idx.cpu().numpy().reshape(-1, k), cnt.cpu().numpy().reshape(-1)
    tol = lse_bounds_for_rows(x, rows, lambda r: gi[r][:gc[r]], SCALE)
    check_attention(out.float().cpu().numpy().reshape(-1, 128, 512)[rows], lse.cpu().numpy().reshape(-1, 128)[rows],
                    oo.reshape(-1, 128, 512)[rows], ol.reshape(-1, 128)[rows], f"noalloc {name}", tol)
