"""The allocation-free attention entry point (csa_sink_attention_decode_noalloc).

It serves callers that cannot allocate device memory on the decode path (a
runtime whose memory is reserved by its own pool, a plugin whose framework owns
allocation, latency-critical code that cannot take cudaMalloc's implicit
synchronisation): the split partials live in the library's static device
scratch instead of a caller workspace. Two calls in a row, on workloads with
different split counts (so the second call starts from the first call's
leftovers), must match the workspace entry point within the attention
tolerances the other tests use. This file is collected last on purpose.
"""
import math

import numpy as np
import pytest
import torch

import synth
from _parity import ATT_COS_MIN, ATT_MAXREL, LSE_ATOL

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(512)


def _selection(csd, x):
    lg = csd.csa_indexer_logits(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q_pos, x.n_comp, x.wl.m)
    return csd.csa_topk(lg, x.q_pos, x.n_comp, x.wl.m, x.wl.k)


def _close(a_out, a_lse, b_out, b_lse, what):
    g = a_out.float().cpu().numpy().astype(np.float64).reshape(-1, 512)
    o = b_out.float().cpu().numpy().astype(np.float64).reshape(-1, 512)
    cos = np.sum(g * o, -1) / np.maximum(np.linalg.norm(g, axis=-1) * np.linalg.norm(o, axis=-1), 1e-300)
    rel = np.max(np.abs(g - o), -1) / np.maximum(np.max(np.abs(o), -1), 1e-300)
    assert cos.min() >= ATT_COS_MIN, f"{what}: cosine {cos.min()}"
    assert rel.max() <= ATT_MAXREL, f"{what}: max rel {rel.max()}"
    assert torch.max(torch.abs(a_lse - b_lse)).item() <= LSE_ATOL, what


def test_noalloc_matches_workspace_entry_point_twice(cuda_lib):
    csd = cuda_lib
    cases = []
    for name in ("csa_b8_ctx16k32k_k512", "csa_b1_ctx1k_k64"):
        x = synth.generate(name, seed=0, device="cuda")
        idx, cnt = _selection(csd, x)
        comp = csd.cache_desc(x.comp, x.wl.ncap, x.seq_stride)
        assert csd.csa_workspace_bytes(csd.OP_ATTENTION, x.wl.B, x.wl.T, x.wl.ncap, x.wl.k) > 0  # splits in use
        ref = csd.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, x.wl.W, idx, cnt, x.q_pos)
        cases.append((name, x, idx, cnt, comp, ref))
    # two calls in a row; the second starts from the first call's scratch contents
    got = [csd.csa_sink_attention_decode_noalloc(x.q, x.sink, SCALE, comp, x.ring, x.wl.W, idx, cnt, x.q_pos)
           for _, x, idx, cnt, comp, _ in cases]
    torch.cuda.synchronize()
    assert csd.csa_read_device_error() == 0
    for (name, _, _, _, _, (ref_out, ref_lse)), (out, lse) in zip(cases, got):
        _close(out, lse, ref_out, ref_lse, name)
