"""GPU parity for many query tokens per sequence ("ROADMAP -- Stage E" §E8:
prefill-style steps with T > 1 spread over many CTAs): T beyond 4 runs the
indexer as token groups (4, 3, 2 or 1 tokens sharing one read of the keys),
the top-k over B*T rows and the attention over B*T query rows, each token with
its own visible range and SWA window. Every step against the oracle."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import (check_attention, check_logits, check_topk_exact, logit_magnitude, lse_bounds_for_rows,
                     oracle_cache)

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
SCALE = 1.0 / math.sqrt(512)


def _inputs(B, T, ncap, k, base, n_comp, seed=11, kind="csa"):
    wl = synth.custom(kind, B=B, T=T, ncap=ncap, k=k, ctx=1 << 20)
    x = synth.generate(wl, seed=seed, device="cuda")
    # consecutive tokens from per-sequence bases: visible ranges step every m tokens
    pos = [[b0 + t for t in range(T)] for b0 in base]
    x.q_pos = torch.tensor(pos, dtype=torch.int32, device="cuda")
    x.n_comp = torch.tensor(n_comp, dtype=torch.int32, device="cuda")
    return x


def _check_csa(csd, x, rows_att):
    wl = x.wl
    B, T = wl.B, wl.T
    lg = csd.csa_indexer_logits(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q_pos, x.n_comp, wl.m)
    idx, cnt = csd.csa_topk(lg, x.q_pos, x.n_comp, wl.m, wl.k)
    comp = csd.cache_desc(x.comp, wl.ncap, x.seq_stride)
    out, lse = csd.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, wl.W, idx, cnt, x.q_pos)
    torch.cuda.synchronize()
    assert csd.csa_read_device_error() == 0
    rows = list(range(B * T))
    ora = oracle.indexer_logits(x.q_idx.cpu(), x.q_idx_scale.cpu(), x.w_idx.cpu(), x.k_idx.cpu(), x.k_idx_scale.cpu(),
                                x.q_pos.cpu(), x.n_comp.cpu(), wl.m, threads=THREADS)
    A = logit_magnitude(x, rows)
    g = lg.cpu().numpy().reshape(-1, wl.ncap)
    for r in rows:
        check_logits(g[r], ora.reshape(-1, wl.ncap)[r], A[r], f"T={T} row {r}")
    oi, oc = oracle.topk(lg.cpu().numpy().astype(np.float64), x.q_pos.cpu(), x.n_comp.cpu(), wl.m, wl.k)
    check_topk_exact(idx.cpu().numpy(), cnt.cpu().numpy(), oi, oc, f"T={T}")
    oo, ol = oracle.csa_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x),
                                  x.ring.cpu().numpy(), wl.W, idx.cpu(), cnt.cpu(), x.q_pos.cpu(), threads=THREADS,
                                  rows=rows_att)
    gi, gc = idx.cpu().numpy().reshape(-1, wl.k), cnt.cpu().numpy().reshape(-1)
    tol = lse_bounds_for_rows(x, rows_att, lambda r: gi[r][:gc[r]], SCALE)
    stats = check_attention(out.float().cpu().numpy().reshape(-1, 128, 512)[rows_att],
                            lse.cpu().numpy().reshape(-1, 128)[rows_att], oo.reshape(-1, 128, 512)[rows_att],
                            ol.reshape(-1, 128)[rows_att], f"T={T}", tol)
    # the whole step in one call gives the same results
    sidx, scnt = torch.empty_like(idx), torch.empty_like(cnt)
    out2, lse2 = csd.csa_decode_step(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q, x.sink, SCALE,
                                     comp, x.ring, wl.W, x.q_pos, x.n_comp, wl.m, wl.k, topk_idx=sidx, topk_cnt=scnt)
    assert torch.equal(sidx, idx) and torch.equal(scnt, cnt) and torch.equal(out2, out) and torch.equal(lse2, lse)
    return stats


@pytest.mark.parametrize("T", [5, 6, 8, 12])
def test_token_groups(cuda_lib, T):
    # sequence bases around block boundaries; capacities with ragged tiles; n_vis from 0 to past the capacity
    x = _inputs(3, T, 700, 48, [1, 1021, 2790], [700, 700, 690])
    stats = _check_csa(cuda_lib, x, list(range(3 * T)))
    print(f"T={T}: min cos {stats[0]:.6f} max rel {stats[1]:.3g}")


def test_prefill_128_tokens(cuda_lib):
    x = _inputs(1, 128, 4096, 256, [4 * 3000 + 1], [4096])
    stats = _check_csa(cuda_lib, x, [0, 1, 2, 3, 4, 63, 126, 127])
    print(f"T=128: min cos {stats[0]:.6f} max rel {stats[1]:.3g}")


def test_hca_128_tokens(cuda_lib):
    csd = cuda_lib
    x = _inputs(2, 128, 600, 0, [128 * 300 - 64, 128 * 599 + 1], [600, 600], kind="hca")
    comp = csd.cache_desc(x.comp, x.wl.ncap, x.seq_stride)
    out, lse = csd.hca_sink_attention_decode(x.q, x.sink, SCALE, comp, x.n_comp, x.ring, x.wl.W, x.q_pos, x.wl.m)
    torch.cuda.synchronize()
    assert csd.csa_read_device_error() == 0
    rows = [0, 63, 64, 127, 128, 255]
    oo, ol = oracle.hca_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x), x.n_comp.cpu(),
                                  x.ring.cpu().numpy(), x.wl.W, x.q_pos.cpu(), x.wl.m, threads=THREADS, rows=rows)
    qp, nc = x.q_pos.cpu().numpy().reshape(-1), x.n_comp.cpu().numpy()
    tol = lse_bounds_for_rows(x, rows, lambda r: np.arange(min(qp[r] // x.wl.m, nc[r // x.wl.T], x.wl.ncap)), SCALE)
    check_attention(out.float().cpu().numpy().reshape(-1, 128, 512)[rows], lse.cpu().numpy().reshape(-1, 128)[rows],
                    oo.reshape(-1, 128, 512)[rows], ol.reshape(-1, 128)[rows], "hca T=128", tol)
