"""GPU parity: every step of the CUDA path, called through the C ABI, against
the CPU oracle on the same seeded inputs. Full-size workloads are checked on
sampled query rows (all rows where the oracle is quick); the small and
edge-case workloads element by element."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import (check_attention, check_logits, check_topk_band, check_topk_exact, logit_magnitude,
                     lse_bounds_for_rows, oracle_cache)

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1
SCALE = 1.0 / math.sqrt(512)

# flat query rows the oracle recomputes at full size (None: every row)
ROWS = {
    "csa_b1_ctx1k_k64": None,
    "csa_b8_ctx16k32k_k512": None,
    "csa_b32_ctx128k_k2048": [0, 13, 31],
    "csa_b4t4_ctx1m_k2048": [0, 7, 12, 15],
    "hca_b64_ctx1m": [0, 37, 63],
}
CSA = [n for n in ROWS if n.startswith("csa")]

_inputs = {}


def inputs(name, paged=False):
    key = (name, paged)
    if key not in _inputs:
        _inputs.clear()
        torch.cuda.empty_cache()
        _inputs[key] = synth.generate(name, seed=0, device="cuda", paged=paged)
    return _inputs[key]


def rows_of(name, x):
    r = ROWS.get(name)
    return list(range(x.wl.B * x.wl.T)) if r is None else r


def gpu_cache(csd, x):
    return csd.cache_desc(x.comp, x.wl.ncap, x.seq_stride, x.block_table, x.page_records if x.block_table is not None else 0)


def run_indexer(csd, x):
    return csd.csa_indexer_logits(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q_pos, x.n_comp, x.wl.m)


def flat(a, rows):
    a = a.reshape(-1, *a.shape[2:])
    return a[rows]


@pytest.mark.parametrize("name", CSA)
def test_indexer_logits(cuda_lib, name):
    x = inputs(name)
    lg = run_indexer(cuda_lib, x)
    assert cuda_lib.csa_read_device_error() == 0
    rows = rows_of(name, x)
    ora = oracle.indexer_logits(x.q_idx.cpu(), x.q_idx_scale.cpu(), x.w_idx.cpu(), x.k_idx.cpu(), x.k_idx_scale.cpu(),
                                x.q_pos.cpu(), x.n_comp.cpu(), x.wl.m, threads=THREADS, rows=rows)
    A = logit_magnitude(x, rows)
    g = lg.cpu().numpy().reshape(-1, x.wl.ncap)
    o = ora.reshape(-1, x.wl.ncap)
    for r in rows:
        check_logits(g[r], o[r], A[r], f"{name} row {r}")


@pytest.mark.parametrize("name", CSA)
def test_topk_exact_on_identical_logits(cuda_lib, name):
    x = inputs(name)
    lg = run_indexer(cuda_lib, x)
    idx, cnt = cuda_lib.csa_topk(lg, x.q_pos, x.n_comp, x.wl.m, x.wl.k)
    oi, oc = oracle.topk(lg.cpu().numpy().astype(np.float64), x.q_pos.cpu(), x.n_comp.cpu(), x.wl.m, x.wl.k,
                         threads=THREADS)
    check_topk_exact(idx.cpu().numpy(), cnt.cpu().numpy(), oi, oc, name)


@pytest.mark.parametrize("name", CSA)
def test_topk_end_to_end_band(cuda_lib, name):
    x = inputs(name)
    lg = run_indexer(cuda_lib, x)
    idx, cnt = cuda_lib.csa_topk(lg, x.q_pos, x.n_comp, x.wl.m, x.wl.k)
    rows = rows_of(name, x)
    ora = oracle.indexer_logits(x.q_idx.cpu(), x.q_idx_scale.cpu(), x.w_idx.cpu(), x.k_idx.cpu(), x.k_idx_scale.cpu(),
                                x.q_pos.cpu(), x.n_comp.cpu(), x.wl.m, threads=THREADS, rows=rows)
    ora = ora.reshape(-1, 1, x.wl.ncap)[rows]
    oi, oc = oracle.topk(ora, np.zeros((len(rows), 1), np.int32) + x.q_pos.cpu().numpy().reshape(-1)[rows][:, None],
                         x.n_comp.cpu().numpy()[[r // x.wl.T for r in rows]], x.wl.m, x.wl.k)
    gi = idx.cpu().numpy().reshape(-1, 1, x.wl.k)[rows]
    gc = cnt.cpu().numpy().reshape(-1, 1)[rows]
    swaps = check_topk_band(gi, gc, ora, oi, oc, x.wl.k, name)
    print(f"{name}: {swaps} index swaps inside the tolerance band over {len(rows)} rows")


@pytest.mark.parametrize("name", CSA)
def test_gather_bytes(cuda_lib, name):
    x = inputs(name)
    lg = run_indexer(cuda_lib, x)
    idx, cnt = cuda_lib.csa_topk(lg, x.q_pos, x.n_comp, x.wl.m, x.wl.k)
    kv, kvc = cuda_lib.csa_gather_swa(gpu_cache(cuda_lib, x), x.ring, x.wl.W, idx, cnt, x.q_pos)
    assert cuda_lib.csa_read_device_error() == 0
    okv, okc = oracle.gather(oracle_cache(x), x.ring.cpu().numpy(), x.wl.W, idx.cpu(), cnt.cpu(), x.q_pos.cpu(),
                             threads=THREADS)
    gkc = kvc.cpu().numpy()
    assert np.array_equal(gkc, okc)
    gkv = kv.cpu().numpy()
    for r in np.ndindex(*gkc.shape):
        n = int(okc[r])
        assert np.array_equal(gkv[r][:n], okv[r][:n]), f"row {r}"


def _oracle_csa_rows(x, idx, cnt, rows):
    B, T = x.wl.B, x.wl.T
    return oracle.csa_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x), x.ring.cpu().numpy(),
                                x.wl.W, idx.cpu(), cnt.cpu(), x.q_pos.cpu(), threads=THREADS, rows=rows)


@pytest.mark.parametrize("name", CSA)
def test_csa_attention(cuda_lib, name):
    x = inputs(name)
    lg = run_indexer(cuda_lib, x)
    idx, cnt = cuda_lib.csa_topk(lg, x.q_pos, x.n_comp, x.wl.m, x.wl.k)
    out, lse = cuda_lib.csa_sink_attention_decode(x.q, x.sink, SCALE, gpu_cache(cuda_lib, x), x.ring, x.wl.W, idx, cnt,
                                                  x.q_pos)
    assert cuda_lib.csa_read_device_error() == 0
    rows = rows_of(name, x)
    oo, ol = _oracle_csa_rows(x, idx, cnt, rows)
    gi, gc = idx.cpu().numpy().reshape(-1, x.wl.k), cnt.cpu().numpy().reshape(-1)
    tol = lse_bounds_for_rows(x, rows, lambda r: gi[r][:gc[r]], SCALE)
    stats = check_attention(flat(out.float().cpu().numpy(), rows), flat(lse.cpu().numpy(), rows), flat(oo, rows),
                            flat(ol, rows), name, tol)
    print(f"{name}: min cos {stats[0]:.6f}  max rel {stats[1]:.3g}  lse err/bound {stats[2]:.3g}")


@pytest.mark.parametrize("name", CSA)
def test_decode_step_equals_separate_calls(cuda_lib, name):
    x = inputs(name)
    comp = gpu_cache(cuda_lib, x)
    lg = run_indexer(cuda_lib, x)
    idx, cnt = cuda_lib.csa_topk(lg, x.q_pos, x.n_comp, x.wl.m, x.wl.k)
    out, lse = cuda_lib.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, x.wl.W, idx, cnt, x.q_pos)
    sidx = torch.empty_like(idx)
    scnt = torch.empty_like(cnt)
    out2, lse2 = cuda_lib.csa_decode_step(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q, x.sink, SCALE,
                                          comp, x.ring, x.wl.W, x.q_pos, x.n_comp, x.wl.m, x.wl.k, topk_idx=sidx,
                                          topk_cnt=scnt)
    assert torch.equal(sidx, idx) and torch.equal(scnt, cnt)
    assert torch.equal(out2, out) and torch.equal(lse2, lse)


def test_hca_attention(cuda_lib):
    name = "hca_b64_ctx1m"
    x = inputs(name)
    out, lse = cuda_lib.hca_sink_attention_decode(x.q, x.sink, SCALE, gpu_cache(cuda_lib, x), x.n_comp, x.ring, x.wl.W,
                                                  x.q_pos, x.wl.m)
    assert cuda_lib.csa_read_device_error() == 0
    rows = rows_of(name, x)
    oo, ol = oracle.hca_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x), x.n_comp.cpu(),
                                  x.ring.cpu().numpy(), x.wl.W, x.q_pos.cpu(), x.wl.m, threads=THREADS, rows=rows)
    qp, nc = x.q_pos.cpu().numpy().reshape(-1), x.n_comp.cpu().numpy()
    tol = lse_bounds_for_rows(x, rows, lambda r: np.arange(min(qp[r] // x.wl.m, nc[r // x.wl.T], x.wl.ncap)), SCALE)
    stats = check_attention(flat(out.float().cpu().numpy(), rows), flat(lse.cpu().numpy(), rows), flat(oo, rows),
                            flat(ol, rows), name, tol)
    print(f"{name}: min cos {stats[0]:.6f}  max rel {stats[1]:.3g}  lse err/bound {stats[2]:.3g}")
