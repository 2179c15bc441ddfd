"""GPU edge cases against the oracle: ragged capacities spanning several tiles
with a ragged tail, T up to 4 with per-token visible ranges, empty visible
ranges, windows shorter than W, k above the visible count, paged caches with
a shuffled block table, heavy ties in top-k, a -inf sink, indices outside
the cache (reported through the caller's status word, never dereferenced),
and bounded waits made to expire (reported, and the device stays usable)."""
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


def _custom(B, T, ncap, k, q_pos, n_comp, paged=False, seed=3):
    wl = synth.custom("csa", B=B, T=T, ncap=ncap, k=k, ctx=1 << 20)
    x = synth.generate(wl, seed=seed, device="cuda", paged=paged)
    x.q_pos = torch.tensor(q_pos, dtype=torch.int32, device="cuda")
    x.n_comp = torch.tensor(n_comp, dtype=torch.int32, device="cuda")
    return x


def _cache(csd, x):
    return csd.cache_desc(x.comp, x.wl.ncap, x.seq_stride, x.block_table,
                          x.page_records if x.block_table is not None else 0)


# q_pos chosen so that n_vis = floor(p/4) covers 0, < k, = k, > k and the
# capacity, and windows shorter than W = 128
EDGE_POS = [[0, 1, 2, 3], [5, 6, 7, 8], [130, 131, 132, 133], [1199, 1200, 1201, 1202], [257, 258, 259, 260]]
EDGE_NCOMP = [300, 300, 300, 300, 64]


def _pipeline(csd, x):
    lg = csd.csa_indexer_logits(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q_pos, x.n_comp, x.wl.m)
    idx, cnt = csd.csa_topk(lg, x.q_pos, x.n_comp, x.wl.m, x.wl.k)
    return lg, idx, cnt


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_ragged_capacity_and_visibility(cuda_lib, T):
    pos = [row[:T] for row in EDGE_POS]
    x = _custom(5, T, 300, 40, pos, EDGE_NCOMP)
    lg, idx, cnt = _pipeline(cuda_lib, x)
    assert cuda_lib.csa_read_device_error() == 0
    rows = list(range(5 * T))
    ora = oracle.indexer_logits(x.q_idx.cpu(), x.q_idx_scale.cpu(), x.w_idx.cpu(), x.k_idx.cpu(),
                                x.k_idx_scale.cpu(), x.q_pos.cpu(), x.n_comp.cpu(), 4, threads=THREADS)
    A = logit_magnitude(x, rows)
    g = lg.cpu().numpy().reshape(-1, 300)
    for r in rows:
        check_logits(g[r], ora.reshape(-1, 300)[r], A[r], f"T={T} row {r}")
    oi, oc = oracle.topk(lg.cpu().numpy().astype(np.float64), x.q_pos.cpu(), x.n_comp.cpu(), 4, 40)
    check_topk_exact(idx.cpu().numpy(), cnt.cpu().numpy(), oi, oc, f"T={T}")
    out, lse = cuda_lib.csa_sink_attention_decode(x.q, x.sink, SCALE, _cache(cuda_lib, x), x.ring, 128, idx, cnt,
                                                  x.q_pos)
    assert cuda_lib.csa_read_device_error() == 0
    oo, ol = oracle.csa_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x),
                                  x.ring.cpu().numpy(), 128, idx.cpu(), cnt.cpu(), x.q_pos.cpu(), threads=THREADS)
    gi, gc = idx.cpu().numpy().reshape(-1, 40), cnt.cpu().numpy().reshape(-1)
    tol = lse_bounds_for_rows(x, rows, lambda r: gi[r][:gc[r]], SCALE)
    check_attention(out.float().cpu().numpy().reshape(-1, 128, 512), lse.cpu().numpy().reshape(-1, 128),
                    oo.reshape(-1, 128, 512), ol.reshape(-1, 128), f"T={T}", tol)
    kv, kvc = cuda_lib.csa_gather_swa(_cache(cuda_lib, x), x.ring, 128, idx, cnt, x.q_pos)
    okv, okc = oracle.gather(oracle_cache(x), x.ring.cpu().numpy(), 128, idx.cpu(), cnt.cpu(), x.q_pos.cpu())
    assert np.array_equal(kvc.cpu().numpy(), okc)
    gkv = kv.cpu().numpy()
    for r in np.ndindex(*okc.shape):
        assert np.array_equal(gkv[r][:okc[r]], okv[r][:okc[r]])


def test_indexer_capacity_not_a_multiple_of_the_tile(cuda_lib):
    for ncap in (1, 127, 129, 1000):
        x = _custom(2, 1, ncap, 1, [[4 * ncap + 8], [4 * ncap - 4]], [ncap, ncap])
        lg = cuda_lib.csa_indexer_logits(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q_pos, x.n_comp, 4)
        ora = oracle.indexer_logits(x.q_idx.cpu(), x.q_idx_scale.cpu(), x.w_idx.cpu(), x.k_idx.cpu(),
                                    x.k_idx_scale.cpu(), x.q_pos.cpu(), x.n_comp.cpu(), 4)
        A = logit_magnitude(x, [0, 1])
        for r in (0, 1):
            check_logits(lg.cpu().numpy().reshape(-1, ncap)[r], ora.reshape(-1, ncap)[r], A[r], f"ncap={ncap}")


def test_paged_cache_matches_contiguous_and_oracle(cuda_lib):
    pos = [[1023, 1024], [4000, 4001]]
    xc = _custom(2, 2, 1000, 64, pos, [1000, 1000], paged=False, seed=7)
    xp = _custom(2, 2, 1000, 64, pos, [1000, 1000], paged=True, seed=7)
    assert xp.block_table is not None
    _, idx, cnt = _pipeline(cuda_lib, xc)
    oc_, lc_ = cuda_lib.csa_sink_attention_decode(xc.q, xc.sink, SCALE, _cache(cuda_lib, xc), xc.ring, 128, idx, cnt,
                                                  xc.q_pos)
    op_, lp_ = cuda_lib.csa_sink_attention_decode(xp.q, xp.sink, SCALE, _cache(cuda_lib, xp), xp.ring, 128, idx, cnt,
                                                  xp.q_pos)
    assert cuda_lib.csa_read_device_error() == 0
    assert torch.equal(oc_, op_) and torch.equal(lc_, lp_)
    oo, ol = oracle.csa_attention(xp.q.view(torch.int16).cpu(), xp.sink.cpu(), SCALE, oracle_cache(xp),
                                  xp.ring.cpu().numpy(), 128, idx.cpu(), cnt.cpu(), xp.q_pos.cpu(), threads=THREADS)
    gi, gc = idx.cpu().numpy().reshape(-1, 64), cnt.cpu().numpy().reshape(-1)
    tol = lse_bounds_for_rows(xp, range(4), lambda r: gi[r][:gc[r]], SCALE)
    check_attention(op_.float().cpu().numpy().reshape(-1, 128, 512), lp_.cpu().numpy().reshape(-1, 128),
                    oo.reshape(-1, 128, 512), ol.reshape(-1, 128), "paged", tol)
    kv, kvc = cuda_lib.csa_gather_swa(_cache(cuda_lib, xp), xp.ring, 128, idx, cnt, xp.q_pos)
    okv, okc = oracle.gather(oracle_cache(xp), xp.ring.cpu().numpy(), 128, idx.cpu(), cnt.cpu(), xp.q_pos.cpu())
    assert np.array_equal(kvc.cpu().numpy(), okc)
    for r in np.ndindex(*okc.shape):
        assert np.array_equal(kv.cpu().numpy()[r][:okc[r]], okv[r][:okc[r]])


# One CTA a row: 5000, 8192 (8 keys a thread), 12289 (16, ragged rows:
# scalar loads), 16384 (16), 20001 (32, ragged) and 32768 (32). Two stages
# (32768-entry slices, then the candidates): 70001 and 131076 (merge of up to
# 16384 candidates, indices staged in shared memory; with k = 7 the merge
# rows are not a multiple of 4: scalar loads), 294913 (ten slices: 20480
# candidates at k = 2048, the 32-key merge reading indices from memory).
@pytest.mark.parametrize("ncap", [5000, 8192, 12289, 16384, 20001, 32768, 70001, 131076, 294913])
def test_topk_heavy_ties_and_extremes(cuda_lib, ncap):
    rng = np.random.default_rng(0)
    B, T = 3, 2
    vals = rng.integers(-5, 6, size=(B, T, ncap)).astype(np.float32)
    vals[0, 0, 100:200] = 1e30
    vals[1, 1, :] = 0.0                       # all equal: lowest indices win
    vals[2, 0, ::7] = -np.float32(np.inf)
    vals[0, 1, :] -= 4.0                      # few positive logits: K* negative for large k
    vals[1, 0, :] = -np.abs(vals[1, 0, :]) - 1.0  # no positive logit
    lg = torch.tensor(vals, device="cuda")
    q_pos = torch.tensor([[4 * ncap, 4 * ncap + 1], [4 * ncap - 4, 4 * ncap - 1], [400, 401]], dtype=torch.int32,
                         device="cuda")
    n_comp = torch.tensor([ncap, ncap, ncap], dtype=torch.int32, device="cuda")
    for k in (1, 7, 64, 1000, 2048):
        idx, cnt = cuda_lib.csa_topk(lg, q_pos, n_comp, 4, k)
        oi, oc = oracle.topk(vals.astype(np.float64), q_pos.cpu(), n_comp.cpu(), 4, k)
        check_topk_exact(idx.cpu().numpy(), cnt.cpu().numpy(), oi, oc, f"ties k={k}")


def test_single_candidate_with_minus_inf_sink(cuda_lib):
    # HCA, query at position 0: no visible entry, a window of one token, and a
    # sink of -inf -> every head returns that token's latent (BF16-rounded)
    wl = synth.custom("hca", B=2, T=1, ncap=16, k=0, ctx=0)
    x = synth.generate(wl, seed=5, device="cuda")
    x.q_pos = torch.zeros((2, 1), dtype=torch.int32, device="cuda")
    sink = torch.full((128,), -float("inf"), device="cuda")
    out, lse = cuda_lib.hca_sink_attention_decode(x.q, sink, SCALE, _cache(cuda_lib, x), x.n_comp, x.ring, 128,
                                                  x.q_pos, 128)
    oo, ol = oracle.hca_attention(x.q.view(torch.int16).cpu(), sink.cpu(), SCALE, oracle_cache(x), x.n_comp.cpu(),
                                  x.ring.cpu().numpy(), 128, x.q_pos.cpu(), 128)
    xv = oo[:, 0, 0, :]                                 # the dequantised slot-0 latent of each sequence
    for h in range(128):
        assert np.array_equal(oo[:, 0, h], xv)
    got = out.float().cpu().numpy()[:, 0]
    assert np.all(np.abs(got - xv[:, None, :]) <= 2.0 ** -8 * np.abs(xv[:, None, :]) + 1e-30)
    tol = lse_bounds_for_rows(x, [0, 1], lambda r: [], SCALE)
    assert np.all(np.abs(lse.cpu().numpy()[:, 0] - ol[:, 0]) <= tol + 1e-5 * (1 + np.abs(ol[:, 0])))


def test_out_of_cache_index_is_reported_not_read(cuda_lib):
    """Indices outside the cache are skipped and reported in the caller's
    status word, read back with the asynchronous check after a caller-side
    synchronisation (an event), also from inside a captured CUDA graph."""
    x = _custom(1, 1, 64, 4, [[1000]], [64])
    idx = torch.tensor([[[3, 64, 1 << 30, -5]]], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([[4]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    host = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    comp = _cache(cuda_lib, x)

    def synced(fn):
        fn()
        ev = torch.cuda.Event()
        ev.record()
        ev.synchronize()
        return int(host.item())

    assert synced(lambda: cuda_lib.csa_check_device_status(host, status=status)) == 0
    cuda_lib.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, 128, idx, cnt, x.q_pos, status=status)
    assert synced(lambda: cuda_lib.csa_check_device_status(host, status=status)) == cuda_lib.ERR_BAD_INDEX
    assert synced(lambda: cuda_lib.csa_check_device_status(host, status=status)) == 0   # the check cleared it
    cuda_lib.csa_gather_swa(comp, x.ring, 128, idx, cnt, x.q_pos, status=status)
    assert synced(lambda: cuda_lib.csa_check_device_status(host, status=status)) == cuda_lib.ERR_BAD_INDEX
    # the binding's default word was not touched by calls given their own
    assert cuda_lib.csa_read_device_error() == 0
    # captured: attention, then the status check, replayed as one graph
    out = torch.empty_like(x.q)
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    ws = cuda_lib.workspace(cuda_lib.OP_ATTENTION, 1, 1, 64, 4, "cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up outside capture (host-side caches)
        cuda_lib.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, 128, idx, cnt, x.q_pos, out=out, lse=lse,
                                           ws=ws, status=status)
        cuda_lib.csa_check_device_status(host, status=status)
    s.synchronize()
    host.fill_(-1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cuda_lib.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, 128, idx, cnt, x.q_pos, out=out, lse=lse,
                                           ws=ws, status=status, stream=s)
        cuda_lib.csa_check_device_status(host, status=status, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert int(host.item()) == cuda_lib.ERR_BAD_INDEX
    good = torch.tensor([[[3, 7, 9, 11]]], dtype=torch.int32, device="cuda")
    idx.copy_(good)
    g.replay()
    torch.cuda.synchronize()
    assert int(host.item()) == 0


def test_late_dominant_candidate_forces_rescale(cuda_lib):
    # 40 sequences (one split each, six 64-candidate chunks); in sequences 0
    # and 7 the newest SWA token (last chunk) is aligned with head 0's query,
    # so that head's running max jumps by far more than 2^8 late in the pass
    # and the accumulated output must be rescaled in place.
    B = 40
    x = _custom(B, 1, 300, 200, [[1200]] * B, [300] * B, seed=11)
    for b, mag in ((0, 1.0), (7, 3.0)):
        q0 = x.q[b, 0, 0].float() * mag
        codes, scales = synth.e4m3_blocks(q0[None, :448], 128)
        rec = synth.pack_records(codes, q0[None, 448:].to(torch.bfloat16), scales)
        x.ring[b, 1200 % x.R] = rec[0]
    lg, idx, cnt = _pipeline(cuda_lib, x)
    out, lse = cuda_lib.csa_sink_attention_decode(x.q, x.sink, SCALE, _cache(cuda_lib, x), x.ring, 128, idx, cnt,
                                                  x.q_pos)
    assert cuda_lib.csa_read_device_error() == 0
    rows = [0, 7, 8]
    oo, ol = oracle.csa_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x),
                                  x.ring.cpu().numpy(), 128, idx.cpu(), cnt.cpu(), x.q_pos.cpu(), threads=THREADS,
                                  rows=rows)
    assert ol[0, 0, 0] > 15 and ol[7, 0, 0] > 50   # the planted token dominates head 0
    gi, gc = idx.cpu().numpy().reshape(-1, 200), cnt.cpu().numpy().reshape(-1)
    tol = lse_bounds_for_rows(x, rows, lambda r: gi[r][:gc[r]], SCALE)
    check_attention(out.float().cpu().numpy().reshape(-1, 128, 512)[rows], lse.cpu().numpy().reshape(-1, 128)[rows],
                    oo.reshape(-1, 128, 512)[rows], ol.reshape(-1, 128)[rows], "rescale", tol)


def test_expired_waits_are_reported_and_the_next_calls_are_correct(cuda_lib):
    """The tensor-core kernels' bounded waits, shortened to 1 ns, expire: the
    kernels record CSA_ERR_TIMEOUT, drain what they issued, free tensor memory
    and exit; with the default limit restored, the same calls on the same
    device give the results they gave before, which match the oracle."""
    x = synth.generate("csa_b8_ctx16k32k_k512", seed=0, device="cuda")
    wl = x.wl
    comp = _cache(cuda_lib, x)
    lg0, idx0, cnt0 = _pipeline(cuda_lib, x)
    out0, lse0 = cuda_lib.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, wl.W, idx0, cnt0, x.q_pos)
    torch.cuda.synchronize()
    assert cuda_lib.csa_read_device_error() == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.csa_debug_set_wait_limit_ns(1)
    try:
        lg1 = cuda_lib.csa_indexer_logits(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q_pos, x.n_comp,
                                          wl.m, status=status)
        torch.cuda.synchronize()
        idx_status = cuda_lib.csa_read_device_error(status=status)
        cuda_lib.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, wl.W, idx0, cnt0, x.q_pos, status=status)
        torch.cuda.synchronize()
        att_status = cuda_lib.csa_read_device_error(status=status)
    finally:
        cuda_lib.csa_debug_set_wait_limit_ns(0)
    assert (idx_status, att_status) == (cuda_lib.ERR_TIMEOUT, cuda_lib.ERR_TIMEOUT)
    del lg1
    # the device is usable and the calls are again exact
    lg2, idx2, cnt2 = _pipeline(cuda_lib, x)
    out2, lse2 = cuda_lib.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, wl.W, idx2, cnt2, x.q_pos,
                                                    status=status)
    torch.cuda.synchronize()
    assert cuda_lib.csa_read_device_error(status=status) == 0
    assert torch.equal(lg2, lg0) and torch.equal(idx2, idx0) and torch.equal(cnt2, cnt0)
    assert torch.equal(out2, out0) and torch.equal(lse2, lse0)
    rows = [0, 5]
    oo, ol = oracle.csa_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x),
                                  x.ring.cpu().numpy(), wl.W, idx2.cpu(), cnt2.cpu(), x.q_pos.cpu(), threads=THREADS,
                                  rows=rows)
    gi, gc = idx2.cpu().numpy().reshape(-1, wl.k), cnt2.cpu().numpy().reshape(-1)
    tol = lse_bounds_for_rows(x, rows, lambda r: gi[r][:gc[r]], SCALE)
    check_attention(out2.float().cpu().numpy().reshape(-1, 128, 512)[rows], lse2.cpu().numpy().reshape(-1, 128)[rows],
                    oo.reshape(-1, 128, 512)[rows], ol.reshape(-1, 128)[rows], "after timeout", tol)
