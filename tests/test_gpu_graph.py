"""The whole decode step under CUDA-graph capture ("ROADMAP -- Stage E",
section E9: once the decode path has no synchronisation and no allocation,
it is capturable): several layers, each with its own paged cache and block
table, captured into one graph. Every replay must reproduce the direct calls
bit for bit, also after the query-side inputs are rewritten in place, and the
replayed selection and outputs of every layer are checked against the
oracle on sampled rows."""
import math
import os
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import check_attention, check_topk_band, lse_bounds_for_rows, oracle_cache

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(512)
LAYERS = 3


def _gpu_cache(csd, x):
    return csd.cache_desc(x.comp, x.wl.ncap, x.seq_stride, x.block_table, x.page_records)


THREADS = os.cpu_count() or 1


def _step(csd, x, comp, out, lse, ws, sel=(None, None)):
    csd.csa_decode_step(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q, x.sink, SCALE, comp, x.ring,
                        x.wl.W, x.q_pos, x.n_comp, x.wl.m, x.wl.k, out=out, lse=lse, ws=ws, topk_idx=sel[0],
                        topk_cnt=sel[1])


def _check_layer_against_oracle(x, out, lse, idx, cnt, rows, what):
    """The replayed selection within the top-k tolerance band of the oracle's
    and the replayed attention against the oracle on that selection."""
    wl = x.wl
    ora = oracle.indexer_logits(x.q_idx.cpu(), x.q_idx_scale.cpu(), x.w_idx.cpu(), x.k_idx.cpu(), x.k_idx_scale.cpu(),
                                x.q_pos.cpu(), x.n_comp.cpu(), wl.m, threads=THREADS, rows=rows)
    ora = ora.reshape(-1, 1, wl.ncap)[rows]
    oi, oc = oracle.topk(ora, np.zeros((len(rows), 1), np.int32) + x.q_pos.cpu().numpy().reshape(-1)[rows][:, None],
                         x.n_comp.cpu().numpy()[[r // wl.T for r in rows]], wl.m, wl.k)
    gi = idx.cpu().numpy().reshape(-1, 1, wl.k)[rows]
    gc = cnt.cpu().numpy().reshape(-1, 1)[rows]
    check_topk_band(gi, gc, ora, oi, oc, wl.k, what)
    oo, ol = oracle.csa_attention(x.q.view(torch.int16).cpu(), x.sink.cpu(), SCALE, oracle_cache(x),
                                  x.ring.cpu().numpy(), wl.W, idx.cpu(), cnt.cpu(), x.q_pos.cpu(), threads=THREADS,
                                  rows=rows)
    fi, fc = idx.cpu().numpy().reshape(-1, wl.k), cnt.cpu().numpy().reshape(-1)
    tol = lse_bounds_for_rows(x, rows, lambda r: fi[r][:fc[r]], SCALE)
    check_attention(out.float().cpu().numpy().reshape(-1, 128, 512)[rows], lse.cpu().numpy().reshape(-1, 128)[rows],
                    oo.reshape(-1, 128, 512)[rows], ol.reshape(-1, 128)[rows], what, tol)


def test_multi_layer_paged_step_graph_replay(cuda_lib):
    csd = cuda_lib
    name = "csa_b8_ctx16k32k_k512"
    layers = [synth.generate(name, seed=10 + i, device="cuda", paged=True) for i in range(LAYERS)]
    wl = layers[0].wl
    assert all(x.block_table is not None for x in layers)
    assert not torch.equal(layers[0].block_table, layers[1].block_table)  # heterogeneous page maps
    comps = [_gpu_cache(csd, x) for x in layers]
    wss = [csd.workspace(csd.OP_DECODE_STEP, wl.B, wl.T, wl.ncap, wl.k, torch.device("cuda")) for _ in layers]
    outs = [(torch.empty_like(x.q), torch.empty((wl.B, wl.T, 128), dtype=torch.float32, device="cuda"))
            for x in layers]
    sels = [(torch.empty((wl.B, wl.T, wl.k), dtype=torch.int32, device="cuda"),
             torch.empty((wl.B, wl.T), dtype=torch.int32, device="cuda")) for _ in layers]

    def direct():
        res = []
        for x, c, w in zip(layers, comps, wss):
            o = torch.empty_like(x.q)
            l = torch.empty((wl.B, wl.T, 128), dtype=torch.float32, device="cuda")
            _step(csd, x, c, o, l, w)
            res.append((o, l))
        torch.cuda.synchronize()
        return res

    want = direct()  # also the warm-up: kernel attributes and tensor maps are set before capture
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for x, c, w, (o, l), sel in zip(layers, comps, wss, outs, sels):
            _step(csd, x, c, o, l, w, sel)
    graph.replay()
    torch.cuda.synchronize()
    for i, ((o, l), (wo, wlse)) in enumerate(zip(outs, want)):
        assert torch.equal(o, wo) and torch.equal(l, wlse), f"layer {i}"

    # new query-side inputs written in place: the replay reads them
    g = torch.Generator(device="cuda").manual_seed(5)
    for x in layers:
        x.q.copy_(torch.randn(x.q.shape, generator=g, device="cuda").to(torch.bfloat16))
        x.w_idx.copy_(torch.randn(x.w_idx.shape, generator=g, device="cuda") / 8.0)
    want = direct()
    graph.replay()
    torch.cuda.synchronize()
    for i, ((o, l), (wo, wlse)) in enumerate(zip(outs, want)):
        assert torch.equal(o, wo) and torch.equal(l, wlse), f"layer {i} after new inputs"
    assert csd.csa_read_device_error() == 0
    # the replayed results of every layer against the oracle
    for i, (x, (o, l), (idx, cnt)) in enumerate(zip(layers, outs, sels)):
        _check_layer_against_oracle(x, o, l, idx, cnt, [0, 5], f"graph replay, layer {i}")

    # replay against direct calls, host clock around 20 iterations of all layers
    def clock(fn, n=20):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / n * 1e6

    def direct_only():
        for x, c, w, (o, l) in zip(layers, comps, wss, outs):
            _step(csd, x, c, o, l, w)

    t_direct = clock(direct_only)
    t_graph = clock(graph.replay)
    print(f"{LAYERS} layers of {name}: direct {t_direct:.1f} us, graph replay {t_graph:.1f} us "
          f"({t_direct / t_graph:.2f}x)")
