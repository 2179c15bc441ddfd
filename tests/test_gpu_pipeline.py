"""The host-I/O pipeline (csa_decode_step_host): every step's host results
equal csa_decode_step's on the same inputs, bit for bit, whatever the depth,
with steps enqueued back to back (copies overlapping kernels) and with host
buffers reused after csa_pipeline_wait."""
import math

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(512)
STEPS = 5


def step_inputs(x, j):
    """Query-side inputs of step j (step 0 = the workload's own), pinned host tensors."""
    B, T = x.wl.B, x.wl.T
    g = torch.Generator().manual_seed(1000 + j)
    if j == 0:
        q_idx, q_idx_scale, w_idx, q, q_pos = (t.cpu() for t in (x.q_idx, x.q_idx_scale, x.w_idx, x.q, x.q_pos))
    else:
        codes = torch.randint(0, 0x7E, (B, T, 64, 128), generator=g, dtype=torch.int32)
        sign = torch.randint(0, 2, (B, T, 64, 128), generator=g, dtype=torch.int32) << 7
        q_idx = (codes | sign).to(torch.uint8).view(x.q_idx.dtype)
        q_idx_scale = torch.rand((B, T, 64), generator=g) * 0.1 + 0.01
        w_idx = torch.randn((B, T, 64), generator=g) / 8.0
        q = torch.randn((B, T, 128, 512), generator=g).to(torch.bfloat16)
        q_pos = torch.clamp(x.q_pos.cpu() - 3 * j, min=0)
    return [t.contiguous().pin_memory() for t in (q_idx, q_idx_scale, w_idx, q, q_pos)]


def expected(csd, x, comp, ins):
    dev = [t.cuda() for t in ins]
    out, lse = csd.csa_decode_step(dev[0], dev[1], dev[2], x.k_idx, x.k_idx_scale, dev[3], x.sink, SCALE, comp, x.ring,
                                   x.wl.W, dev[4], x.n_comp, x.wl.m, x.wl.k)
    return out.cpu(), lse.cpu()


def host_out(x):
    B, T = x.wl.B, x.wl.T
    return (torch.empty((B, T, 128, 512), dtype=torch.bfloat16).pin_memory(),
            torch.empty((B, T, 128), dtype=torch.float32).pin_memory())


# 16 tokens a sequence: the indexer's token groups inside the pipelined step
CUSTOM = {"csa_b2t16_ctx20k_k128": synth.custom("csa", B=2, T=16, ncap=5000, k=128, ctx=20000,
                                               name="csa_b2t16_ctx20k_k128")}


@pytest.mark.parametrize("name,depth", [("csa_b1_ctx1k_k64", 2), ("csa_b8_ctx16k32k_k512", 2),
                                        ("csa_b8_ctx16k32k_k512", 3), ("csa_b4t4_ctx1m_k2048", 4),
                                        ("csa_b2t16_ctx20k_k128", 2)])
def test_pipeline_matches_decode_step(cuda_lib, name, depth):
    csd = cuda_lib
    x = synth.generate(CUSTOM.get(name, name), seed=0, device="cuda")
    comp = csd.cache_desc(x.comp, x.wl.ncap, x.seq_stride)
    ins = [step_inputs(x, j) for j in range(STEPS)]
    want = [expected(csd, x, comp, i) for i in ins]
    ws = csd.workspace(csd.OP_DECODE_STEP, x.wl.B, x.wl.T, x.wl.ncap, x.wl.k, x.q.device)
    pl = csd.HostPipeline(x.wl.B, x.wl.T, depth=depth)
    try:
        outs = [host_out(x) for _ in range(STEPS)]
        # back to back: no wait between steps
        steps = [pl.step(*ins[j], x.k_idx, x.k_idx_scale, x.sink, SCALE, comp, x.ring, x.wl.W, x.n_comp, x.wl.m,
                         x.wl.k, *outs[j], ws) for j in range(STEPS)]
        assert steps == list(range(STEPS))
        for j in range(STEPS):
            pl.wait(j)
            assert torch.equal(outs[j][0], want[j][0]), f"step {j} out"
            assert torch.equal(outs[j][1], want[j][1]), f"step {j} lse"
        # one host buffer set reused: refilled only after the previous step's wait
        buf = [torch.empty_like(t).pin_memory() for t in ins[0]]
        ob = host_out(x)
        for j in (3, 1, 4):
            for d, s in zip(buf, ins[j]):
                d.copy_(s)
            i = pl.step(*buf, x.k_idx, x.k_idx_scale, x.sink, SCALE, comp, x.ring, x.wl.W, x.n_comp, x.wl.m, x.wl.k,
                        *ob, ws)
            pl.wait(i)
            assert torch.equal(ob[0], want[j][0]) and torch.equal(ob[1], want[j][1]), f"reused buffers, step {j}"
        with pytest.raises(csd.CsaError):
            pl.wait(10 ** 6)  # not enqueued
        pl.sync()
        assert csd.csa_read_device_error() == 0
    finally:
        pl.close()


def test_pipeline_rejects_device_tensors_for_host_arguments(cuda_lib):
    csd = cuda_lib
    x = synth.generate("csa_b1_ctx1k_k64", seed=0, device="cuda")
    comp = csd.cache_desc(x.comp, x.wl.ncap, x.seq_stride)
    ws = csd.workspace(csd.OP_DECODE_STEP, x.wl.B, x.wl.T, x.wl.ncap, x.wl.k, x.q.device)
    pl = csd.HostPipeline(x.wl.B, x.wl.T)
    try:
        ins = step_inputs(x, 0)
        ins[3] = x.q  # a device tensor where host memory is expected
        with pytest.raises(ValueError):
            pl.step(*ins, x.k_idx, x.k_idx_scale, x.sink, SCALE, comp, x.ring, x.wl.W, x.n_comp, x.wl.m, x.wl.k,
                    *host_out(x), ws)
        # a bad device argument is rejected before anything is enqueued: the
        # next step still gets ordinal 0
        ins = step_inputs(x, 0)
        with pytest.raises(csd.CsaError):
            pl.step(*ins, x.k_idx, x.k_idx_scale, x.sink, 0.0, comp, x.ring, x.wl.W, x.n_comp, x.wl.m, x.wl.k,
                    *host_out(x), ws)
        assert pl.step(*ins, x.k_idx, x.k_idx_scale, x.sink, SCALE, comp, x.ring, x.wl.W, x.n_comp, x.wl.m, x.wl.k,
                       *host_out(x), ws) == 0
        pl.sync()
    finally:
        pl.close()
