"""Seeded synthetic inputs for CSA / HCA decode.

This module serves both the CUDA library's tests and benchmark and the CPU
oracle, and holds none of the method's arithmetic: it draws random numbers,
stores them in the cache formats through library casts (torch's
``float8_e4m3fn`` and ``bfloat16`` conversions, round-to-nearest-even), and
packs bytes into records.

Record layout (one compressed entry or SWA token, 592 bytes, 16-B aligned):

    bytes [0, 448)    448 nope dims, FP8 E4M3
    bytes [448, 576)  64 rope dims, BF16
    bytes [576, 592)  4 fp32 dequantisation scales; scale i covers nope dims
                      [128 i, min(128 i + 128, 448)) (the last block has 64)

Stored scale = amax(|block|) / 448 (1 when the block is all zero), code =
e4m3(x / scale): the FP8-with-scale storage the pages describe for the
latent's nope dims ("DSV4 Audit", B1) and for the indexer keys (B2).

Distributions (same for every workload): latents, SWA tokens and q ~ N(0,1);
sink logits ~ N(0,1); indexer q and keys ~ N(0,1) before FP8 quantisation
with one scale per (token, head) and per key; indexer head weights ~
N(0, 1/64).
"""
from __future__ import annotations

import dataclasses
import math

import torch

H, D, DN, DR, SB = 128, 512, 448, 64, 128
HI, DI = 64, 128
W_SWA = 128
REC_BYTES = DN + 2 * DR + 4 * ((DN + SB - 1) // SB)  # 592
E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode step's shape. ``ctx`` is the context length in tokens; the
    query of a sequence with context L sits at 0-based position L."""
    name: str
    kind: str              # "csa" or "hca"
    B: int
    T: int
    ncap: int              # compressed-entry capacity per sequence
    m: int                 # tokens per compressed entry (4 CSA, 128 HCA)
    k: int                 # top-k (CSA only)
    ctx: int | None        # fixed context length, or None for per-sequence draws
    ctx_range: tuple[int, int] | None = None
    W: int = W_SWA


WORKLOADS = {
    w.name: w for w in [
        Workload("csa_b1_ctx1k_k64", "csa", B=1, T=1, ncap=256, m=4, k=64, ctx=1024),
        Workload("csa_b8_ctx16k32k_k512", "csa", B=8, T=1, ncap=8192, m=4, k=512, ctx=None,
                 ctx_range=(16384, 32768)),
        Workload("csa_b32_ctx128k_k2048", "csa", B=32, T=1, ncap=32768, m=4, k=2048, ctx=131072),
        Workload("csa_b4t4_ctx1m_k2048", "csa", B=4, T=4, ncap=262144, m=4, k=2048, ctx=1 << 20),
        Workload("hca_b64_ctx1m", "hca", B=64, T=1, ncap=8192, m=128, k=0, ctx=1 << 20),
    ]
}
HEADLINE = "csa_b32_ctx128k_k2048"


@dataclasses.dataclass
class Inputs:
    wl: Workload
    q: torch.Tensor            # [B,T,H,D] bfloat16
    sink: torch.Tensor         # [H] float32
    comp: torch.Tensor         # [n_records, REC_BYTES] uint8
    seq_stride: int            # records per sequence when block_table is None
    block_table: torch.Tensor | None   # [B, max_pages] int32
    page_records: int
    ring: torch.Tensor         # [B, R, REC_BYTES] uint8
    q_pos: torch.Tensor        # [B,T] int32
    n_comp: torch.Tensor       # [B] int32
    q_idx: torch.Tensor | None          # [B,T,HI,DI] uint8 (e4m3 codes)
    q_idx_scale: torch.Tensor | None    # [B,T,HI] float32
    w_idx: torch.Tensor | None          # [B,T,HI] float32
    k_idx: torch.Tensor | None          # [B,ncap,DI] uint8 (e4m3 codes)
    k_idx_scale: torch.Tensor | None    # [B,ncap] float32

    @property
    def R(self) -> int:
        return int(self.ring.shape[1])

    def to(self, device) -> "Inputs":
        kw = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            kw[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return Inputs(**kw)

    def clone(self) -> "Inputs":
        kw = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            kw[f.name] = v.clone() if isinstance(v, torch.Tensor) else v
        return Inputs(**kw)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def e4m3_blocks(x: torch.Tensor, block: int):
    """Quantise the last dim of x (float32) to E4M3 codes with one fp32 scale
    per ``block`` elements (ragged last block). Returns (uint8 codes, scales)."""
    d = x.shape[-1]
    nblk = (d + block - 1) // block
    codes, scales = [], []
    for i in range(nblk):
        xb = x[..., i * block:min(d, (i + 1) * block)]
        amax = xb.abs().amax(dim=-1, keepdim=True)
        s = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
        c = (xb / s).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
        codes.append(c)
        scales.append(s)
    return torch.cat(codes, dim=-1), torch.cat(scales, dim=-1).to(torch.float32)


def pack_records(nope_codes: torch.Tensor, rope: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """Byte-pack [..., DN] uint8, [..., DR] bf16, [..., nblk] fp32 into
    [..., REC_BYTES] uint8."""
    lead = nope_codes.shape[:-1]
    parts = [nope_codes.contiguous(),
             rope.contiguous().view(torch.uint8).reshape(*lead, -1),
             scales.contiguous().view(torch.uint8).reshape(*lead, -1)]
    rec = torch.cat(parts, dim=-1)
    assert rec.shape[-1] == REC_BYTES
    return rec


def random_records(n: int, g: torch.Generator, device, chunk: int = 1 << 16) -> torch.Tensor:
    """n latent records from N(0,1) (nope quantised per 128-dim block, rope BF16)."""
    out = torch.empty((n, REC_BYTES), dtype=torch.uint8, device=device)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn((e - s, D), generator=g, device=device, dtype=torch.float32)
        codes, scales = e4m3_blocks(x[:, :DN], SB)
        out[s:e] = pack_records(codes, x[:, DN:].to(torch.bfloat16), scales)
    return out


def positions(wl: Workload, g: torch.Generator, device):
    """q_pos [B,T] and n_comp [B] for a workload. Tokens of one sequence are
    consecutive; sequence b of the 1M-context T=4 workload starts at 2^20-4+b,
    so its tokens straddle a block boundary and differ in visible range."""
    B, T = wl.B, wl.T
    if wl.ctx is None:
        lo, hi = wl.ctx_range
        L = torch.randint(lo, hi + 1, (B,), generator=g, device=device, dtype=torch.int64)
        q_pos = L[:, None] + torch.arange(T, device=device)[None, :]
        n_comp = torch.clamp(L // wl.m, max=wl.ncap)
    elif T > 1:
        base = wl.ctx - T + torch.arange(B, device=device)
        q_pos = base[:, None] + torch.arange(T, device=device)[None, :]
        n_comp = torch.full((B,), wl.ncap, device=device, dtype=torch.int64)
    else:
        q_pos = torch.full((B, T), wl.ctx, device=device, dtype=torch.int64)
        n_comp = torch.full((B,), min(wl.ncap, wl.ctx // wl.m), device=device, dtype=torch.int64)
    return q_pos.to(torch.int32).contiguous(), n_comp.to(torch.int32).contiguous()


def generate(wl: Workload | str, seed: int = 0, device="cpu", paged: bool = False,
             page_records: int | None = None) -> Inputs:
    """Draw one decode step's inputs. With ``paged``, the compressed cache is a
    pool of 128-token pages (32 CSA entries, 1 HCA entry per page) addressed
    through a block table holding a seeded random permutation of the pages."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    device = torch.device(device)
    g = _gen(seed, device)
    B, T = wl.B, wl.T
    q_pos, n_comp = positions(wl, g, device)
    q = torch.randn((B, T, H, D), generator=g, device=device).to(torch.bfloat16)
    sink = torch.randn((H,), generator=g, device=device, dtype=torch.float32)
    comp = random_records(B * wl.ncap, g, device)
    R = wl.W + T - 1
    ring = random_records(B * R, g, device).view(B, R, REC_BYTES)
    block_table = None
    seq_stride = wl.ncap
    pr = page_records or (128 // wl.m)
    if paged:
        max_pages = (wl.ncap + pr - 1) // pr
        n_pages = B * max_pages
        perm = torch.randperm(n_pages, generator=g, device=device).to(torch.int32)
        block_table = perm.view(B, max_pages).contiguous()
        # physical page block_table[b, j] holds logical entries [j*pr, (j+1)*pr) of b
        pool = torch.zeros((n_pages * pr, REC_BYTES), dtype=torch.uint8, device=device)
        logical = comp.view(B, wl.ncap, REC_BYTES)
        padded = torch.zeros((B, max_pages * pr, REC_BYTES), dtype=torch.uint8, device=device)
        padded[:, :wl.ncap] = logical
        pool.view(n_pages, pr, REC_BYTES)[block_table.view(-1).long()] = padded.view(B * max_pages, pr, REC_BYTES)
        comp = pool
        seq_stride = 0
    q_idx = q_idx_scale = w_idx = k_idx = k_idx_scale = None
    if wl.kind == "csa":
        qi = torch.randn((B, T, HI, DI), generator=g, device=device)
        q_idx, q_idx_scale = e4m3_blocks(qi, DI)
        q_idx_scale = q_idx_scale[..., 0].contiguous()
        w_idx = (torch.randn((B, T, HI), generator=g, device=device) / math.sqrt(HI)).contiguous()
        k_idx = torch.empty((B, wl.ncap, DI), dtype=torch.uint8, device=device)
        k_idx_scale = torch.empty((B, wl.ncap), dtype=torch.float32, device=device)
        for b in range(B):
            for s in range(0, wl.ncap, 1 << 16):
                e = min(wl.ncap, s + (1 << 16))
                ki = torch.randn((e - s, DI), generator=g, device=device)
                c, sc = e4m3_blocks(ki, DI)
                k_idx[b, s:e] = c
                k_idx_scale[b, s:e] = sc[:, 0]
    return Inputs(wl=wl, q=q.contiguous(), sink=sink, comp=comp.contiguous(), seq_stride=seq_stride,
                  block_table=block_table, page_records=pr, ring=ring.contiguous(), q_pos=q_pos,
                  n_comp=n_comp, q_idx=q_idx, q_idx_scale=q_idx_scale, w_idx=w_idx, k_idx=k_idx,
                  k_idx_scale=k_idx_scale)


def custom(kind: str, B: int, T: int, ncap: int, k: int, ctx: int | None = None, m: int | None = None,
           ctx_range=None, W: int = W_SWA, name: str = "custom") -> Workload:
    """A workload of arbitrary size for edge-case tests."""
    return Workload(name, kind, B=B, T=T, ncap=ncap, m=m or (4 if kind == "csa" else 128), k=k,
                    ctx=ctx, ctx_range=ctx_range, W=W)
