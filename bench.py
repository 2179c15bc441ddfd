#!/usr/bin/env python
"""Benchmark of one CSA decode layer step on GB300.

A step is one pass of the whole hot path over one batch of query tokens:
lightning-indexer logits -> top-k -> sink-merged attention over the selected
entries and the SWA window (the gather is fused into the attention kernel).
The default workload is 32 sequences at 128K context (32768 compressed
entries each), top-k 2048, SWA 128.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the CPU oracle on a bounded sample)

Prints one JSON line (rank 0). With N > 1 (torchrun), every rank runs an
independent replica on its own GPU (the path has no exchange step): weak
scaling, value = tokens of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import ctypes as C
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA decode tokens/s at 128K ctx; achieved HBM GB/s and % of roofline"
UNIT = "tokens/s"
SCALE = 1.0 / math.sqrt(512)
N_COPIES = 3  # rotating input copies: each step's inputs are not L2-resident
SAMPLE_EVERY = 8  # timed-region steps: the indexer is bracketed by events on steps i % 8 == 0, the attention on i % 8 == 4


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--report-configs", action="store_true",
                    help="print one JSON line of per-kernel times for every workload instead of the benchmark line")
    ap.add_argument("--epilogue", action="store_true",
                    help="time the attention with its output epilogues (inverse RoPE, E2M1 output)")
    ap.add_argument("--prefill", type=int, default=0, metavar="T",
                    help="time T tokens of one 128K sequence as one step against T single-token steps")
    ap.add_argument("--graph-replay", type=int, default=0, metavar="LAYERS",
                    help="time LAYERS decode steps (one per layer, each with its own paged cache) as direct calls "
                         "and as one replayed CUDA graph, on --workload (default: the 1K-context one)")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(values, device, world: int) -> list[float]:
    """Element-wise maximum of per-rank timings over all ranks (the slowest
    rank sets the whole job's time); identity on one rank."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(units_per_rank: int, world: int, ms: float) -> float:
    """Units of all ranks per second of the slowest rank (weak scaling)."""
    return units_per_rank * world / (ms / 1e3)


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.samples: list[tuple[float, list[str]]] = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        mine = [(t, p) for t, p in self.samples if not self.uuid or self.uuid in p[0]]
        inside = [(t, p) for t, p in mine if t0 - 0.05 <= t <= t1 + 0.05]
        window = "timed region"
        if not inside and mine:  # region shorter than the sampling period: nearest samples
            mine.sort(key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))
            inside = mine[:3]
            window = "nearest samples to a timed region shorter than the sampling period"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        reasons = set()
        for _, p in inside:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), p[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(inside[0][1][2]),
                "power_w_max": max((num(p[3]) or 0.0) for _, p in inside), "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


# --------------------------------------------------------------------------
# algorithmic bytes (the roofline's numerator)
# --------------------------------------------------------------------------

def indexer_bytes(x) -> int:
    """Bytes the indexer must move per launch: each key visible to any token
    of its sequence (128 B codes + 4 B scale, read once for all T tokens),
    each token's indexer query (64x128 B codes + 64 fp32 scales + 64 fp32
    weights + position), and the fp32 logits row written in full."""
    import numpy as np
    wl = x.wl
    q_pos = x.q_pos.cpu().numpy()
    n_comp = x.n_comp.cpu().numpy()
    nv = np.minimum(np.minimum(q_pos // wl.m, n_comp[:, None]), wl.ncap).max(axis=1)
    keys = int(nv.sum()) * (128 + 4)
    per_tok = 64 * 128 + 64 * 4 + 64 * 4 + 4
    return keys + wl.B * wl.T * (per_tok + 4 * wl.ncap)


def attention_work(cnt, x) -> tuple[int, float]:
    """Bytes the attention must move and the flops it must do: 592 B and
    2 x 128 x 512 x 2 flops (QK and PV) per candidate record per query (top-k
    entries + SWA window), plus the BF16 query and output rows (128 KB each)
    and the fp32 LSE."""
    import numpy as np
    q_pos = x.q_pos.cpu().numpy().reshape(-1)
    nswa = np.minimum(q_pos + 1, x.wl.W)
    cands = int(cnt.sum()) + int(nswa.sum())
    return cands * 592 + x.wl.B * x.wl.T * (2 * 128 * 512 * 2 + 128 * 4), 262144.0 * cands


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

class Runner:
    """Pre-marshalled C-ABI calls for one input copy (pointers computed once,
    so the timed loop spends its host time in the library, not in Python)."""

    def __init__(self, csd, x, stream):
        import torch
        self.csd, self.x, self.lib = csd, x, csd.load()
        wl = x.wl
        B, T, N, k = wl.B, wl.T, wl.ncap, wl.k
        dev = x.q.device
        self.logits = torch.empty((B, T, N), dtype=torch.float32, device=dev)
        self.idx = torch.empty((B, T, k), dtype=torch.int32, device=dev)
        self.cnt = torch.empty((B, T), dtype=torch.int32, device=dev)
        self.out = torch.empty((B, T, 128, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, T, 128), dtype=torch.float32, device=dev)
        self.ws_topk = csd.workspace(csd.OP_TOPK, B, T, N, k, dev)
        self.ws_att = csd.workspace(csd.OP_ATTENTION, B, T, N, k, dev)
        self.ws_step = csd.workspace(csd.OP_DECODE_STEP, B, T, N, k, dev)
        self.comp = csd.cache_desc(x.comp, N, x.seq_stride, x.block_table,
                                   x.page_records if x.block_table is not None else 0)
        s = C.c_void_p(stream.cuda_stream)
        p = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None
        st = p(csd.status_word(dev))
        nb = lambda t: C.c_size_t(0 if t is None else t.numel())
        R = x.ring.shape[1]
        self.a_idx = [p(x.q_idx), p(x.q_idx_scale), p(x.w_idx), p(x.k_idx), p(x.k_idx_scale), p(x.q_pos),
                      p(x.n_comp), B, T, N, wl.m, p(self.logits), st, s]
        self.a_topk = [p(self.logits), p(x.q_pos), p(x.n_comp), B, T, N, wl.m, k, p(self.idx), p(self.cnt),
                       p(self.ws_topk), nb(self.ws_topk), st, s]
        self.a_att = [p(x.q), p(x.sink), C.c_float(SCALE), self.comp, p(x.ring), R, wl.W, p(self.idx), p(self.cnt),
                      p(x.q_pos), B, T, k, p(self.out), p(self.lse), p(self.ws_att), nb(self.ws_att), st, s]
        self.a_step = [p(x.q_idx), p(x.q_idx_scale), p(x.w_idx), p(x.k_idx), p(x.k_idx_scale), p(x.q), p(x.sink),
                       C.c_float(SCALE), self.comp, p(x.ring), R, wl.W, p(x.q_pos), p(x.n_comp), B, T, N, wl.m, k,
                       p(self.out), p(self.lse), None, None, p(self.ws_step), nb(self.ws_step), st, s]

    def indexer(self):
        st = self.lib.csa_indexer_logits(*self.a_idx)
        if st:
            raise RuntimeError(f"csa_indexer_logits: {self.csd.status_string(st)}")

    def topk(self):
        st = self.lib.csa_topk(*self.a_topk)
        if st:
            raise RuntimeError(f"csa_topk: {self.csd.status_string(st)}")

    def attention(self):
        st = self.lib.csa_sink_attention_decode(*self.a_att)
        if st:
            raise RuntimeError(f"csa_sink_attention_decode: {self.csd.status_string(st)}")

    def decode_step(self):
        st = self.lib.csa_decode_step(*self.a_step)
        if st:
            raise RuntimeError(f"csa_decode_step: {self.csd.status_string(st)}")


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import compressed_sparse_decode_gb300 as csd
    import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    csd.build()
    csd.load()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    name = args.workload or synth.HEADLINE
    base = synth.generate(name, seed=0, device=dev)
    wl = base.wl
    if wl.kind != "csa":
        raise SystemExit("the decode-step benchmark runs a CSA workload")
    copies = [base] + [base.clone() for _ in range(N_COPIES - 1)]
    stream = torch.cuda.Stream(device=dev)
    runners = [Runner(csd, x, stream) for x in copies]

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # warm-up: at least W steps and about half a second of continuous work
    with torch.cuda.stream(stream):
        t_end = time.time() + 0.5
        i = 0
        while i < args.warmup or time.time() < t_end:
            r = runners[i % N_COPIES]
            r.indexer(); r.topk(); r.attention()
            i += 1
            if i % 20 == 0:
                stream.synchronize()
    stream.synchronize()
    if csd.csa_read_device_error(stream):
        raise RuntimeError("device error word set during warm-up")

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    # Events inside the timed loop bracket the two roofline kernels, each on
    # one step in SAMPLE_EVERY (the indexer on steps i % 8 == 0, the attention
    # with its split combine on steps i % 8 == 4): an event between two kernels
    # stops the next one from being set up while its predecessor drains
    # (programmatic dependent launch), which costs a few us per bracket.
    ev_idx = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for i in range(args.steps) if i % SAMPLE_EVERY == 0}
    ev_att = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for i in range(args.steps) if i % SAMPLE_EVERY == SAMPLE_EVERY // 2}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # keep the GPU busy right up to the timed region (clock samples stay meaningful)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            r = runners[i % N_COPIES]
            r.indexer(); r.topk(); r.attention()
    barrier()
    torch.cuda.synchronize(dev)
    launches0 = csd.csa_kernel_launches()
    t0 = time.time()
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(args.steps):
            r = runners[i % N_COPIES]
            if i in ev_idx:
                ev_idx[i][0].record(stream)
                r.indexer()
                ev_idx[i][1].record(stream)
            else:
                r.indexer()
            r.topk()
            if i in ev_att:
                ev_att[i][0].record(stream)
                r.attention()
                ev_att[i][1].record(stream)
            else:
                r.attention()
        end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier()
    launches = csd.csa_kernel_launches() - launches0
    time.sleep(0.1)
    clocks.stop()
    total_ms = start.elapsed_time(end)
    t_idx = [a.elapsed_time(b) for a, b in ev_idx.values()]
    t_att_live = [a.elapsed_time(b) for a, b in ev_att.values()]
    # per-kernel breakdown (after the timed region, same inputs): events around
    # every kernel, which serialises their boundaries
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(min(args.steps, 12))]
    with torch.cuda.stream(stream):
        for i, (b0, b1, b2, b3) in enumerate(bev):
            r = runners[i % N_COPIES]
            b0.record(stream); r.indexer(); b1.record(stream); r.topk(); b2.record(stream); r.attention(); b3.record(stream)
    torch.cuda.synchronize(dev)
    t_topk = [b.elapsed_time(c) for _, b, c, _ in bev]
    t_att = [c.elapsed_time(d) for _, _, c, d in bev]
    (total_ms,) = max_over_ranks([total_ms], dev, world)
    if csd.csa_read_device_error(stream):
        raise RuntimeError("device error word set during the timed region")

    value = job_throughput(wl.B * wl.T * args.steps, world, total_ms)
    peaks = load_peaks()
    idx_bytes = indexer_bytes(base)
    att_bytes, att_flops = attention_work(runners[0].cnt.cpu().numpy(), base)
    idx_ms = statistics.mean(t_idx)
    att_ms = statistics.mean(t_att_live) if t_att_live else statistics.mean(t_att)
    idx_gbs = idx_bytes / (idx_ms / 1e3) / 1e9
    att_gbs = att_bytes / (att_ms / 1e3) / 1e9
    att_tflops = att_flops / (att_ms / 1e3) / 1e12

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3xe4m3->f32 indexer; bf16xbf16->f32 attention",
        "data": "synthetic (seeded N(0,1) latents/queries, FP8 E4M3 per-block scales; no weights needed)",
        "config": {"workload": name, "batch": wl.B, "tokens_per_seq": wl.T, "context_tokens": wl.ctx,
                   "compressed_entries": wl.ncap, "m": wl.m, "topk": wl.k, "swa": wl.W,
                   "l2": f"inputs larger than L2: {N_COPIES} rotating copies, each step reads a different one",
                   "parallelism": f"replicas x{world}"},
        "kernel_ms": {"indexer": round(idx_ms, 5), "topk": round(statistics.mean(t_topk), 5),
                      "attention": round(att_ms, 5),
                      "source": f"indexer and attention (+ split combine): events around one launch in "
                                f"{SAMPLE_EVERY} in the timed region ({len(t_idx)} and {len(t_att_live)} launches); "
                                "topk: a breakdown pass after it with events around every kernel"},
        # the dominant kernel (the attention and its split combine, the largest
        # share of the step): algorithmic bytes / its mean live launch time
        "roofline": {"kernel": "attention_tc_kernel + attention_combine_kernel", "bound": "hbm",
                     "achieved": round(att_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(att_gbs / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
                     "traffic": measured_traffic("attention_traffic.json", name, ("attention.cu",)),
                     "algorithmic_bytes": att_bytes, "flops": att_flops,
                     "tensor": {"dtype": "bf16", "achieved_tflops": round(att_tflops, 1),
                                "peak_tflops": peaks["bf16_tflops"],
                                "frac": round(att_tflops / peaks["bf16_tflops"], 4)}},
        "roofline_indexer": {"kernel": "indexer_tc_kernel", "bound": "hbm", "achieved": round(idx_gbs, 1),
                             "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(idx_gbs / peaks["hbm_gbs"], 4),
                             "peak_source": peaks["source"],
                             "traffic": measured_traffic("indexer_traffic.json", name, ("indexer.cu",)),
                             "algorithmic_bytes": idx_bytes},
        "gpu_launches": launches,
        "clocks": clocks.summary(t0, t1),
    }
    if not args.no_e2e:
        line["e2e"] = run_e2e(args, csd, copies, runners, stream, dev, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(base)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_e2e(args, csd, copies, runners, stream, dev, world):
    """Same metric through the public host-I/O entry point, csa_decode_step_host:
    every step copies its query-side inputs (q_idx, q_idx_scale, w_idx, q,
    q_pos) from pinned host memory, runs the decode step, and copies out and
    lse back to pinned host memory. The caches (compressed entries, indexer
    keys, SWA ring) are the layer's device-resident state, as in decode. The
    pipeline's copy streams overlap a step's copies with its neighbours'
    kernels (2 staging slots). Timed on the host clock, from a synchronised
    start to csa_pipeline_sync, max over ranks. `serialized` is the same loop
    with every copy and kernel in order on one stream (csa_decode_step between
    torch copies), for comparison."""
    import time

    import torch
    lib = csd.load()
    host_in = []
    for x in copies:
        host_in.append([t.cpu().pin_memory() for t in (x.q_idx, x.q_idx_scale, x.w_idx, x.q, x.q_pos)])
    host_out = [(torch.empty_like(r.out, device="cpu").pin_memory(), torch.empty_like(r.lse, device="cpu").pin_memory())
                for r in runners]
    bi = sum(t.numel() * t.element_size() for t in host_in[0])
    bo = sum(t.numel() * t.element_size() for t in host_out[0])
    wl = copies[0].wl
    pl = csd.HostPipeline(wl.B, wl.T, depth=2, device=dev, stream=stream)
    p = lambda t: C.c_void_p(t.data_ptr())
    step_args = []
    for i, (x, r) in enumerate(zip(copies, runners)):
        hi, (ho, hl) = host_in[i], host_out[i]
        step_args.append([C.c_void_p(pl.handle), p(hi[0]), p(hi[1]), p(hi[2]), p(hi[3]), p(hi[4]), p(x.k_idx),
                          p(x.k_idx_scale), p(x.sink), C.c_float(SCALE), r.comp, p(x.ring), x.ring.shape[1], wl.W,
                          p(x.n_comp), wl.ncap, wl.m, wl.k, p(ho), p(hl), p(r.ws_step), C.c_size_t(r.ws_step.numel()),
                          p(csd.status_word(dev)), None])

    def pipelined(n):
        for i in range(n):
            st = lib.csa_decode_step_host(*step_args[i % N_COPIES])
            if st:
                raise RuntimeError(f"csa_decode_step_host: {csd.status_string(st)}")

    def timed(fn, n):
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        fn(n)
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t0) * 1e3

    def serial(n):
        with torch.cuda.stream(stream):
            for i in range(n):
                x, r = copies[i % N_COPIES], runners[i % N_COPIES]
                for dst, src in zip((x.q_idx, x.q_idx_scale, x.w_idx, x.q, x.q_pos), host_in[i % N_COPIES]):
                    dst.copy_(src, non_blocking=True)
                r.decode_step()
                ho, hl = host_out[i % N_COPIES]
                ho.copy_(r.out, non_blocking=True)
                hl.copy_(r.lse, non_blocking=True)

    def sync_pl(n):
        pipelined(n)
        pl.sync()

    timed(sync_pl, max(args.warmup, 3))
    ms = timed(sync_pl, args.steps)
    timed(serial, max(args.warmup, 3))
    ms_serial = timed(serial, args.steps)
    pl.close()
    ms, ms_serial = max_over_ranks([ms, ms_serial], dev, world)
    tok = wl.B * wl.T * args.steps
    return {"value": round(job_throughput(tok, world, ms), 1), "unit": UNIT,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": round(ms / args.steps, 5),
            "call": "csa_decode_step_host (host inputs and outputs; copies overlap neighbouring steps' kernels)",
            "clock": "host wall clock, synchronised start to csa_pipeline_sync",
            "serialized": {"value": round(job_throughput(tok, world, ms_serial), 1),
                           "ms_per_step": round(ms_serial / args.steps, 5),
                           "call": "torch H2D copies, csa_decode_step, torch D2H copies, one stream"}}


def kernel_hash(files=("indexer.cu",)) -> str:
    """Hash of a kernel's sources (with the shared headers): a recorded ncu
    traffic figure is used only while it matches."""
    import hashlib
    h = hashlib.sha256()
    for f in tuple(files) + ("common.cuh", "ptx.cuh"):
        h.update(open(os.path.join(ROOT, "compressed_sparse_decode_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(record: str, workload: str, files) -> int | None:
    """DRAM bytes per launch from a committed ncu record under profiles/, or
    None when there is none for this workload or the kernel changed since."""
    p = os.path.join(ROOT, "profiles", record)
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("workload") == workload and d.get("kernel_source_hash") == kernel_hash(files):
        return d.get("dram_bytes_per_launch")
    return None


# --------------------------------------------------------------------------
# the oracle (CPU baseline and reference arm)
# --------------------------------------------------------------------------

def _oracle_host_inputs(x):
    import oracle
    import torch
    h = {"q_idx": x.q_idx.cpu(), "q_idx_scale": x.q_idx_scale.cpu(), "w_idx": x.w_idx.cpu(), "k_idx": x.k_idx.cpu(),
         "k_idx_scale": x.k_idx_scale.cpu(), "q_pos": x.q_pos.cpu(), "n_comp": x.n_comp.cpu(),
         "q": x.q.view(torch.int16).cpu(), "sink": x.sink.cpu(), "ring": x.ring.cpu().numpy()}
    h["cache"] = oracle.Cache(x.comp.cpu().numpy(), seq_stride=x.seq_stride, seq_capacity=x.wl.ncap)
    return h


def _oracle_rows(h, wl, rows, threads):
    """The oracle's full step (indexer -> top-k -> attention) on query rows."""
    import numpy as np
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    def one(r):
        lg = oracle.indexer_logits(h["q_idx"], h["q_idx_scale"], h["w_idx"], h["k_idx"], h["k_idx_scale"], h["q_pos"],
                                   h["n_comp"], wl.m, rows=[r])
        b = r // wl.T
        sl = lg.reshape(-1, wl.ncap)[r][None, None]
        idx, cnt = oracle.topk(sl, h["q_pos"].numpy().reshape(-1)[r:r + 1][None], h["n_comp"].numpy()[b:b + 1],
                               wl.m, wl.k)
        full_idx = np.full((wl.B * wl.T, wl.k), -1, np.int32)
        full_cnt = np.zeros((wl.B * wl.T,), np.int32)
        full_idx[r], full_cnt[r] = idx[0, 0], cnt[0, 0]
        oracle.csa_attention(h["q"], h["sink"], SCALE, h["cache"], h["ring"], wl.W,
                             full_idx.reshape(wl.B, wl.T, wl.k), full_cnt.reshape(wl.B, wl.T), h["q_pos"], rows=[r])

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, rows))


def cpu_baseline(x) -> dict:
    """The oracle (as it stands) on the host cores: the whole step of the
    workload (every query token: indexer, top-k, attention), one token per
    thread on os.cpu_count() threads; plus a 1-thread timing of the two small
    workloads (1K and 16K-32K context), whole."""
    import synth
    cores = os.cpu_count() or 1
    wl = x.wl
    h = _oracle_host_inputs(x)
    rows = list(range(wl.B * wl.T))
    t0 = time.time()
    _oracle_rows(h, wl, rows, cores)
    dt = time.time() - t0
    single = {}
    for small in ("csa_b1_ctx1k_k64", "csa_b8_ctx16k32k_k512"):
        xs = synth.generate(small, seed=0, device="cpu")
        hs = _oracle_host_inputs(xs)
        n = xs.wl.B * xs.wl.T
        ts = time.time()
        _oracle_rows(hs, xs.wl, list(range(n)), 1)
        single[small] = round(n / (time.time() - ts), 3)
    return {"value": round(len(rows) / dt, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the whole step: all {len(rows)} query tokens of the workload (indexer, top-k, attention), "
                      f"one token per thread, {dt:.1f} s wall",
            "single_thread_tokens_per_s": single}


def run_reference(args, rank, world, local_rank):
    if rank != 0:
        return
    import torch
    import synth
    name = args.workload or synth.HEADLINE
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x = synth.generate(name, seed=0, device=dev)
    wl = x.wl
    h = _oracle_host_inputs(x)
    cores = os.cpu_count() or 1
    per_step = max(1, min(wl.B * wl.T, cores))
    rows_all = list(range(wl.B * wl.T))
    for i in range(args.warmup):
        _oracle_rows(h, wl, [rows_all[(i * per_step + j) % len(rows_all)] for j in range(per_step)], per_step)
    t0 = time.time()
    for i in range(args.steps):
        _oracle_rows(h, wl, [rows_all[(i * per_step + j) % len(rows_all)] for j in range(per_step)], per_step)
    dt = time.time() - t0
    value = per_step * args.steps / dt
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": name, "batch": wl.B, "tokens_per_seq": wl.T, "context_tokens": wl.ctx,
                       "compressed_entries": wl.ncap, "m": wl.m, "topk": wl.k, "swa": wl.W},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": per_step, "kind": "oracle",
                             "sample": f"each step: {per_step} of the {wl.B * wl.T} query tokens of the workload"},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def report_configs():
    """Per-kernel times of every workload in synth.WORKLOADS, one JSON line
    per workload (not the benchmark's line): events around each call, five
    warm-up calls, the median of 30 timed calls over rotating input copies,
    with nvidia-smi clocks sampled during each workload's timed calls.
    Roofline = max(algorithmic bytes / measured HBM peak, flops / FP8 peak),
    FP8 dense peak taken as twice the measured BF16 one (the pages' method
    computes on FP8 data); the attention's tensor fraction is also given
    against the BF16 peak, the precision its MMAs run in."""
    import numpy as np
    import torch

    import compressed_sparse_decode_gb300 as csd
    import synth
    csd.build()
    csd.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    hbm = peaks["hbm_gbs"] * 1e9
    fp8 = 2 * peaks["bf16_tflops"] * 1e12
    bf16 = peaks["bf16_tflops"] * 1e12
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    for name, wl in synth.WORKLOADS.items():
        base = synth.generate(name, seed=0, device=dev)
        copies = [base] + [base.clone() for _ in range(N_COPIES - 1)]
        stream = torch.cuda.Stream(device=dev)
        q_pos = base.q_pos.cpu().numpy()
        n_comp = base.n_comp.cpu().numpy()
        nvis = np.minimum(np.minimum(q_pos // wl.m, n_comp[:, None]), wl.ncap)  # [B, T]
        nswa = np.minimum(q_pos + 1, wl.W)
        work = {}
        if wl.kind == "csa":
            runners = [Runner(csd, x, stream) for x in copies]
            with torch.cuda.stream(stream):
                for r in runners:
                    r.indexer(); r.topk(); r.attention()
            torch.cuda.synchronize(dev)
            ab, af = attention_work(runners[0].cnt.cpu().numpy(), base)
            work["indexer"] = (lambda i: runners[i].indexer(), indexer_bytes(base), 16384 * float(nvis.sum()))
            work["topk"] = (lambda i: runners[i].topk(), 4 * int(nvis.sum()) + 4 * wl.B * wl.T * wl.k, 0.0)
            work["attention"] = (lambda i: runners[i].attention(), ab, af)
        else:
            comps = [csd.cache_desc(x.comp, wl.ncap, x.seq_stride) for x in copies]
            outs = [(torch.empty_like(x.q), torch.empty((wl.B, wl.T, 128), dtype=torch.float32, device=dev),
                     csd.workspace(csd.OP_HCA_ATTENTION, wl.B, wl.T, wl.ncap, 0, dev)) for x in copies]

            def hca(i):
                x, (o, l, w) = copies[i], outs[i]
                csd.hca_sink_attention_decode(x.q, x.sink, SCALE, comps[i], x.n_comp, x.ring, wl.W, x.q_pos, wl.m,
                                              out=o, lse=l, ws=w, stream=stream)
            cands = int(nvis.sum() + nswa.sum())
            work["hca attention"] = (hca, cands * 592 + wl.B * wl.T * (2 * 128 * 512 * 2 + 128 * 4), 262144.0 * cands)
        kernels = {}
        clocks = ClockSampler(uuid)
        clocks.start()
        time.sleep(0.3)
        t0 = time.time()
        for kern, (fn, nbytes, flops) in work.items():
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(30)]
            with torch.cuda.stream(stream):
                for i in range(5):
                    fn(i % N_COPIES)
                for i, (a, b) in enumerate(ev):
                    a.record(stream)
                    fn(i % N_COPIES)
                    b.record(stream)
            torch.cuda.synchronize(dev)
            us = float(np.median([a.elapsed_time(b) * 1e3 for a, b in ev]))
            roof = max(nbytes / hbm, flops / fp8) * 1e6
            entry = {"us_median": round(us, 2), "algorithmic_mb": round(nbytes / 1e6, 3),
                     "gflop": round(flops / 1e9, 3), "roofline_us": round(roof, 3), "frac": round(roof / us, 4),
                     "bound": "hbm" if nbytes / hbm >= flops / fp8 else "tensor",
                     "achieved_gbs": round(nbytes / (us / 1e6) / 1e9, 1)}
            if "attention" in kern:
                entry["tensor_frac_bf16"] = round(flops / bf16 * 1e6 / us, 4)
            kernels[kern] = entry
        t1 = time.time()
        time.sleep(0.1)
        clocks.stop()
        if csd.csa_read_device_error(stream):
            raise RuntimeError(f"device error word set on {name}")
        step_us = sum(v["us_median"] for v in kernels.values())
        print(json.dumps({"workload": name, "kind": wl.kind, "batch": wl.B, "tokens_per_seq": wl.T,
                          "compressed_entries": wl.ncap, "topk": wl.k, "kernels": kernels,
                          "sum_of_kernels_us": round(step_us, 2),
                          "tokens_per_s_from_sum": round(wl.B * wl.T / (step_us / 1e6), 1),
                          "clocks": clocks.summary(t0, t1),
                          "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
                                    "fp8_tflops_taken": 2 * peaks["bf16_tflops"], "source": peaks["source"]},
                          "timing": "events around each C-ABI call (no programmatic-launch overlap), 5 warm-up "
                                    "calls, median of 30 over 3 rotating input copies"}), flush=True)
        del copies, base, work
        torch.cuda.empty_cache()


def graph_replay(args):
    """Whole-step CUDA graph ("ROADMAP -- Stage E", section E9): LAYERS decode
    steps, each layer with its own paged cache and block table, issued as
    direct C-ABI calls and as one captured graph; host clock around 50
    iterations of all layers after warm-up; the replay checked bit for bit
    against the direct calls first."""
    import torch

    import compressed_sparse_decode_gb300 as csd
    import synth
    csd.build()
    csd.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    name = args.workload or "csa_b1_ctx1k_k64"
    layers = [synth.generate(name, seed=100 + i, device=dev, paged=True) for i in range(args.graph_replay)]
    wl = layers[0].wl
    comps = [csd.cache_desc(x.comp, wl.ncap, x.seq_stride, x.block_table, x.page_records) for x in layers]
    wss = [csd.workspace(csd.OP_DECODE_STEP, wl.B, wl.T, wl.ncap, wl.k, dev) for _ in layers]
    outs = [(torch.empty_like(x.q), torch.empty((wl.B, wl.T, 128), dtype=torch.float32, device=dev)) for x in layers]
    stream = torch.cuda.Stream(device=dev)
    status = csd.status_word(dev)
    lib = csd.load()
    p = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None
    calls = [[p(x.q_idx), p(x.q_idx_scale), p(x.w_idx), p(x.k_idx), p(x.k_idx_scale), p(x.q), p(x.sink),
              C.c_float(SCALE), c, p(x.ring), x.ring.shape[1], wl.W, p(x.q_pos), p(x.n_comp), wl.B, wl.T, wl.ncap,
              wl.m, wl.k, p(o), p(l), None, None, p(w), C.c_size_t(w.numel()), p(status),
              C.c_void_p(stream.cuda_stream)] for x, c, w, (o, l) in zip(layers, comps, wss, outs)]

    def direct():
        for a in calls:
            st = lib.csa_decode_step(*a)
            if st:
                raise RuntimeError(f"csa_decode_step: {csd.status_string(st)}")

    with torch.cuda.stream(stream):
        for _ in range(5):
            direct()
    torch.cuda.synchronize(dev)
    want = [(o.clone(), l.clone()) for o, l in outs]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        direct()
    graph.replay()
    torch.cuda.synchronize(dev)
    if not all(torch.equal(o, wo) and torch.equal(l, wlse) for (o, l), (wo, wlse) in zip(outs, want)):
        raise RuntimeError("graph replay differs from the direct calls")

    def clock(fn, n=50):
        with torch.cuda.stream(stream):
            for _ in range(5):
                fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(n):
                fn()
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t0) / n * 1e6

    n0 = csd.csa_kernel_launches()
    with torch.cuda.stream(stream):
        direct()
    launches = csd.csa_kernel_launches() - n0
    t_direct = clock(direct)
    t_graph = clock(graph.replay)
    if csd.csa_read_device_error(stream):
        raise RuntimeError("device error word set")
    print(json.dumps({"graph_replay": {"workload": name, "layers": args.graph_replay,
                                       "direct_us_per_step": round(t_direct, 2),
                                       "graph_us_per_step": round(t_graph, 2),
                                       "speedup": round(t_direct / t_graph, 3),
                                       "launches_per_step": launches,
                                       "clock": "host wall clock around 50 iterations of all layers",
                                       "check": "replay bit-identical to the direct calls"}}), flush=True)


def prefill(args):
    """Many query tokens per sequence in one step ("ROADMAP -- Stage E",
    section E8: prefill spread over many CTAs): T consecutive tokens of one
    128K-context sequence (top-2048) as one csa_decode_step over B*T rows,
    against the same tokens issued as T single-token steps (one query row per
    launch). Each variant is replayed from a CUDA graph (no host call overhead
    in the device time); CUDA events on the replay stream, median of 20 after 3
    warm-ups."""
    import torch

    import compressed_sparse_decode_gb300 as csd
    import synth
    csd.build()
    csd.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    T = args.prefill
    wl = synth.custom("csa", B=1, T=T, ncap=32768, k=2048, ctx=131072, name=f"csa_b1_t{T}_ctx128k_k2048")
    x = synth.generate(wl, seed=0, device=dev)
    comp = csd.cache_desc(x.comp, wl.ncap, x.seq_stride)
    out = torch.empty_like(x.q)
    lse = torch.empty((1, T, 128), dtype=torch.float32, device=dev)
    ws = csd.workspace(csd.OP_DECODE_STEP, 1, T, wl.ncap, wl.k, dev)
    ws1 = csd.workspace(csd.OP_DECODE_STEP, 1, 1, wl.ncap, wl.k, dev)
    one = [(x.q_idx[:, t:t + 1].contiguous(), x.q_idx_scale[:, t:t + 1].contiguous(), x.w_idx[:, t:t + 1].contiguous(),
            x.q[:, t:t + 1].contiguous(), x.q_pos[:, t:t + 1].contiguous(), torch.empty_like(x.q[:, t:t + 1]),
            torch.empty((1, 1, 128), dtype=torch.float32, device=dev)) for t in range(T)]

    def batched():
        csd.csa_decode_step(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q, x.sink, SCALE, comp, x.ring,
                            wl.W, x.q_pos, x.n_comp, wl.m, wl.k, out=out, lse=lse, ws=ws)

    def token_loop():
        for qi, qs, wi, q, qp, o, l in one:
            csd.csa_decode_step(qi, qs, wi, x.k_idx, x.k_idx_scale, q, x.sink, SCALE, comp, x.ring, wl.W, qp, x.n_comp,
                                wl.m, wl.k, out=o, lse=l, ws=ws1)

    # each variant captured once into a CUDA graph, so that the host's call
    # overhead (a Python call per step) does not enter the device time
    stream = torch.cuda.Stream(device=dev)

    def graphed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    def timed(g, n=20):
        ts = []
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            for _ in range(n):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b) * 1e3)
        return float(statistics.median(ts))

    t_b, t_l = timed(graphed(batched)), timed(graphed(token_loop))
    if csd.csa_read_device_error():
        raise RuntimeError("device error word set")
    # the batched step's rows agree with the single-token steps' rows
    cos = min(float(torch.nn.functional.cosine_similarity(out[0, t].float(), one[t][5][0, 0].float(), dim=-1).min())
              for t in range(T))
    print(json.dumps({"prefill": {"workload": wl.name, "tokens": T, "batched_us": round(t_b, 2),
                                  "token_loop_us": round(t_l, 2), "speedup": round(t_l / t_b, 2),
                                  "batched_tokens_per_s": round(T / t_b * 1e6, 1),
                                  "min_cos_batched_vs_loop": round(cos, 6),
                                  "clock": "CUDA events, median of 20 after 3 warm-ups"}}), flush=True)


def epilogue_timing(args):
    """The attention's output epilogue ("DSV4 Audit" section A4, "ROADMAP --
    Stage E" section E6) on the 128K and HCA workloads: the attention call
    with BF16 output, with the inverse RoPE, with E2M1 output, and with both.
    Device time with CUDA events around 10 back-to-back calls, median of 20
    after 3 warm-ups, inputs resident (the same call repeated); output bytes
    per call alongside."""
    import torch

    import compressed_sparse_decode_gb300 as csd
    import synth
    csd.build()
    csd.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    res = {}
    for name in ("csa_b32_ctx128k_k2048", "hca_b64_ctx1m"):
        x = synth.generate(name, seed=0, device=dev)
        wl = x.wl
        comp = csd.cache_desc(x.comp, wl.ncap, x.seq_stride)
        rows = wl.B * wl.T
        if wl.kind == "csa":
            lg = csd.csa_indexer_logits(x.q_idx, x.q_idx_scale, x.w_idx, x.k_idx, x.k_idx_scale, x.q_pos, x.n_comp,
                                        wl.m)
            idx, cnt = csd.csa_topk(lg, x.q_pos, x.n_comp, wl.m, wl.k)
            ws = csd.workspace(csd.OP_ATTENTION, wl.B, wl.T, wl.ncap, wl.k, dev)
            call = lambda **e: csd.csa_sink_attention_decode(x.q, x.sink, SCALE, comp, x.ring, wl.W, idx, cnt,
                                                             x.q_pos, ws=ws, **e)
        else:
            ws = csd.workspace(csd.OP_HCA_ATTENTION, wl.B, wl.T, wl.ncap, 0, dev)
            call = lambda **e: csd.hca_sink_attention_decode(x.q, x.sink, SCALE, comp, x.n_comp, x.ring, wl.W,
                                                             x.q_pos, wl.m, ws=ws, **e)
        out = torch.empty_like(x.q)
        f4 = torch.empty((wl.B, wl.T, 128, 256), dtype=torch.uint8, device=dev)
        f4s = torch.empty((wl.B, wl.T, 128, 4), dtype=torch.float32, device=dev)
        variants = {"bf16": dict(out=out), "bf16+inverse_rope": dict(out=out, inverse_rope=True),
                    "e2m1": dict(fp4_out=True, out_fp4=f4, out_fp4_scale=f4s),
                    "e2m1+inverse_rope": dict(fp4_out=True, out_fp4=f4, out_fp4_scale=f4s, inverse_rope=True)}
        row = {}
        for v, kw in variants.items():
            for _ in range(3):
                call(**kw)
            ts = []
            for _ in range(20):
                # 10 calls back to back per event pair: the device stays busy
                # while the host issues the next call
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize(dev)
                a.record()
                for _ in range(10):
                    call(**kw)
                b.record()
                torch.cuda.synchronize(dev)
                ts.append(a.elapsed_time(b) * 1e3 / 10)
            out_bytes = rows * 128 * (512 * 2 if v.startswith("bf16") else 256 + 16)
            row[v] = {"us": round(statistics.median(ts), 2), "output_bytes": out_bytes}
        if csd.csa_read_device_error():
            raise RuntimeError("device error word set")
        res[name] = row
    print(json.dumps({"epilogue": res, "clock": "CUDA events around 10 back-to-back calls, median of 20"}),
          flush=True)


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.epilogue:
        if rank == 0:
            epilogue_timing(args)
        return
    if args.prefill:
        if rank == 0:
            prefill(args)
        return
    if args.graph_replay:
        if rank == 0:
            graph_replay(args)
        return
    if args.report_configs:
        if rank == 0:
            report_configs()
        return
    if args.impl == "reference":
        run_reference(args, rank, world, local_rank)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
