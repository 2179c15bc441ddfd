"""CPU oracle for CSA / HCA decode -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package. The product path (the CUDA library and
its binding) never does, and this package never imports it: the two share no
code. The arithmetic lives in ``csa_oracle.c`` (plain C, double precision,
every step the definition from the project's pages written out as loops); this
module only compiles it, marshals numpy arrays through ctypes and splits query
rows across host threads (the C code releases the GIL through ctypes).

Function-level citations are in ``csa_oracle.c``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libcsa_oracle.so")
_lock = threading.Lock()
_lib = None

# Production shapes (the pages' DSV4 configuration).
H, DN, DR, SB, HI, DI = 128, 448, 64, 128, 64, 128

OK, BAD_INDEX, BAD_ARG, NO_MEMORY = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, so x86 and Arm agree)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # CSA_ORACLE_LIB points the test suite at a deliberately mutated
            # build of the oracle (tests/test_oracle_mutants.py).
            path = os.environ.get("CSA_ORACLE_LIB")
            if not path:
                build()
                path = _LIB_PATH
            lib = C.CDLL(path)
            P = C.c_void_p
            i32, i64, dbl = C.c_int, C.c_int64, C.c_double
            lib.oracle_e4m3_value.argtypes = [C.c_uint8]
            lib.oracle_e4m3_value.restype = dbl
            lib.oracle_bf16_value.argtypes = [C.c_uint16]
            lib.oracle_bf16_value.restype = dbl
            lib.oracle_n_visible.argtypes = [i32, i32, i32, i32]
            lib.oracle_n_visible.restype = i32
            lib.oracle_indexer_logits.argtypes = [P, P, P, P, P, P, P] + [i32] * 8 + [P]
            lib.oracle_indexer_logits.restype = i32
            lib.oracle_topk.argtypes = [P, P, P] + [i32] * 7 + [P, P]
            lib.oracle_topk.restype = i32
            cache = [P, i64, P, i32, i32, i64, i32]
            lib.oracle_attention_row.argtypes = [P, P, dbl, P, i32, i32, i32, i32, i32, P, P]
            lib.oracle_attention_row.restype = i32
            lib.oracle_csa_attention.argtypes = ([P, P, dbl] + cache + [P, i32, i32, P, P, P]
                                                 + [i32] * 10 + [P, P])
            lib.oracle_csa_attention.restype = i32
            lib.oracle_hca_attention.argtypes = ([P, P, dbl] + cache + [P, P, i32, i32, P]
                                                 + [i32] * 10 + [P, P])
            lib.oracle_hca_attention.restype = i32
            lib.oracle_gather.argtypes = cache + [P, i32, i32, P, P, P] + [i32] * 6 + [P, P]
            lib.oracle_gather.restype = i32
            lib.oracle_e2m1_value.argtypes = [C.c_uint8]
            lib.oracle_e2m1_value.restype = dbl
            lib.oracle_e2m1_code.argtypes = [dbl]
            lib.oracle_e2m1_code.restype = C.c_uint8
            lib.oracle_e2m1_quantize.argtypes = [P, i32, i32, P, P]
            lib.oracle_e2m1_quantize.restype = None
            lib.oracle_inverse_rope.argtypes = [P, i32, i32, i32, dbl]
            lib.oracle_inverse_rope.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _np(a, dtype) -> np.ndarray:
    """Accept numpy arrays or CPU torch tensors; return a contiguous numpy view."""
    if hasattr(a, "detach"):
        a = a.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "uiV" and np.dtype(dtype).kind in "uiV":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _check(rc: int, what: str):
    if rc != OK:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _rows(n_rows: int, threads: int | None, fn):
    """Run fn(row_begin, row_end) over [0, n_rows) split into contiguous ranges."""
    threads = max(1, min(threads or 1, n_rows))
    if threads == 1:
        fn(0, n_rows)
        return
    bounds = np.linspace(0, n_rows, threads + 1).astype(int)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        futs = [ex.submit(fn, int(bounds[i]), int(bounds[i + 1])) for i in range(threads)
                if bounds[i + 1] > bounds[i]]
        for f in futs:
            f.result()


# --------------------------------------------------------------------------
# Scalars
# --------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(code)


def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(bits)


def n_visible(p: int, m: int, n_comp: int, capacity: int) -> int:
    return _load().oracle_n_visible(p, m, n_comp, capacity)


# --------------------------------------------------------------------------
# Cache descriptor (same meaning as the library's, defined independently)
# --------------------------------------------------------------------------

class Cache:
    """A compressed cache of fixed-size records.

    ``records`` is a uint8 array [n_records, rec_bytes]. Without a block table,
    entry c of sequence b is record b*seq_stride + c; with one, it is record
    block_table[b, c // page_records] * page_records + c % page_records.
    """

    def __init__(self, records, seq_stride: int, seq_capacity: int,
                 block_table=None, page_records: int = 1):
        self.records = _np(records, np.uint8)
        self.records = self.records.reshape(-1, self.records.shape[-1])
        self.rec_bytes = int(self.records.shape[1])
        self.n_records = int(self.records.shape[0])
        self.seq_stride = int(seq_stride)
        self.seq_capacity = int(seq_capacity)
        self.block_table = None if block_table is None else _np(block_table, np.int32)
        self.page_records = int(page_records)
        self.max_pages = 0 if self.block_table is None else int(self.block_table.shape[-1])

    def args(self):
        return [_ptr(self.records), self.seq_stride, _ptr(self.block_table), self.page_records,
                self.max_pages, self.n_records, self.seq_capacity]


# --------------------------------------------------------------------------
# Steps
# --------------------------------------------------------------------------

def indexer_logits(q8, q_scale, w, k8, k_scale, q_pos, n_comp, m: int, threads: int = 1,
                   rows=None) -> np.ndarray:
    """a2. q8 [B,T,Hi,Di] uint8 e4m3, q_scale/w [B,T,Hi] f32, k8 [B,Ncap,Di] uint8,
    k_scale [B,Ncap] f32, q_pos [B,T] i32, n_comp [B] i32 -> [B,T,Ncap] float64.
    ``rows`` optionally restricts the computed flat rows (others stay NaN)."""
    lib = _load()
    q8 = _np(q8, np.uint8); k8 = _np(k8, np.uint8)
    q_scale = _np(q_scale, np.float32); w = _np(w, np.float32); k_scale = _np(k_scale, np.float32)
    q_pos = _np(q_pos, np.int32); n_comp = _np(n_comp, np.int32)
    B, T, Hi, Di = q8.shape
    Ncap = k8.shape[1]
    out = np.full((B, T, Ncap), np.nan, dtype=np.float64)

    def run(r0, r1):
        _check(lib.oracle_indexer_logits(_ptr(q8), _ptr(q_scale), _ptr(w), _ptr(k8), _ptr(k_scale),
                                         _ptr(q_pos), _ptr(n_comp), B, T, Ncap, Hi, Di, m,
                                         r0, r1, _ptr(out)), "indexer_logits")
    if rows is None:
        _rows(B * T, threads, run)
    else:
        for r in rows:
            run(int(r), int(r) + 1)
    return out


def topk(scores, q_pos, n_comp, m: int, k: int, threads: int = 1):
    """a3. scores [B,T,Ncap] (any float dtype, widened exactly to double)
    -> (idx [B,T,k] int32 in sorted order, -1 padded; cnt [B,T] int32)."""
    lib = _load()
    scores = _np(scores, np.float64)
    q_pos = _np(q_pos, np.int32); n_comp = _np(n_comp, np.int32)
    B, T, Ncap = scores.shape
    idx = np.empty((B, T, k), dtype=np.int32)
    cnt = np.empty((B, T), dtype=np.int32)

    def run(r0, r1):
        _check(lib.oracle_topk(_ptr(scores), _ptr(q_pos), _ptr(n_comp), B, T, Ncap, m, k, r0, r1,
                               _ptr(idx), _ptr(cnt)), "topk")
    _rows(B * T, threads, run)
    return idx, cnt


def attention_row(q, sink, scale: float, records, Dn=DN, Dr=DR, sb=SB):
    """a5 on one explicit candidate list: q [H,D] bf16 bits (uint16), records
    [n, rec_bytes] uint8 -> (out [H,D] float64, lse [H] float64)."""
    lib = _load()
    q = _np(q, np.uint16); sink = _np(sink, np.float32)
    records = _np(records, np.uint8)
    Hh, D = q.shape
    n = records.shape[0] if records.ndim == 2 else 0
    ptrs = (C.c_void_p * max(n, 1))(*[records.ctypes.data + i * records.shape[1] for i in range(n)])
    out = np.empty((Hh, D), dtype=np.float64)
    lse = np.empty((Hh,), dtype=np.float64)
    _check(lib.oracle_attention_row(_ptr(q), _ptr(sink), float(scale), C.cast(ptrs, C.c_void_p), n,
                                    Hh, Dn, Dr, sb, _ptr(out), _ptr(lse)), "attention_row")
    return out, lse


def csa_attention(q, sink, scale: float, cache: Cache, ring, W: int, topk_idx, topk_cnt, q_pos,
                  Dn=DN, Dr=DR, sb=SB, threads: int = 1, rows=None):
    """a5. q [B,T,H,D] bf16 bits, ring [B,R,rec] uint8, topk_idx [B,T,k] i32,
    topk_cnt [B,T] i32 -> (out [B,T,H,D] f64, lse [B,T,H] f64)."""
    lib = _load()
    q = _np(q, np.uint16); sink = _np(sink, np.float32)
    ring = _np(ring, np.uint8)
    topk_idx = _np(topk_idx, np.int32); topk_cnt = _np(topk_cnt, np.int32)
    q_pos = _np(q_pos, np.int32)
    B, T, Hh, D = q.shape
    R = ring.shape[1]
    k = topk_idx.shape[2]
    out = np.full((B, T, Hh, D), np.nan, dtype=np.float64)
    lse = np.full((B, T, Hh), np.nan, dtype=np.float64)

    def run(r0, r1):
        _check(lib.oracle_csa_attention(_ptr(q), _ptr(sink), float(scale), *cache.args(), _ptr(ring),
                                        R, W, _ptr(topk_idx), _ptr(topk_cnt), _ptr(q_pos),
                                        B, T, k, Hh, Dn, Dr, sb, cache.rec_bytes, r0, r1,
                                        _ptr(out), _ptr(lse)), "csa_attention")
    if rows is None:
        _rows(B * T, threads, run)
    else:
        for r in rows:
            run(int(r), int(r) + 1)
    return out, lse


def hca_attention(q, sink, scale: float, cache: Cache, n_comp, ring, W: int, q_pos, m_hca: int,
                  Dn=DN, Dr=DR, sb=SB, threads: int = 1, rows=None):
    """a6. Same shapes as csa_attention; candidates are every visible entry."""
    lib = _load()
    q = _np(q, np.uint16); sink = _np(sink, np.float32)
    ring = _np(ring, np.uint8)
    n_comp = _np(n_comp, np.int32); q_pos = _np(q_pos, np.int32)
    B, T, Hh, D = q.shape
    R = ring.shape[1]
    out = np.full((B, T, Hh, D), np.nan, dtype=np.float64)
    lse = np.full((B, T, Hh), np.nan, dtype=np.float64)

    def run(r0, r1):
        _check(lib.oracle_hca_attention(_ptr(q), _ptr(sink), float(scale), *cache.args(),
                                        _ptr(n_comp), _ptr(ring), R, W, _ptr(q_pos), B, T, m_hca,
                                        Hh, Dn, Dr, sb, cache.rec_bytes, r0, r1,
                                        _ptr(out), _ptr(lse)), "hca_attention")
    if rows is None:
        _rows(B * T, threads, run)
    else:
        for r in rows:
            run(int(r), int(r) + 1)
    return out, lse


def gather(cache: Cache, ring, W: int, topk_idx, topk_cnt, q_pos, threads: int = 1):
    """a4. -> (kv_out [B,T,k+W,rec] uint8 (unwritten slots zero), kv_cnt [B,T] i32)."""
    lib = _load()
    ring = _np(ring, np.uint8)
    topk_idx = _np(topk_idx, np.int32); topk_cnt = _np(topk_cnt, np.int32)
    q_pos = _np(q_pos, np.int32)
    B, T, k = topk_idx.shape
    R = ring.shape[1]
    kv_out = np.zeros((B, T, k + W, cache.rec_bytes), dtype=np.uint8)
    kv_cnt = np.zeros((B, T), dtype=np.int32)

    def run(r0, r1):
        _check(lib.oracle_gather(*cache.args(), _ptr(ring), R, W, _ptr(topk_idx), _ptr(topk_cnt),
                                 _ptr(q_pos), B, T, k, cache.rec_bytes, r0, r1,
                                 _ptr(kv_out), _ptr(kv_cnt)), "gather")
    _rows(B * T, threads, run)
    return kv_out, kv_cnt


# --------------------------------------------------------------------------
# Attention output epilogue (inverse RoPE, E2M1 output)
# --------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(code)


def e2m1_code(v: float) -> int:
    return int(_load().oracle_e2m1_code(float(v)))


def e2m1_quantize(x, block: int = 128):
    """x [..., n] (any float dtype, widened exactly to double) -> (codes
    [..., n] uint8, one code per byte; scales [..., ceil(n/block)] float64)."""
    lib = _load()
    x = _np(x, np.float64)
    n = x.shape[-1]
    flat = x.reshape(-1, n)
    nb = (n + block - 1) // block
    codes = np.empty(flat.shape, dtype=np.uint8)
    scales = np.empty((flat.shape[0], nb), dtype=np.float64)
    for i in range(flat.shape[0]):
        lib.oracle_e2m1_quantize(_ptr(flat[i]), n, block, _ptr(codes[i]), _ptr(scales[i]))
    return codes.reshape(x.shape), scales.reshape(*x.shape[:-1], nb)


def inverse_rope(o, pos, theta: float, Dn=DN, Dr=DR):
    """o [rows, ..., Dn+Dr] float64 (a copy is rotated), pos [rows] -> the rows
    with their rope dims turned back by RoPE(-pos)."""
    lib = _load()
    out = np.array(_np(o, np.float64), copy=True)
    pos = np.asarray(pos).reshape(-1)
    D = out.shape[-1]
    view = out.reshape(len(pos), -1, D)
    for r in range(len(pos)):
        for j in range(view.shape[1]):
            row = np.ascontiguousarray(view[r, j])
            lib.oracle_inverse_rope(_ptr(row), Dn, Dr, int(pos[r]), float(theta))
            view[r, j] = row
    return out
