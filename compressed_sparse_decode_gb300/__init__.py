"""Python binding of libcsa, the GB300 (sm_103a) CSA decode library.

Argument marshalling only: every function below checks tensor devices,
dtypes and shapes, passes raw device pointers and the current CUDA stream to
the extern "C" entry point of the same name (include/csa.h), and raises
``CsaError`` on a non-zero status. All compute runs in the library's CUDA
kernels. There is no fallback: if libcsa.so is missing or cannot be loaded,
``load()`` raises.

PyTorch supplies device memory and streams only.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

from ._build import LIB, build  # noqa: F401  (build() compiles libcsa.so in-tree)

HEADS, DIM, NOPE, ROPE, SCALE_BLOCK, RECORD_BYTES = 128, 512, 448, 64, 128, 592
IDX_HEADS, IDX_DIM = 64, 128
MAX_TOKENS_PER_SEQ, MAX_TOPK, MAX_SWA_WINDOW = 128, 2048, 512

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_BAD_INDEX = range(7)
OP_INDEXER, OP_TOPK, OP_ATTENTION, OP_HCA_ATTENTION, OP_DECODE_STEP = range(5)

EXPORTED = ["csa_workspace_bytes", "csa_indexer_logits", "csa_topk", "csa_gather_swa",
            "csa_sink_attention_decode", "hca_sink_attention_decode", "csa_decode_step",
            "csa_check_device_status", "csa_read_device_error", "csa_debug_set_wait_limit_ns",
            "csa_status_string", "csa_version", "csa_kernel_launches",
            "csa_sink_attention_decode_noalloc", "csa_pipeline_staging_bytes", "csa_pipeline_create",
            "csa_decode_step_host", "csa_pipeline_wait", "csa_pipeline_sync", "csa_pipeline_destroy",
            "csa_sink_attention_decode_ex", "hca_sink_attention_decode_ex", "csa_decode_step_ex"]
PIPELINE_MAX_DEPTH = 4


class CsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({status_string(status)})")
        self.status = status


class csa_cache_desc(C.Structure):
    _fields_ = [("base", C.c_void_p), ("n_records", C.c_int64), ("seq_stride", C.c_int64),
                ("block_table", C.c_void_p), ("page_records", C.c_int32), ("max_pages", C.c_int32),
                ("seq_capacity", C.c_int32)]


class csa_attention_epilogue(C.Structure):
    _fields_ = [("inverse_rope", C.c_int32), ("rope_theta", C.c_float), ("out_fp4", C.c_void_p),
                ("out_fp4_scale", C.c_void_p)]


_lib = None
_lock = threading.Lock()


def load(path: str | None = None):
    """Load libcsa.so (built in-tree by ``build()``); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libcsa.so not found at {path}: run compressed_sparse_decode_gb300.build()")
        lib = C.CDLL(path)
        P, i32, sz, f32 = C.c_void_p, C.c_int, C.c_size_t, C.c_float
        st = C.c_int
        lib.csa_version.restype = C.c_int
        lib.csa_kernel_launches.restype = C.c_uint64
        lib.csa_status_string.argtypes = [C.c_int]
        lib.csa_status_string.restype = C.c_char_p
        lib.csa_workspace_bytes.argtypes = [C.c_int, i32, i32, i32, i32]
        lib.csa_workspace_bytes.restype = sz
        lib.csa_indexer_logits.argtypes = [P] * 7 + [i32] * 4 + [P, P, P]
        lib.csa_indexer_logits.restype = st
        lib.csa_topk.argtypes = [P, P, P] + [i32] * 5 + [P, P, P, sz, P, P]
        lib.csa_topk.restype = st
        lib.csa_gather_swa.argtypes = [csa_cache_desc, P, i32, i32, P, P, P, i32, i32, i32, P, P, P, P]
        lib.csa_gather_swa.restype = st
        lib.csa_sink_attention_decode.argtypes = ([P, P, f32, csa_cache_desc, P, i32, i32, P, P, P, i32, i32, i32,
                                                   P, P, P, sz, P, P])
        lib.csa_sink_attention_decode.restype = st
        lib.hca_sink_attention_decode.argtypes = ([P, P, f32, csa_cache_desc, P, P, i32, i32, P, i32, i32, i32,
                                                   P, P, P, sz, P, P])
        lib.hca_sink_attention_decode.restype = st
        lib.csa_decode_step.argtypes = ([P] * 7 + [f32, csa_cache_desc, P, i32, i32, P, P] + [i32] * 5
                                        + [P, P, P, P, P, sz, P, P])
        lib.csa_decode_step.restype = st
        lib.csa_sink_attention_decode_noalloc.argtypes = ([P, P, f32, csa_cache_desc, P, i32, i32, P, P, P, i32, i32,
                                                           i32, P, P, P, P])
        lib.csa_sink_attention_decode_noalloc.restype = st
        EP = C.POINTER(csa_attention_epilogue)
        lib.csa_sink_attention_decode_ex.argtypes = ([P, P, f32, csa_cache_desc, P, i32, i32, P, P, P, i32, i32, i32,
                                                      P, P, EP, P, sz, P, P])
        lib.csa_sink_attention_decode_ex.restype = st
        lib.hca_sink_attention_decode_ex.argtypes = ([P, P, f32, csa_cache_desc, P, P, i32, i32, P, i32, i32, i32,
                                                      P, P, EP, P, sz, P, P])
        lib.hca_sink_attention_decode_ex.restype = st
        lib.csa_decode_step_ex.argtypes = ([P] * 7 + [f32, csa_cache_desc, P, i32, i32, P, P] + [i32] * 5
                                           + [P, P, P, P, EP, P, sz, P, P])
        lib.csa_decode_step_ex.restype = st
        lib.csa_pipeline_staging_bytes.argtypes = [i32, i32, i32]
        lib.csa_pipeline_staging_bytes.restype = sz
        lib.csa_pipeline_create.argtypes = [C.POINTER(C.c_void_p), i32, i32, i32, P, sz, P]
        lib.csa_pipeline_create.restype = st
        lib.csa_decode_step_host.argtypes = ([P] * 9 + [f32, csa_cache_desc, P, i32, i32, P] + [i32] * 3
                                             + [P, P, P, sz, P, C.POINTER(C.c_int64)])
        lib.csa_decode_step_host.restype = st
        lib.csa_pipeline_wait.argtypes = [P, C.c_int64]
        lib.csa_pipeline_wait.restype = st
        lib.csa_pipeline_sync.argtypes = [P]
        lib.csa_pipeline_sync.restype = st
        lib.csa_pipeline_destroy.argtypes = [P]
        lib.csa_pipeline_destroy.restype = st
        lib.csa_check_device_status.argtypes = [P, P, P]
        lib.csa_check_device_status.restype = st
        lib.csa_read_device_error.argtypes = [P, C.POINTER(C.c_int32), P]
        lib.csa_read_device_error.restype = st
        lib.csa_debug_set_wait_limit_ns.argtypes = [C.c_uint64]
        lib.csa_debug_set_wait_limit_ns.restype = None
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().csa_status_string(int(status)).decode()


def csa_version() -> int:
    return int(load().csa_version())


def csa_kernel_launches() -> int:
    """Kernels launched so far by this process through the library."""
    return int(load().csa_kernel_launches())


def _check(status: int, where: str):
    if status != OK:
        raise CsaError(status, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor | None, name: str, dtype=None, shape=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


_status_words: dict[int, torch.Tensor] = {}


def status_word(device=None) -> torch.Tensor:
    """The binding's default status word for a device: one int32 in device
    memory (created zeroed on first use), passed to the library by every call
    below that is not given its own ``status`` tensor."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    with _lock:
        w = _status_words.get(dev.index)
        if w is None:
            w = torch.zeros(1, dtype=torch.int32, device=dev)
            _status_words[dev.index] = w
    return w


def _status(status, device) -> int:
    if status is None:
        status = status_word(device)
    return _ptr(status, "status", torch.int32, (1,))


def cache_desc(records: torch.Tensor, seq_capacity: int, seq_stride: int = 0,
               block_table: torch.Tensor | None = None, page_records: int = 0) -> csa_cache_desc:
    """Describe a cache of latent records: ``records`` is uint8 [n, 592] (or
    [B, Ncap, 592]); contiguous mode uses ``seq_stride``, paged mode a
    ``block_table`` [B, max_pages] int32 and ``page_records``."""
    rec = records.reshape(-1, RECORD_BYTES) if records.dim() != 2 else records
    _ptr(rec, "records", torch.uint8)
    if rec.shape[1] != RECORD_BYTES:
        raise ValueError("records must be [n, 592] uint8")
    d = csa_cache_desc()
    d.base = rec.data_ptr()
    d.n_records = rec.shape[0]
    d.seq_stride = int(seq_stride)
    d.seq_capacity = int(seq_capacity)
    if block_table is not None:
        _ptr(block_table, "block_table", torch.int32)
        d.block_table = block_table.data_ptr()
        d.page_records = int(page_records)
        d.max_pages = int(block_table.shape[-1])
    d._keepalive = (rec, block_table)  # noqa: SLF001
    return d


def csa_workspace_bytes(op: int, B: int, T: int, Ncap: int, k: int) -> int:
    return int(load().csa_workspace_bytes(int(op), B, T, Ncap, k))


def workspace(op: int, B: int, T: int, Ncap: int, k: int, device=None) -> torch.Tensor | None:
    """Allocate (through PyTorch) a workspace of the size the library asks for."""
    n = csa_workspace_bytes(op, B, T, Ncap, k)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def csa_indexer_logits(q_idx, q_idx_scale, w_idx, k_idx, k_idx_scale, q_pos, n_comp, m: int,
                       logits: torch.Tensor | None = None, stream=None, status=None) -> torch.Tensor:
    B, T = q_pos.shape
    Ncap = k_idx.shape[1]
    if logits is None:
        logits = torch.empty((B, T, Ncap), dtype=torch.float32, device=q_idx.device)
    u8 = (torch.uint8, torch.float8_e4m3fn)
    args = [_ptr(q_idx, "q_idx", u8, (B, T, IDX_HEADS, IDX_DIM)),
            _ptr(q_idx_scale, "q_idx_scale", torch.float32, (B, T, IDX_HEADS)),
            _ptr(w_idx, "w_idx", torch.float32, (B, T, IDX_HEADS)),
            _ptr(k_idx, "k_idx", u8, (B, Ncap, IDX_DIM)),
            _ptr(k_idx_scale, "k_idx_scale", torch.float32, (B, Ncap)),
            _ptr(q_pos, "q_pos", torch.int32, (B, T)), _ptr(n_comp, "n_comp", torch.int32, (B,))]
    _check(load().csa_indexer_logits(*args, B, T, Ncap, int(m),
                                     _ptr(logits, "logits", torch.float32, (B, T, Ncap)),
                                     _status(status, q_idx.device), _stream(stream)),
           "csa_indexer_logits")
    return logits


def csa_topk(logits, q_pos, n_comp, m: int, k: int, topk_idx=None, topk_cnt=None, ws=None, stream=None,
             status=None):
    B, T, Ncap = logits.shape
    dev = logits.device
    if topk_idx is None:
        topk_idx = torch.empty((B, T, k), dtype=torch.int32, device=dev)
    if topk_cnt is None:
        topk_cnt = torch.empty((B, T), dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(OP_TOPK, B, T, Ncap, k, dev)
    _check(load().csa_topk(_ptr(logits, "logits", torch.float32), _ptr(q_pos, "q_pos", torch.int32, (B, T)),
                           _ptr(n_comp, "n_comp", torch.int32, (B,)), B, T, Ncap, int(m), int(k),
                           _ptr(topk_idx, "topk_idx", torch.int32, (B, T, k)),
                           _ptr(topk_cnt, "topk_cnt", torch.int32, (B, T)),
                           _ptr(ws, "workspace", torch.uint8), 0 if ws is None else ws.numel(),
                           _status(status, dev), _stream(stream)),
           "csa_topk")
    return topk_idx, topk_cnt


def csa_gather_swa(comp: csa_cache_desc, swa_ring, W: int, topk_idx, topk_cnt, q_pos, kv_out=None, kv_cnt=None,
                   stream=None, status=None):
    B, T, k = topk_idx.shape
    R = swa_ring.shape[1]
    dev = swa_ring.device
    if kv_out is None:
        kv_out = torch.empty((B, T, k + W, RECORD_BYTES), dtype=torch.uint8, device=dev)
    if kv_cnt is None:
        kv_cnt = torch.empty((B, T), dtype=torch.int32, device=dev)
    _check(load().csa_gather_swa(comp, _ptr(swa_ring, "swa_ring", torch.uint8, (B, R, RECORD_BYTES)), R, int(W),
                                 _ptr(topk_idx, "topk_idx", torch.int32), _ptr(topk_cnt, "topk_cnt", torch.int32, (B, T)),
                                 _ptr(q_pos, "q_pos", torch.int32, (B, T)), B, T, k,
                                 _ptr(kv_out, "kv_out", torch.uint8, (B, T, k + W, RECORD_BYTES)),
                                 _ptr(kv_cnt, "kv_cnt", torch.int32, (B, T)), _status(status, dev), _stream(stream)),
           "csa_gather_swa")
    return kv_out, kv_cnt


def _epilogue(B: int, T: int, dev, inverse_rope: bool, rope_theta: float, fp4_out: bool, out_fp4, out_fp4_scale):
    """The output-epilogue struct (None when neither step is asked for) and
    the E2M1 output tensors."""
    if not inverse_rope and not fp4_out:
        return None, None, None
    if fp4_out:
        if out_fp4 is None:
            out_fp4 = torch.empty((B, T, HEADS, DIM // 2), dtype=torch.uint8, device=dev)
        if out_fp4_scale is None:
            out_fp4_scale = torch.empty((B, T, HEADS, DIM // SCALE_BLOCK), dtype=torch.float32, device=dev)
    epi = csa_attention_epilogue(1 if inverse_rope else 0, float(rope_theta),
                                 _ptr(out_fp4, "out_fp4", torch.uint8, (B, T, HEADS, DIM // 2)) if fp4_out else None,
                                 _ptr(out_fp4_scale, "out_fp4_scale", torch.float32,
                                      (B, T, HEADS, DIM // SCALE_BLOCK)) if fp4_out else None)
    return epi, out_fp4, out_fp4_scale


def csa_sink_attention_decode(q, sink, softmax_scale: float, comp: csa_cache_desc, swa_ring, W: int, topk_idx,
                              topk_cnt, q_pos, out=None, lse=None, ws=None, stream=None, status=None,
                              inverse_rope: bool = False, rope_theta: float = 10000.0, fp4_out: bool = False,
                              out_fp4=None, out_fp4_scale=None):
    """Returns (out, lse); with fp4_out, ((out_fp4, out_fp4_scale), lse).
    inverse_rope / fp4_out select the output epilogue (csa_attention_epilogue)."""
    B, T = q_pos.shape
    k = topk_idx.shape[2]
    R = swa_ring.shape[1]
    dev = q.device
    epi, out_fp4, out_fp4_scale = _epilogue(B, T, dev, inverse_rope, rope_theta, fp4_out, out_fp4, out_fp4_scale)
    if out is None and not fp4_out:
        out = torch.empty((B, T, HEADS, DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, T, HEADS), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(OP_ATTENTION, B, T, comp.seq_capacity, k, dev)
    args = [_ptr(q, "q", torch.bfloat16, (B, T, HEADS, DIM)), _ptr(sink, "sink", torch.float32, (HEADS,)),
            float(softmax_scale), comp, _ptr(swa_ring, "swa_ring", torch.uint8, (B, R, RECORD_BYTES)), R, int(W),
            _ptr(topk_idx, "topk_idx", torch.int32, (B, T, k)), _ptr(topk_cnt, "topk_cnt", torch.int32, (B, T)),
            _ptr(q_pos, "q_pos", torch.int32, (B, T)), B, T, k,
            _ptr(out, "out", torch.bfloat16, (B, T, HEADS, DIM)), _ptr(lse, "lse", torch.float32, (B, T, HEADS))]
    tail = [_ptr(ws, "workspace", torch.uint8), 0 if ws is None else ws.numel(), _status(status, dev), _stream(stream)]
    if epi is None:
        _check(load().csa_sink_attention_decode(*args, *tail), "csa_sink_attention_decode")
    else:
        _check(load().csa_sink_attention_decode_ex(*args, C.byref(epi), *tail), "csa_sink_attention_decode_ex")
    return ((out_fp4, out_fp4_scale) if fp4_out else out), lse


def csa_sink_attention_decode_noalloc(q, sink, softmax_scale: float, comp: csa_cache_desc, swa_ring, W: int, topk_idx,
                                      topk_cnt, q_pos, out=None, lse=None, stream=None, status=None):
    """csa_sink_attention_decode without a workspace: for callers that cannot
    allocate device memory on the decode path (see include/csa.h); the split
    partials use the library's static device scratch."""
    B, T = q_pos.shape
    k = topk_idx.shape[2]
    R = swa_ring.shape[1]
    dev = q.device
    if out is None:
        out = torch.empty((B, T, HEADS, DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, T, HEADS), dtype=torch.float32, device=dev)
    _check(load().csa_sink_attention_decode_noalloc(
        _ptr(q, "q", torch.bfloat16, (B, T, HEADS, DIM)), _ptr(sink, "sink", torch.float32, (HEADS,)),
        float(softmax_scale), comp, _ptr(swa_ring, "swa_ring", torch.uint8, (B, R, RECORD_BYTES)), R, int(W),
        _ptr(topk_idx, "topk_idx", torch.int32, (B, T, k)), _ptr(topk_cnt, "topk_cnt", torch.int32, (B, T)),
        _ptr(q_pos, "q_pos", torch.int32, (B, T)), B, T, k,
        _ptr(out, "out", torch.bfloat16, (B, T, HEADS, DIM)), _ptr(lse, "lse", torch.float32, (B, T, HEADS)),
        _status(status, dev), _stream(stream)), "csa_sink_attention_decode_noalloc")
    return out, lse


def hca_sink_attention_decode(q, sink, softmax_scale: float, comp: csa_cache_desc, n_comp, swa_ring, W: int, q_pos,
                              m_hca: int = 128, out=None, lse=None, ws=None, stream=None, status=None,
                              inverse_rope: bool = False, rope_theta: float = 10000.0, fp4_out: bool = False,
                              out_fp4=None, out_fp4_scale=None):
    """Returns (out, lse); with fp4_out, ((out_fp4, out_fp4_scale), lse)."""
    B, T = q_pos.shape
    R = swa_ring.shape[1]
    dev = q.device
    epi, out_fp4, out_fp4_scale = _epilogue(B, T, dev, inverse_rope, rope_theta, fp4_out, out_fp4, out_fp4_scale)
    if out is None and not fp4_out:
        out = torch.empty((B, T, HEADS, DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, T, HEADS), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(OP_HCA_ATTENTION, B, T, comp.seq_capacity, 0, dev)
    args = [_ptr(q, "q", torch.bfloat16, (B, T, HEADS, DIM)), _ptr(sink, "sink", torch.float32, (HEADS,)),
            float(softmax_scale), comp, _ptr(n_comp, "n_comp", torch.int32, (B,)),
            _ptr(swa_ring, "swa_ring", torch.uint8, (B, R, RECORD_BYTES)), R, int(W),
            _ptr(q_pos, "q_pos", torch.int32, (B, T)), B, T, int(m_hca),
            _ptr(out, "out", torch.bfloat16, (B, T, HEADS, DIM)), _ptr(lse, "lse", torch.float32, (B, T, HEADS))]
    tail = [_ptr(ws, "workspace", torch.uint8), 0 if ws is None else ws.numel(), _status(status, dev), _stream(stream)]
    if epi is None:
        _check(load().hca_sink_attention_decode(*args, *tail), "hca_sink_attention_decode")
    else:
        _check(load().hca_sink_attention_decode_ex(*args, C.byref(epi), *tail), "hca_sink_attention_decode_ex")
    return ((out_fp4, out_fp4_scale) if fp4_out else out), lse


def csa_decode_step(q_idx, q_idx_scale, w_idx, k_idx, k_idx_scale, q, sink, softmax_scale: float,
                    comp: csa_cache_desc, swa_ring, W: int, q_pos, n_comp, m: int, k: int, out=None, lse=None,
                    topk_idx=None, topk_cnt=None, ws=None, stream=None, status=None, inverse_rope: bool = False,
                    rope_theta: float = 10000.0, fp4_out: bool = False, out_fp4=None, out_fp4_scale=None):
    """Returns (out, lse); with fp4_out, ((out_fp4, out_fp4_scale), lse)."""
    B, T = q_pos.shape
    Ncap = k_idx.shape[1]
    R = swa_ring.shape[1]
    dev = q.device
    epi, out_fp4, out_fp4_scale = _epilogue(B, T, dev, inverse_rope, rope_theta, fp4_out, out_fp4, out_fp4_scale)
    if out is None and not fp4_out:
        out = torch.empty((B, T, HEADS, DIM), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, T, HEADS), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(OP_DECODE_STEP, B, T, Ncap, k, dev)
    u8 = (torch.uint8, torch.float8_e4m3fn)
    args = [_ptr(q_idx, "q_idx", u8, (B, T, IDX_HEADS, IDX_DIM)),
            _ptr(q_idx_scale, "q_idx_scale", torch.float32, (B, T, IDX_HEADS)),
            _ptr(w_idx, "w_idx", torch.float32, (B, T, IDX_HEADS)), _ptr(k_idx, "k_idx", u8, (B, Ncap, IDX_DIM)),
            _ptr(k_idx_scale, "k_idx_scale", torch.float32, (B, Ncap)),
            _ptr(q, "q", torch.bfloat16, (B, T, HEADS, DIM)), _ptr(sink, "sink", torch.float32, (HEADS,)),
            float(softmax_scale), comp, _ptr(swa_ring, "swa_ring", torch.uint8, (B, R, RECORD_BYTES)), R, int(W),
            _ptr(q_pos, "q_pos", torch.int32, (B, T)), _ptr(n_comp, "n_comp", torch.int32, (B,)),
            B, T, Ncap, int(m), int(k),
            _ptr(out, "out", torch.bfloat16, (B, T, HEADS, DIM)), _ptr(lse, "lse", torch.float32, (B, T, HEADS)),
            _ptr(topk_idx, "topk_idx", torch.int32, (B, T, k)), _ptr(topk_cnt, "topk_cnt", torch.int32, (B, T))]
    tail = [_ptr(ws, "workspace", torch.uint8), 0 if ws is None else ws.numel(), _status(status, dev), _stream(stream)]
    if epi is None:
        _check(load().csa_decode_step(*args, *tail), "csa_decode_step")
    else:
        _check(load().csa_decode_step_ex(*args, C.byref(epi), *tail), "csa_decode_step_ex")
    return ((out_fp4, out_fp4_scale) if fp4_out else out), lse


def _hptr(t: torch.Tensor, name: str, dtype, shape):
    """Host tensor check for the pipeline: CPU, contiguous, dtype, shape."""
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def csa_pipeline_staging_bytes(B: int, T: int, depth: int) -> int:
    return int(load().csa_pipeline_staging_bytes(B, T, depth))


def csa_pipeline_create(B: int, T: int, depth: int, staging: torch.Tensor, stream=None) -> int:
    """Handle of a new host-I/O pipeline on the current device; ``staging`` is
    a uint8 device tensor of at least csa_pipeline_staging_bytes(B, T, depth)."""
    h = C.c_void_p()
    _check(load().csa_pipeline_create(C.byref(h), B, T, depth, _ptr(staging, "staging", torch.uint8),
                                      staging.numel(), _stream(stream)), "csa_pipeline_create")
    return h.value


def csa_decode_step_host(pipeline: int, B: int, T: int, h_q_idx, h_q_idx_scale, h_w_idx, h_q, h_q_pos, k_idx,
                         k_idx_scale, sink, softmax_scale: float, comp: csa_cache_desc, swa_ring, W: int, n_comp,
                         m: int, k: int, h_out, h_lse, ws, status=None) -> int:
    """Enqueue one step; h_* are host tensors (page-locked for overlap), the
    rest is the device-resident layer state. Returns the step's ordinal."""
    Ncap = k_idx.shape[1]
    R = swa_ring.shape[1]
    u8 = (torch.uint8, torch.float8_e4m3fn)
    step = C.c_int64(-1)
    _check(load().csa_decode_step_host(
        C.c_void_p(pipeline), _hptr(h_q_idx, "h_q_idx", u8, (B, T, IDX_HEADS, IDX_DIM)),
        _hptr(h_q_idx_scale, "h_q_idx_scale", torch.float32, (B, T, IDX_HEADS)),
        _hptr(h_w_idx, "h_w_idx", torch.float32, (B, T, IDX_HEADS)),
        _hptr(h_q, "h_q", torch.bfloat16, (B, T, HEADS, DIM)), _hptr(h_q_pos, "h_q_pos", torch.int32, (B, T)),
        _ptr(k_idx, "k_idx", u8, (B, Ncap, IDX_DIM)), _ptr(k_idx_scale, "k_idx_scale", torch.float32, (B, Ncap)),
        _ptr(sink, "sink", torch.float32, (HEADS,)), float(softmax_scale), comp,
        _ptr(swa_ring, "swa_ring", torch.uint8, (B, R, RECORD_BYTES)), R, int(W),
        _ptr(n_comp, "n_comp", torch.int32, (B,)), Ncap, int(m), int(k),
        _hptr(h_out, "h_out", torch.bfloat16, (B, T, HEADS, DIM)), _hptr(h_lse, "h_lse", torch.float32, (B, T, HEADS)),
        _ptr(ws, "workspace", torch.uint8), 0 if ws is None else ws.numel(), _status(status, k_idx.device),
        C.byref(step)), "csa_decode_step_host")
    return int(step.value)


def csa_pipeline_wait(pipeline: int, step: int):
    _check(load().csa_pipeline_wait(C.c_void_p(pipeline), int(step)), "csa_pipeline_wait")


def csa_pipeline_sync(pipeline: int):
    _check(load().csa_pipeline_sync(C.c_void_p(pipeline)), "csa_pipeline_sync")


def csa_pipeline_destroy(pipeline: int):
    _check(load().csa_pipeline_destroy(C.c_void_p(pipeline)), "csa_pipeline_destroy")


class HostPipeline:
    """Owns a pipeline handle and its device staging area (torch memory).
    ``step(...)`` enqueues csa_decode_step_host and returns the ordinal;
    ``wait(i)`` / ``sync()`` block until results are in host memory."""

    def __init__(self, B: int, T: int, depth: int = 2, device=None, stream=None):
        n = csa_pipeline_staging_bytes(B, T, depth)
        if n == 0:
            raise ValueError(f"unsupported pipeline sizes B={B} T={T} depth={depth}")
        self.B, self.T, self.depth = B, T, depth
        self.staging = torch.empty(n, dtype=torch.uint8, device=device or torch.device("cuda"))
        self.handle = csa_pipeline_create(B, T, depth, self.staging, stream)

    def step(self, h_q_idx, h_q_idx_scale, h_w_idx, h_q, h_q_pos, k_idx, k_idx_scale, sink, softmax_scale, comp,
             swa_ring, W, n_comp, m, k, h_out, h_lse, ws, status=None) -> int:
        return csa_decode_step_host(self.handle, self.B, self.T, h_q_idx, h_q_idx_scale, h_w_idx, h_q, h_q_pos,
                                    k_idx, k_idx_scale, sink, softmax_scale, comp, swa_ring, W, n_comp, m, k,
                                    h_out, h_lse, ws, status)

    def wait(self, step: int):
        csa_pipeline_wait(self.handle, step)

    def sync(self):
        csa_pipeline_sync(self.handle)

    def close(self):
        if self.handle:
            h, self.handle = self.handle, None
            csa_pipeline_destroy(h)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def csa_check_device_status(host_status: torch.Tensor, status: torch.Tensor | None = None, stream=None,
                            device=None):
    """Enqueue (no synchronisation) a copy of the status word into
    ``host_status`` (an int32 CPU tensor of one element, page-locked for an
    asynchronous copy) and a reset of the word. Read ``host_status`` once the
    stream has passed this point."""
    if host_status.is_cuda or host_status.dtype != torch.int32 or host_status.numel() != 1:
        raise ValueError("host_status must be a one-element int32 CPU tensor")
    dev = status.device if status is not None else device
    _check(load().csa_check_device_status(_status(status, dev), host_status.data_ptr(), _stream(stream)),
           "csa_check_device_status")


def csa_read_device_error(stream=None, status: torch.Tensor | None = None, device=None) -> int:
    """Read and clear a status word (the device's default one unless given);
    blocking: synchronises the stream. For tests and diagnostics."""
    code = C.c_int32(0)
    dev = status.device if status is not None else device
    _check(load().csa_read_device_error(_status(status, dev), C.byref(code), _stream(stream)), "csa_read_device_error")
    return int(code.value)


def csa_debug_set_wait_limit_ns(ns: int):
    """Diagnostic: limit of the kernels' bounded waits for later launches (0 =
    the default of one second); see include/csa.h."""
    load().csa_debug_set_wait_limit_ns(int(ns))
