"""The C-ABI library builds, loads and exports every symbol include/csa.h
declares; host-side validation rejects bad arguments before any launch.
No test here needs a GPU (no call reaches a kernel)."""
import ctypes as C
import os
import re
import subprocess

import pytest

import compressed_sparse_decode_gb300 as csd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    csd.build()
    return csd.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "csa.h")).read()
    return sorted(set(re.findall(r"CSA_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)))


def test_header_declares_the_binding_names():
    assert _declared() == sorted(csd.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", csd.LIB], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in _declared():
        assert name in exported, name
        assert hasattr(lib, name)
    # nothing else leaks out of the library's C namespace
    assert not [s for s in exported if s.startswith("csa") and s not in _declared()]


def test_version_and_status_strings(lib):
    assert csd.csa_version() == 100
    assert csd.status_string(csd.OK) == "ok"
    assert "workspace" in csd.status_string(csd.ERR_WORKSPACE)
    assert csd.status_string(99) == "unknown status"


def test_workspace_sizes(lib):
    assert csd.csa_workspace_bytes(csd.OP_INDEXER, 32, 1, 32768, 2048) == 0
    step = csd.csa_workspace_bytes(csd.OP_DECODE_STEP, 32, 1, 32768, 2048)
    assert step >= 4 * 32 * 32768 + 2 * 4 * 32 * 2048
    assert step % 256 == 0
    assert csd.csa_workspace_bytes(csd.OP_TOPK, 0, 1, 10, 1) == 0
    # rows up to 32768 entries: one pass, no workspace; longer rows whose
    # slices' candidates fit one pass: per (row, slice) k indices + k keys + its k-th key
    assert csd.csa_workspace_bytes(csd.OP_TOPK, 32, 1, 32768, 2048) == 0
    assert csd.csa_workspace_bytes(csd.OP_TOPK, 4, 4, 262144, 2048) == 4 * (16 * 8) * (2 * 2048 + 1)
    assert csd.csa_workspace_bytes(csd.OP_TOPK, 3, 2, 70001, 1000) == 4 * (6 * 3) * (2 * 1000 + 1)
    assert csd.csa_workspace_bytes(csd.OP_TOPK, 1, 1, 40000, 7) == 4 * (16 + 14 + 2)  # keys 16-byte aligned
    assert csd.csa_workspace_bytes(csd.OP_TOPK, 1, 1, 17 * 32768, 2048) == 0  # 17 slices x 2048 > 32768


def test_host_validation_rejects_before_launch(lib):
    P = C.c_void_p
    fake = P(0x1000)  # never dereferenced: validation fails first
    # null pointers
    assert lib.csa_indexer_logits(None, None, None, None, None, None, None, 1, 1, 8, 4, None, None, None) == csd.ERR_INVALID_ARG
    # T beyond the supported maximum
    assert lib.csa_indexer_logits(fake, fake, fake, fake, fake, fake, fake, 1, 129, 8, 4, fake, None, None) == csd.ERR_INVALID_ARG
    # misaligned logits pointer
    assert lib.csa_indexer_logits(fake, fake, fake, fake, fake, fake, fake, 1, 1, 8, 4, P(0x1004), None, None) == csd.ERR_INVALID_ARG
    # k larger than the capacity / the maximum
    assert lib.csa_topk(fake, fake, fake, 1, 1, 8, 4, 9, fake, fake, None, 0, None, None) == csd.ERR_UNSUPPORTED
    assert lib.csa_topk(fake, fake, fake, 1, 1, 10000, 4, 4096, fake, fake, None, 0, None, None) == csd.ERR_UNSUPPORTED
    # cache descriptor without records, window larger than the ring
    bad = csd.csa_cache_desc()
    assert lib.csa_gather_swa(bad, fake, 128, 128, fake, fake, fake, 1, 1, 4, fake, fake, None, None) == csd.ERR_INVALID_ARG
    good = csd.csa_cache_desc()
    good.base, good.n_records, good.seq_stride, good.seq_capacity = 0x1000, 10, 10, 10
    assert lib.csa_gather_swa(good, fake, 64, 128, fake, fake, fake, 1, 1, 4, fake, fake, None, None) == csd.ERR_INVALID_ARG
    # contiguous mode with overlapping sequences
    over = csd.csa_cache_desc()
    over.base, over.n_records, over.seq_stride, over.seq_capacity = 0x1000, 100, 5, 10
    assert lib.csa_gather_swa(over, fake, 128, 128, fake, fake, fake, 2, 1, 4, fake, fake, None, None) == csd.ERR_INVALID_ARG
    # non-positive softmax scale
    assert lib.csa_sink_attention_decode(fake, fake, C.c_float(0.0), good, fake, 128, 128, fake, fake, fake, 1, 1, 4,
                                         fake, fake, None, 0, None, None) == csd.ERR_INVALID_ARG
    # decode step without workspace
    assert lib.csa_decode_step(fake, fake, fake, fake, fake, fake, fake, C.c_float(0.1), good, fake, 128, 128, fake,
                               fake, 1, 1, 10, 4, 4, fake, fake, None, None, None, 0, None, None) == csd.ERR_WORKSPACE


def test_pipeline_staging_sizes(lib):
    B, T = 32, 1
    def up(n):
        return (n + 255) // 256 * 256
    # q_idx, q_idx_scale, w_idx, q, q_pos, out, lse
    one = (up(B * T * 64 * 128) + 2 * up(B * T * 64 * 4) + up(B * T * 128 * 512 * 2) + up(B * T * 4)
           + up(B * T * 128 * 512 * 2) + up(B * T * 128 * 4))
    assert csd.csa_pipeline_staging_bytes(B, T, 2) == 2 * one
    assert csd.csa_pipeline_staging_bytes(B, T, 3) == 3 * one
    assert csd.csa_pipeline_staging_bytes(B, T, 1) == 0          # depth below 2
    assert csd.csa_pipeline_staging_bytes(B, T, 5) == 0          # depth above the maximum
    assert csd.csa_pipeline_staging_bytes(B, 129, 2) == 0        # T above the maximum
    assert csd.csa_pipeline_staging_bytes(0, 1, 2) == 0


def test_pipeline_validation_before_any_cuda_call(lib):
    P = C.c_void_p
    h = C.c_void_p(0)
    need = csd.csa_pipeline_staging_bytes(4, 1, 2)
    assert lib.csa_pipeline_create(None, 4, 1, 2, P(0x1000), need, None) == csd.ERR_INVALID_ARG
    assert lib.csa_pipeline_create(C.byref(h), 4, 1, 1, P(0x1000), need, None) == csd.ERR_INVALID_ARG
    assert lib.csa_pipeline_create(C.byref(h), 4, 1, 2, None, need, None) == csd.ERR_INVALID_ARG
    assert lib.csa_pipeline_create(C.byref(h), 4, 1, 2, P(0x1080), need, None) == csd.ERR_INVALID_ARG  # not 256-aligned
    assert lib.csa_pipeline_create(C.byref(h), 4, 1, 2, P(0x1000), need - 1, None) == csd.ERR_INVALID_ARG
    assert h.value is None
    good = csd.csa_cache_desc()
    good.base, good.n_records, good.seq_stride, good.seq_capacity = 0x1000, 10, 10, 10
    fake = P(0x1000)
    step = C.c_int64(-1)
    assert lib.csa_decode_step_host(None, *([fake] * 8), C.c_float(0.1), good, fake, 128, 128, fake, 10, 4, 4,
                                    fake, fake, fake, 1 << 20, None, C.byref(step)) == csd.ERR_INVALID_ARG
    assert step.value == -1
    assert lib.csa_pipeline_wait(None, 0) == csd.ERR_INVALID_ARG
    assert lib.csa_pipeline_sync(None) == csd.ERR_INVALID_ARG
    assert lib.csa_pipeline_destroy(None) == csd.OK


def test_decode_step_checks_every_argument_before_launching(lib):
    fake = C.c_void_p(0x1000)
    good = csd.csa_cache_desc()
    good.base, good.n_records, good.seq_stride, good.seq_capacity = 0x1000, 10, 10, 10
    ws = csd.csa_workspace_bytes(csd.OP_DECODE_STEP, 1, 1, 10, 4)
    args = [fake] * 7 + [C.c_float(0.1), good, fake, 128, 128, fake, fake, 1, 1, 10, 4, 4, fake, fake, None, None,
                         fake, ws, None, None]
    # a null sink (an attention argument) is reported before the indexer launches
    bad = list(args)
    bad[6] = None
    assert lib.csa_decode_step(*bad) == csd.ERR_INVALID_ARG
    # a window larger than the ring
    bad = list(args)
    bad[10] = 64
    assert lib.csa_decode_step(*bad) == csd.ERR_INVALID_ARG
    # misaligned output
    bad = list(args)
    bad[19] = C.c_void_p(0x1004)
    assert lib.csa_decode_step(*bad) == csd.ERR_INVALID_ARG


def test_status_word_checks(lib):
    P = C.c_void_p
    host = C.c_int32(7)
    # null or misaligned words are rejected before anything is enqueued
    assert lib.csa_check_device_status(None, C.byref(host), None) == csd.ERR_INVALID_ARG
    assert lib.csa_check_device_status(P(0x1002), C.byref(host), None) == csd.ERR_INVALID_ARG
    assert lib.csa_check_device_status(P(0x1000), None, None) == csd.ERR_INVALID_ARG
    assert lib.csa_read_device_error(None, C.byref(host), None) == csd.ERR_INVALID_ARG
    assert host.value == 7
    # a misaligned status word is an argument error of every compute call
    fake = P(0x1000)
    assert lib.csa_indexer_logits(fake, fake, fake, fake, fake, fake, fake, 1, 1, 8, 4, fake, P(0x1001),
                                  None) == csd.ERR_INVALID_ARG
    assert lib.csa_topk(fake, fake, fake, 1, 1, 8, 4, 4, fake, fake, None, 0, P(0x1002), None) == csd.ERR_INVALID_ARG
    good = csd.csa_cache_desc()
    good.base, good.n_records, good.seq_stride, good.seq_capacity = 0x1000, 10, 10, 10
    assert lib.csa_sink_attention_decode(fake, fake, C.c_float(0.1), good, fake, 128, 128, fake, fake, fake, 1, 1, 4,
                                         fake, fake, None, 0, P(0x1003), None) == csd.ERR_INVALID_ARG
    assert lib.csa_sink_attention_decode_noalloc(fake, fake, C.c_float(0.1), good, fake, 128, 128, fake, fake, fake,
                                                 1, 1, 4, fake, fake, P(0x1003), None) == csd.ERR_INVALID_ARG


def test_noalloc_rejects_like_the_workspace_call(lib):
    """The allocation-free attention entry runs the same host checks as the
    workspace entry: each bad argument gets the same status from both."""
    fake = C.c_void_p(0x1000)
    good = csd.csa_cache_desc()
    good.base, good.n_records, good.seq_stride, good.seq_capacity = 0x1000, 10, 10, 10
    bad_cache = csd.csa_cache_desc()
    over = csd.csa_cache_desc()
    over.base, over.n_records, over.seq_stride, over.seq_capacity = 0x1000, 100, 5, 10
    cases = [
        dict(q=None), dict(comp=bad_cache), dict(comp=over, B=2), dict(W=600, R=600), dict(R=64),
        dict(scale=0.0), dict(k=4096), dict(T=129), dict(out=C.c_void_p(0x1008)),
    ]
    for c in cases:
        a = dict(q=fake, comp=good, R=128, W=128, B=1, T=1, k=4, out=fake, scale=0.1)
        a.update(c)
        common = (a["q"], fake, C.c_float(a["scale"]), a["comp"], fake, a["R"], a["W"], fake, fake, fake, a["B"],
                  a["T"], a["k"], a["out"], fake)
        ws_status = lib.csa_sink_attention_decode(*common, None, 0, None, None)
        na_status = lib.csa_sink_attention_decode_noalloc(*common, None, None)
        assert ws_status == na_status != csd.OK, c


def test_epilogue_entry_points_validate_before_launch(lib):
    """The _ex calls check the same arguments as the plain calls (a NULL
    epilogue gives the same status) and reject a bad epilogue up front."""
    fake = C.c_void_p(0x1000)
    good = csd.csa_cache_desc()
    good.base, good.n_records, good.seq_stride, good.seq_capacity = 0x1000, 10, 10, 10
    for c in [dict(q=None), dict(R=64), dict(scale=0.0), dict(k=4096), dict(T=129), dict(out=C.c_void_p(0x1008))]:
        a = dict(q=fake, R=128, W=128, T=1, k=4, out=fake, scale=0.1)
        a.update(c)
        common = (a["q"], fake, C.c_float(a["scale"]), good, fake, a["R"], a["W"], fake, fake, fake, 1, a["T"], a["k"],
                  a["out"], fake)
        plain = lib.csa_sink_attention_decode(*common, None, 0, None, None)
        ex = lib.csa_sink_attention_decode_ex(*common, None, None, 0, None, None)
        assert plain == ex != csd.OK, c
    common = (fake, fake, C.c_float(0.1), good, fake, 128, 128, fake, fake, fake, 1, 1, 4)
    hca_common = (fake, fake, C.c_float(0.1), good, fake, fake, 128, 128, fake, 1, 1, 128)
    E = csd.csa_attention_epilogue
    bad = [E(1, 1.0, None, None),                 # theta must exceed 1
           E(1, float("nan"), None, None),
           E(0, 0.0, 0x2000, None),               # E2M1 output without its multipliers
           E(0, 0.0, 0x2008, 0x3000),             # misaligned E2M1 output
           E(0, 0.0, 0x2000, 0x3004)]             # misaligned multipliers
    for e in bad:
        assert lib.csa_sink_attention_decode_ex(*common, fake, fake, C.byref(e), None, 0, None, None) == \
            csd.ERR_INVALID_ARG
        assert lib.hca_sink_attention_decode_ex(*hca_common, fake, fake, C.byref(e), None, 0, None, None) == \
            csd.ERR_INVALID_ARG
    # without E2M1 output `out` is required; with it, `out` may be NULL (then a later check fails: no ring)
    assert lib.csa_sink_attention_decode_ex(*common, None, fake, C.byref(E(1, 1e4, None, None)), None, 0, None,
                                            None) == csd.ERR_INVALID_ARG
    nor = (fake, fake, C.c_float(0.1), good, None, 128, 128, fake, fake, fake, 1, 1, 4)
    assert lib.csa_sink_attention_decode_ex(*nor, None, fake, C.byref(E(0, 0.0, 0x2000, 0x3000)), None, 0, None,
                                            None) == csd.ERR_INVALID_ARG


def test_decode_step_ex_checks_its_epilogue_before_launching(lib):
    fake = C.c_void_p(0x1000)
    good = csd.csa_cache_desc()
    good.base, good.n_records, good.seq_stride, good.seq_capacity = 0x1000, 10, 10, 10
    args = (fake, fake, fake, fake, fake, fake, fake, C.c_float(0.1), good, fake, 128, 128, fake, fake, 1, 1, 10, 4, 4)
    E = csd.csa_attention_epilogue
    # a bad epilogue is reported before the missing workspace
    assert lib.csa_decode_step_ex(*args, fake, fake, None, None, C.byref(E(1, 0.5, None, None)), None, 0, None,
                                  None) == csd.ERR_INVALID_ARG
    assert lib.csa_decode_step_ex(*args, None, fake, None, None, C.byref(E(0, 0.0, 0x2000, None)), None, 0, None,
                                  None) == csd.ERR_INVALID_ARG
    # NULL epilogue: the same status as csa_decode_step
    assert lib.csa_decode_step_ex(*args, fake, fake, None, None, None, None, 0, None, None) == \
        lib.csa_decode_step(*args, fake, fake, None, None, None, 0, None, None) == csd.ERR_WORKSPACE
    # E2M1 output stands in for `out`
    assert lib.csa_decode_step_ex(*args, None, fake, None, None, C.byref(E(0, 0.0, 0x2000, 0x3000)), None, 0, None,
                                  None) == csd.ERR_WORKSPACE


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "compressed_sparse_decode_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "csa_oracle" not in text, f
