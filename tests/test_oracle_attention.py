"""Pins for the oracle's sink-merged attention (a5), its candidate lists (a4)
and the HCA variant (a6)."""
import math

import numpy as np
import pytest
import torch

import oracle
from _lib_refs import (bf16_to_f64, dequant_records, make_records, random_bf16_bits,
                       softmax_attention_with_sink)

# small generic shapes: 3 scale blocks with a ragged last one (20 = 8+8+4)
H, DN, DR, SB = 3, 20, 6, 8
D = DN + DR
SCALE = 1.0 / math.sqrt(D)


def _row(q, sink, recs, scale=SCALE):
    return oracle.attention_row(q, np.asarray(sink, np.float32), scale, recs, DN, DR, SB)


def test_single_candidate_with_minus_inf_sink_returns_its_value_exactly():
    rng = np.random.default_rng(0)
    recs = make_records(rng, 1, DN, DR, SB)
    q = random_bf16_bits(rng, (H, D))
    o, lse = _row(q, [-np.inf] * H, recs)
    x = dequant_records(recs, DN, DR, SB).numpy()[0]
    for h in range(H):
        assert np.array_equal(o[h], x)
    z = SCALE * (bf16_to_f64(q).numpy() @ x)
    np.testing.assert_allclose(lse, z, rtol=0, atol=1e-13)


def test_textbook_softmax_with_minus_inf_sink():
    rng = np.random.default_rng(1)
    recs = make_records(rng, 17, DN, DR, SB)
    q = random_bf16_bits(rng, (H, D))
    o, lse = _row(q, [-np.inf] * H, recs)
    ref_o, ref_lse = softmax_attention_with_sink(q, [-np.inf] * H, SCALE,
                                                 dequant_records(recs, DN, DR, SB))
    np.testing.assert_allclose(o, ref_o.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-13, atol=1e-13)


def test_finite_sink_is_a_zero_value_logit():
    rng = np.random.default_rng(2)
    recs = make_records(rng, 9, DN, DR, SB)
    q = random_bf16_bits(rng, (H, D))
    sink = np.array([-0.5, 0.0, 3.0], np.float32)
    o, lse = _row(q, sink, recs)
    ref_o, ref_lse = softmax_attention_with_sink(q, sink, SCALE, dequant_records(recs, DN, DR, SB))
    np.testing.assert_allclose(o, ref_o.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-13, atol=1e-13)


def test_identical_candidates_closed_form():
    rng = np.random.default_rng(3)
    rec = make_records(rng, 1, DN, DR, SB)
    q = random_bf16_bits(rng, (H, D))
    sink = np.array([0.25, -1.0, 2.0], np.float32)
    x = dequant_records(rec, DN, DR, SB).numpy()[0]
    z = SCALE * (bf16_to_f64(q).numpy() @ x)
    for n in (1, 2, 5):
        o, lse = _row(q, sink, np.repeat(rec, n, axis=0))
        for h in range(H):
            w = n * math.exp(z[h]) / (math.exp(float(sink[h])) + n * math.exp(z[h]))
            np.testing.assert_allclose(o[h], w * x, rtol=1e-13, atol=1e-15)
            assert abs(lse[h] - math.log(math.exp(float(sink[h])) + n * math.exp(z[h]))) < 1e-13


def test_large_sink_drives_output_to_zero_and_lse_to_sink():
    rng = np.random.default_rng(4)
    recs = make_records(rng, 4, DN, DR, SB)
    q = random_bf16_bits(rng, (H, D))
    o, lse = _row(q, [800.0] * H, recs)
    assert np.max(np.abs(o)) < 1e-300
    np.testing.assert_allclose(lse, 800.0, rtol=0, atol=1e-12)


def test_hand_worked_example():
    # H=1, Dn=2 (one scale block), Dr=2, scale 1, sink 0.
    # x1: nope codes 1.0, 2.0 with scale 0.5 -> (0.5, 1.0); rope (1.0, 0.0)
    # x2: nope codes -1.0, 0 with scale 2.0 -> (-2.0, 0.0); rope (0.0, 2.0)
    # q = (1, 1, 0, 0.5): z1 = 1.5, z2 = -1.0
    # o = (e^1.5 x1 + e^-1 x2) / (1 + e^1.5 + e^-1), lse = ln(1 + e^1.5 + e^-1)
    def rec(n0, n1, r0, r1, s):
        b = bytes([n0, n1]) + np.array([r0, r1], np.uint16).tobytes() + np.array([s], np.float32).tobytes()
        return np.frombuffer(b, np.uint8)
    recs = np.stack([rec(0x38, 0x40, 0x3F80, 0x0000, 0.5), rec(0xB8, 0x00, 0x0000, 0x4000, 2.0)])
    q = np.array([[0x3F80, 0x3F80, 0x0000, 0x3F00]], np.uint16)
    o, lse = oracle.attention_row(q, np.array([0.0], np.float32), 1.0, recs, 2, 2, 2)
    den = 1 + math.exp(1.5) + math.exp(-1.0)
    x1, x2 = np.array([0.5, 1.0, 1.0, 0.0]), np.array([-2.0, 0.0, 0.0, 2.0])
    np.testing.assert_allclose(o[0], (math.exp(1.5) * x1 + math.exp(-1.0) * x2) / den, rtol=1e-15, atol=1e-16)
    assert abs(lse[0] - math.log(den)) < 1e-15


def test_lse_merge_of_two_segments_equals_joint():
    rng = np.random.default_rng(5)
    recs = make_records(rng, 12, DN, DR, SB)
    q = random_bf16_bits(rng, (H, D))
    sink = np.array([0.3, -2.0, 1.0], np.float32)
    o, lse = _row(q, sink, recs)
    o1, l1 = _row(q, [-np.inf] * H, recs[:5])
    o2, l2 = _row(q, [-np.inf] * H, recs[5:])
    for h in range(H):
        w = np.array([l1[h], l2[h], float(sink[h])])
        M = w.max()
        den = np.exp(w - M).sum()
        merged = (math.exp(l1[h] - M) * o1[h] + math.exp(l2[h] - M) * o2[h]) / den
        np.testing.assert_allclose(o[h], merged, rtol=1e-12, atol=1e-15)
        assert abs(lse[h] - (M + math.log(den))) < 1e-12


def test_empty_candidate_list():
    q = np.zeros((H, D), np.uint16)
    o, lse = _row(q, [0.5, -np.inf, 2.0], np.zeros((0, DN + 2 * DR + 12), np.uint8))
    assert np.all(o == 0)
    assert lse[0] == np.float32(0.5) and np.isneginf(lse[1]) and lse[2] == 2.0


# --------------------------------------------------------------------------
# batched CSA / HCA drivers and the candidate list
# --------------------------------------------------------------------------

def _cache_setup(rng, B, N, R, paged=False, pr=4):
    recs = make_records(rng, B * N, DN, DR, SB)
    ring = make_records(rng, B * R, DN, DR, SB).reshape(B, R, -1)
    if not paged:
        return oracle.Cache(recs, seq_stride=N, seq_capacity=N), recs.reshape(B, N, -1), ring
    max_pages = (N + pr - 1) // pr
    perm = rng.permutation(B * max_pages).astype(np.int32).reshape(B, max_pages)
    pool = np.zeros((B * max_pages * pr, recs.shape[1]), np.uint8)
    logical = recs.reshape(B, N, -1)
    for b in range(B):
        for c in range(N):
            pool[perm[b, c // pr] * pr + c % pr] = logical[b, c]
    return oracle.Cache(pool, seq_stride=0, seq_capacity=N, block_table=perm, page_records=pr), logical, ring


def _candidates(logical, ring, sel, cnt, p, W):
    R = ring.shape[0]
    win = list(range(max(0, p - W + 1), p + 1))
    return np.concatenate([logical[sel[:cnt]], ring[[j % R for j in win]]], axis=0) if (cnt or win) else \
        np.zeros((0, logical.shape[-1]), np.uint8)


@pytest.mark.parametrize("paged", [False, True])
def test_csa_attention_equals_library_softmax_on_gathered_candidates(paged):
    rng = np.random.default_rng(6)
    B, T, N, R, W, k = 2, 2, 23, 6, 5, 4
    cache, logical, ring = _cache_setup(rng, B, N, R, paged=paged)
    q = random_bf16_bits(rng, (B, T, H, D))
    sink = np.array([0.1, -0.4, 1.2], np.float32)
    q_pos = np.array([[3, 4], [60, 61]], np.int32)
    topk_idx = np.full((B, T, k), -1, np.int32)
    topk_cnt = np.array([[0, 1], [4, 3]], np.int32)
    topk_idx[0, 1, :1] = [0]
    topk_idx[1, 0] = [14, 3, 9, 0]
    topk_idx[1, 1, :3] = [2, 14, 7]
    o, lse = oracle.csa_attention(q, sink, SCALE, cache, ring, W, topk_idx, topk_cnt, q_pos, DN, DR, SB)
    for b in range(B):
        for t in range(T):
            cands = _candidates(logical[b], ring[b], topk_idx[b, t], topk_cnt[b, t], q_pos[b, t], W)
            ro, rl = softmax_attention_with_sink(q[b, t], sink, SCALE, dequant_records(cands, DN, DR, SB))
            np.testing.assert_allclose(o[b, t], ro.numpy(), rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(lse[b, t], rl.numpy(), rtol=1e-13, atol=1e-13)
    kv, kvc = oracle.gather(cache, ring, W, topk_idx, topk_cnt, q_pos)
    for b in range(B):
        for t in range(T):
            cands = _candidates(logical[b], ring[b], topk_idx[b, t], topk_cnt[b, t], q_pos[b, t], W)
            assert kvc[b, t] == len(cands)
            assert np.array_equal(kv[b, t, :len(cands)], cands)


def test_permutation_invariance_of_selected_set():
    rng = np.random.default_rng(7)
    B, T, N, R, W, k = 1, 1, 40, 5, 5, 16
    cache, logical, ring = _cache_setup(rng, B, N, R)
    q = random_bf16_bits(rng, (B, T, H, D))
    sink = np.zeros(H, np.float32)
    q_pos = np.array([[200]], np.int32)
    sel = rng.choice(N, size=k, replace=False).astype(np.int32)
    o1, l1 = oracle.csa_attention(q, sink, SCALE, cache, ring, W, sel[None, None], np.array([[k]], np.int32), q_pos,
                                  DN, DR, SB)
    o2, l2 = oracle.csa_attention(q, sink, SCALE, cache, ring, W, rng.permutation(sel)[None, None],
                                  np.array([[k]], np.int32), q_pos, DN, DR, SB)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(l1, l2, rtol=1e-14, atol=1e-14)


def test_overlap_counts_a_token_twice():
    # a SWA token byte-identical to a selected compressed record doubles its
    # weight: softmax over {A, A, C} with sink -inf
    rng = np.random.default_rng(8)
    cache, logical, ring = _cache_setup(rng, 1, 8, 4)
    ring = ring.copy()
    A = logical[0, 5]
    W = 2
    p = 10  # window = positions 9, 10 -> slots 1, 2
    ring[0, 1] = A
    q = random_bf16_bits(rng, (1, 1, H, D))
    o, _ = oracle.csa_attention(q, np.full(H, -np.inf, np.float32), SCALE, cache, ring, W,
                                np.array([[[5]]], np.int32), np.array([[1]], np.int32),
                                np.array([[p]], np.int32), DN, DR, SB)
    xa = dequant_records(A[None], DN, DR, SB).numpy()[0]
    xc = dequant_records(ring[0, 2][None], DN, DR, SB).numpy()[0]
    qd = bf16_to_f64(q[0, 0]).numpy()
    for h in range(H):
        za, zc = SCALE * qd[h] @ xa, SCALE * qd[h] @ xc
        ref = (2 * math.exp(za) * xa + math.exp(zc) * xc) / (2 * math.exp(za) + math.exp(zc))
        np.testing.assert_allclose(o[0, 0, h], ref, rtol=1e-12, atol=1e-15)


def test_hca_equals_csa_with_every_visible_entry_selected():
    rng = np.random.default_rng(9)
    B, T, N, R, W, m = 2, 1, 12, 4, 4, 8
    cache, logical, ring = _cache_setup(rng, B, N, R)
    q = random_bf16_bits(rng, (B, T, H, D))
    sink = np.array([0.0, 1.0, -1.0], np.float32)
    q_pos = np.array([[70], [33]], np.int32)   # n_vis = 8, 4
    n_comp = np.array([12, 12], np.int32)
    oh, lh = oracle.hca_attention(q, sink, SCALE, cache, n_comp, ring, W, q_pos, m, DN, DR, SB)
    k = N
    idx = np.full((B, T, k), -1, np.int32)
    cnt = np.zeros((B, T), np.int32)
    for b in range(B):
        nv = min(q_pos[b, 0] // m, n_comp[b])
        idx[b, 0, :nv] = np.arange(nv)
        cnt[b, 0] = nv
    oc, lc = oracle.csa_attention(q, sink, SCALE, cache, ring, W, idx, cnt, q_pos, DN, DR, SB)
    assert np.array_equal(oh, oc) and np.array_equal(lh, lc)


def test_hca_causality_poisoned_future_entries():
    rng = np.random.default_rng(10)
    B, N, R, W, m = 1, 10, 4, 4, 16
    cache, logical, ring = _cache_setup(rng, B, N, R)
    q = random_bf16_bits(rng, (B, 1, H, D))
    sink = np.zeros(H, np.float32)
    q_pos = np.array([[100]], np.int32)  # n_vis = 6
    a = oracle.hca_attention(q, sink, SCALE, cache, np.array([N], np.int32), ring, W, q_pos, m, DN, DR, SB)
    poisoned = cache.records.copy()
    poisoned[6:, :DN] = 0x7E
    poisoned[6:, DN + 2 * DR:] = np.frombuffer(np.full(3, 1e4, np.float32).tobytes(), np.uint8)
    cache2 = oracle.Cache(poisoned, seq_stride=N, seq_capacity=N)
    b = oracle.hca_attention(q, sink, SCALE, cache2, np.array([N], np.int32), ring, W, q_pos, m, DN, DR, SB)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_out_of_cache_index_is_an_error():
    rng = np.random.default_rng(11)
    cache, logical, ring = _cache_setup(rng, 1, 8, 4)
    q = random_bf16_bits(rng, (1, 1, H, D))
    with pytest.raises(RuntimeError):
        oracle.csa_attention(q, np.zeros(H, np.float32), SCALE, cache, ring, 4, np.array([[[8]]], np.int32),
                             np.array([[1]], np.int32), np.array([[50]], np.int32), DN, DR, SB)


def test_brute_force_pipeline_against_python_restatement():
    """Tiny end-to-end case (indexer -> top-k -> attention) against a short
    pure-Python fp64 restatement written independently of the C oracle."""
    import brute_force as bf
    rng = np.random.default_rng(12)
    for trial in range(6):
        B, T, N, R, W, k, m, Hi, Di = 1, 2, 8, 4, 4, 3, 4, 2, 4
        cache, logical, ring = _cache_setup(rng, B, N, R)
        qc = rng.integers(0, 0x7E, size=(B, T, Hi, Di), dtype=np.uint8) ^ (rng.integers(0, 2, (B, T, Hi, Di), dtype=np.uint8) << 7)
        kc = rng.integers(0, 0x7E, size=(B, N, Di), dtype=np.uint8) ^ (rng.integers(0, 2, (B, N, Di), dtype=np.uint8) << 7)
        qs = rng.random((B, T, Hi)).astype(np.float32) + 0.5
        ks = rng.random((B, N)).astype(np.float32) + 0.5
        w = rng.standard_normal((B, T, Hi)).astype(np.float32)
        q_pos = np.array([[17 + trial, 18 + trial]], np.int32)
        n_comp = np.array([N], np.int32)
        q = random_bf16_bits(rng, (B, T, H, D))
        sink = rng.standard_normal(H).astype(np.float32)
        logits = oracle.indexer_logits(qc, qs, w, kc, ks, q_pos, n_comp, m)
        idx, cnt = oracle.topk(logits, q_pos, n_comp, m, k)
        o, lse = oracle.csa_attention(q, sink, SCALE, cache, ring, W, idx, cnt, q_pos, DN, DR, SB)
        for t in range(T):
            bl, bsel, bo, blse = bf.decode_one(qc[0, t], qs[0, t], w[0, t], kc[0], ks[0], int(q_pos[0, t]), m, N, k,
                                               q[0, t], sink, SCALE, logical[0], ring[0], W, DN, DR, SB)
            fin = np.isfinite(logits[0, t])
            np.testing.assert_allclose(logits[0, t][fin], np.array(bl)[fin], rtol=1e-12, atol=1e-12)
            assert sorted(idx[0, t, :cnt[0, t]].tolist()) == sorted(bsel)
            np.testing.assert_allclose(o[0, t], np.array(bo), rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(lse[0, t], np.array(blse), rtol=1e-12, atol=1e-12)
