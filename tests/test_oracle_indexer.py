"""Pins for the oracle's lightning-indexer logits (a2)."""
import numpy as np
import torch

import oracle
from _lib_refs import e4m3_to_f64


def _inputs(rng, B, T, N, Hi, Di, spread=1.0):
    def q8(shape):
        x = torch.as_tensor(rng.standard_normal(shape) * spread, dtype=torch.float32)
        amax = x.abs().amax(-1, keepdim=True)
        s = torch.where(amax > 0, amax / 448, torch.ones_like(amax))
        return (x / s).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy(), \
            s[..., 0].numpy().astype(np.float32).copy()
    qc, qs = q8((B, T, Hi, Di))
    kc, ks = q8((B, N, Di))
    w = (rng.standard_normal((B, T, Hi)) / 8).astype(np.float32)
    return qc, qs, w, kc, ks


def _library_logits(qc, qs, w, kc, ks, q_pos, n_comp, m):
    """torch fp64 einsum -> relu -> weighted head sum, masked by visibility."""
    q = e4m3_to_f64(qc) * torch.as_tensor(qs, dtype=torch.float64)[..., None]
    k = e4m3_to_f64(kc) * torch.as_tensor(ks, dtype=torch.float64)[..., None]
    dots = torch.einsum("bthd,bcd->bthc", q, k)
    out = (torch.as_tensor(w, dtype=torch.float64)[..., None] * torch.relu(dots)).sum(2)
    N = kc.shape[1]
    for b in range(out.shape[0]):
        for t in range(out.shape[1]):
            nv = min(int(q_pos[b, t]) // m, int(n_comp[b]), N)
            out[b, t, nv:] = -np.inf
    return out.numpy()


def test_indexer_matches_library_einsum():
    rng = np.random.default_rng(1)
    B, T, N, Hi, Di, m = 2, 3, 37, 5, 16, 4
    qc, qs, w, kc, ks = _inputs(rng, B, T, N, Hi, Di)
    q_pos = np.array([[100, 101, 102], [40, 41, 42]], np.int32)
    n_comp = np.array([30, 37], np.int32)
    got = oracle.indexer_logits(qc, qs, w, kc, ks, q_pos, n_comp, m)
    ref = _library_logits(qc, qs, w, kc, ks, q_pos, n_comp, m)
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    fin = np.isfinite(ref)
    np.testing.assert_allclose(got[fin], ref[fin], rtol=1e-12, atol=1e-12)


def test_single_head_unit_weight_is_relu_of_scaled_dot():
    rng = np.random.default_rng(2)
    qc, qs, w, kc, ks = _inputs(rng, 1, 1, 9, 1, 8)
    w[:] = 1.0
    got = oracle.indexer_logits(qc, qs, w, kc, ks, np.array([[400]], np.int32), np.array([9], np.int32), 4)
    q = e4m3_to_f64(qc[0, 0, 0]).numpy() * qs[0, 0, 0]
    for c in range(9):
        k = e4m3_to_f64(kc[0, c]).numpy() * ks[0, c]
        assert abs(got[0, 0, c] - max(0.0, float(q @ k))) <= 1e-12 * (1 + abs(float(q @ k)))


def test_relu_identity_under_query_negation():
    # relu(x) - relu(-x) = x, so I(q) - I(-q) = sum_h w_h * (scaled dot_h):
    # a linear closed form that a missing ReLU, a ReLU before the scales of the
    # wrong sign, or a dropped weight all violate.
    rng = np.random.default_rng(3)
    B, T, N, Hi, Di = 1, 2, 11, 6, 16
    qc, qs, w, kc, ks = _inputs(rng, B, T, N, Hi, Di)
    neg = qc ^ np.uint8(0x80)  # flip the E4M3 sign bit
    pos = np.array([[1000, 1001]], np.int32)
    nc = np.array([N], np.int32)
    a = oracle.indexer_logits(qc, qs, w, kc, ks, pos, nc, 4)
    b = oracle.indexer_logits(neg, qs, w, kc, ks, pos, nc, 4)
    q = e4m3_to_f64(qc).numpy() * qs[..., None]
    k = e4m3_to_f64(kc).numpy() * ks[..., None]
    lin = np.einsum("bth,bthd,bcd->btc", w.astype(np.float64), q, k)
    np.testing.assert_allclose(a - b, lin, rtol=1e-11, atol=1e-11)
    # and relu(x) + relu(-x) = |x|
    absf = np.einsum("bth,bthc->btc", w.astype(np.float64), np.abs(np.einsum("bthd,bcd->bthc", q, k)))
    np.testing.assert_allclose(a + b, absf, rtol=1e-11, atol=1e-11)


def test_negative_weight_sign():
    rng = np.random.default_rng(4)
    qc, qs, w, kc, ks = _inputs(rng, 1, 1, 5, 2, 8)
    pos, nc = np.array([[100]], np.int32), np.array([5], np.int32)
    base = oracle.indexer_logits(qc, qs, w, kc, ks, pos, nc, 4)
    w2 = w.copy()
    w2[..., 1] *= -1
    flipped = oracle.indexer_logits(qc, qs, w2, kc, ks, pos, nc, 4)
    q = e4m3_to_f64(qc).numpy() * qs[..., None]
    k = e4m3_to_f64(kc).numpy() * ks[..., None]
    head1 = np.maximum(np.einsum("d,cd->c", q[0, 0, 1], k[0]), 0) * w[0, 0, 1]
    np.testing.assert_allclose(base[0, 0] - flipped[0, 0], 2 * head1, rtol=1e-11, atol=1e-12)


def test_causality_poisoned_future_keys_do_not_change_visible_logits():
    rng = np.random.default_rng(5)
    B, T, N, Hi, Di, m = 2, 2, 40, 4, 16, 4
    qc, qs, w, kc, ks = _inputs(rng, B, T, N, Hi, Di)
    q_pos = np.array([[80, 81], [119, 120]], np.int32)  # n_vis 20,20 and 29,30
    n_comp = np.array([40, 40], np.int32)
    a = oracle.indexer_logits(qc, qs, w, kc, ks, q_pos, n_comp, m)
    kc2, ks2 = kc.copy(), ks.copy()
    kc2[0, 20:] = 0x7E
    ks2[0, 20:] = 1e6
    kc2[1, 30:] = 0x7E
    ks2[1, 30:] = 1e6
    b = oracle.indexer_logits(qc, qs, w, kc2, ks2, q_pos, n_comp, m)
    assert np.array_equal(a, b)
    assert np.all(np.isneginf(a[0, :, 20:])) and np.all(np.isfinite(a[0, :, :20]))
    assert np.all(np.isneginf(a[1, 0, 29:])) and np.all(np.isfinite(a[1, 1, :30]))
