"""Pins for the oracle's top-k selection (a3)."""
import numpy as np
import torch

import oracle


def _rows(scores):
    return np.asarray(scores, np.float64)[None, None, :]


def _sel(scores, n_vis, k, m=1):
    idx, cnt = oracle.topk(_rows(scores), np.array([[n_vis * m]], np.int32),
                           np.array([n_vis], np.int32), m, k)
    return idx[0, 0], int(cnt[0, 0])


def test_k_at_least_visible_selects_everything():
    rng = np.random.default_rng(0)
    s = rng.standard_normal(50)
    for n_vis in (0, 1, 7, 50):
        idx, cnt = _sel(s, n_vis, 64)
        assert cnt == n_vis
        assert sorted(idx[:cnt].tolist()) == list(range(n_vis))
        assert np.all(idx[cnt:] == -1)


def test_distinct_scores_match_torch_topk():
    rng = np.random.default_rng(1)
    for n, k in [(100, 10), (257, 64), (31, 31), (1000, 1)]:
        s = rng.permutation(n).astype(np.float64) + rng.random() * 0.5
        idx, cnt = _sel(s, n, k)
        ref = torch.topk(torch.as_tensor(s), k).indices.numpy()
        assert cnt == k
        assert idx[:cnt].tolist() == ref.tolist()  # distinct: order is the sorted order


def test_selection_properties_with_ties_brute_force():
    rng = np.random.default_rng(2)
    for trial in range(200):
        n = int(rng.integers(1, 24))
        k = int(rng.integers(1, 12))
        s = rng.integers(-3, 4, size=n).astype(np.float64)  # heavy ties
        idx, cnt = _sel(s, n, k)
        sel = set(idx[:cnt].tolist())
        assert cnt == min(k, n) and len(sel) == cnt
        uns = [i for i in range(n) if i not in sel]
        if uns and sel:
            lo = min(s[i] for i in sel)
            assert lo >= max(s[i] for i in uns)
            # ties at the threshold go to lower indices
            tied_sel = [i for i in sel if s[i] == lo]
            tied_uns = [i for i in uns if s[i] == lo]
            if tied_uns:
                assert max(tied_sel) < min(tied_uns)


def test_invisible_entries_never_selected():
    s = np.arange(20, dtype=np.float64)  # the largest scores sit at the end
    idx, cnt = oracle.topk(_rows(s), np.array([[40]], np.int32), np.array([20], np.int32), 4, 5)
    # n_vis = 40 // 4 = 10 -> the top 5 of entries 0..9
    assert int(cnt[0, 0]) == 5
    assert sorted(idx[0, 0].tolist()) == [5, 6, 7, 8, 9]


def test_negative_infinity_and_large_values():
    s = np.array([-np.inf, 3.0, -np.inf, 1e300, -1e300, 0.0])
    idx, cnt = _sel(s, 6, 3)
    assert sorted(idx[:cnt].tolist()) == [1, 3, 5]
