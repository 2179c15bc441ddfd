"""Pins for the causal visible range and the SWA window (a1)."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_visible_range_worked_cases():
    spec = json.load(open(os.path.join(GOLDEN, "visible_range.json")))
    for c in spec["cases"]:
        assert oracle.n_visible(c["p"], c["m"], c["n_comp"], c["cap"]) == c["n_vis"], c


def test_visible_range_brute_force_block_membership():
    # brute force: enumerate every block and keep those whose last token lies
    # strictly before the query's own block start
    for m in (1, 2, 4, 7, 128):
        for p in range(0, 3 * m + 3):
            own_block_start = (p // m) * m
            brute = sum(1 for c in range(0, p + 1) if (c + 1) * m <= own_block_start)
            assert oracle.n_visible(p, m, 10 ** 6, 10 ** 6) == brute, (m, p)


def _window_through_gather(p, W, R):
    """Read the SWA window back out of the oracle's gather: ring slot s of a
    1-record ring carries its own slot number in byte 0."""
    rec = 16
    ring = np.zeros((1, R, rec), dtype=np.uint8)
    ring[0, :, 0] = np.arange(R, dtype=np.uint8)
    cache = oracle.Cache(np.zeros((1, rec), np.uint8), seq_stride=1, seq_capacity=1)
    kv, cnt = oracle.gather(cache, ring, W, np.full((1, 1, 1), -1, np.int32), np.zeros((1, 1), np.int32),
                            np.array([[p]], np.int32))
    return [int(s) for s in kv[0, 0, :cnt[0, 0], 0]]


def test_swa_window_worked_cases():
    spec = json.load(open(os.path.join(GOLDEN, "swa_window.json")))
    for c in spec["cases"]:
        R = max(c["W"], 131)
        slots = _window_through_gather(c["p"], c["W"], R)
        expect = [(j % R) for j in range(c["first"], c["first"] + c["count"])]
        assert slots == expect, c
