"""Pins for the oracle's attention-output epilogue: the E2M1 format and its
quantisation ("ROADMAP -- Stage E" §E6) and the inverse RoPE ("DSV4 Audit"
§A4)."""
import math

import numpy as np
import pytest

import oracle

# OCP Microscaling Formats spec, FP4 E2M1 element encodings: codes 0..7 are
# the positive magnitudes, codes 8..15 the same with the sign bit set.
OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_values_match_the_ocp_table():
    for c in range(16):
        v = oracle.e2m1_value(c)
        want = OCP_E2M1[c & 7]
        assert abs(v) == want
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)


def test_e2m1_code_round_trips_every_code():
    for c in range(16):
        assert oracle.e2m1_code(oracle.e2m1_value(c)) == c


@pytest.mark.parametrize("v,code", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),    # ties: even mantissa
    (0.2499, 0), (0.2501, 1), (2.49, 4), (2.51, 5), (4.99, 6), (5.01, 7),        # either side of a tie
    (6.0, 7), (7.0, 7), (1e30, 7),                                               # saturation
    (-0.75, 10), (-5.0, 14), (-9.0, 15), (-0.1, 8), (0.0, 0),                    # sign bit
])
def test_e2m1_rounding_cases(v, code):
    assert oracle.e2m1_code(v) == code


def test_e2m1_code_is_the_nearest_value_brute_force():
    rng = np.random.default_rng(0)
    for v in rng.uniform(-7, 7, 4000):
        c = oracle.e2m1_code(v)
        d = abs(oracle.e2m1_value(c) - v)
        assert all(d <= abs(m - abs(v)) + 1e-15 for m in OCP_E2M1)


def test_e2m1_quantize_blocks():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 300))
    x[1, 128:256] = 0.0  # an all-zero block
    codes, scales = oracle.e2m1_quantize(x, 128)
    assert codes.shape == (3, 300) and scales.shape == (3, 3)
    for r in range(3):
        for b in range(3):
            blk = x[r, 128 * b:128 * (b + 1)]
            amax = np.abs(blk).max()
            if amax == 0:
                assert scales[r, b] == 1.0 and not codes[r, 128 * b:128 * (b + 1)].any()
                continue
            assert scales[r, b] == amax / 6.0
            i = int(np.abs(blk).argmax())
            assert codes[r, 128 * b + i] & 7 == 7  # the block's largest magnitude maps to 6
            deq = np.array([oracle.e2m1_value(c) for c in codes[r, 128 * b:128 * (b + 1)]]) * scales[r, b]
            # error at most half the spacing around each value: 0.25 below 2, 0.5 below 4, 1 above
            half = np.where(np.abs(blk) / scales[r, b] < 2, 0.25, np.where(np.abs(blk) / scales[r, b] < 4, 0.5, 1.0))
            assert np.all(np.abs(deq - blk) <= half * scales[r, b] * (1 + 1e-12))


def _forward_rope(o, pos, theta, Dn, Dr):
    """RoPE(+t) as a complex multiplication of each pair (x + iy) by e^{i a}."""
    out = o.copy()
    i = np.arange(Dr // 2)
    a = pos * theta ** (-2.0 * i / Dr)
    z = (o[..., Dn::2][..., :Dr // 2] + 1j * o[..., Dn + 1::2][..., :Dr // 2]) * np.exp(1j * a)
    out[..., Dn::2] = z.real
    out[..., Dn + 1::2] = z.imag
    return out


def test_inverse_rope_hand_values():
    # Dn = 2, Dr = 4, theta = 10000, t = 1: pair 0 turns by 1 rad, pair 1 by 0.01 rad
    o = np.array([[7.0, -3.0, 1.0, 0.0, 1.0, 0.0]])
    r = oracle.inverse_rope(o, [1], 10000.0, Dn=2, Dr=4)
    np.testing.assert_allclose(r[0], [7.0, -3.0, math.cos(1.0), -math.sin(1.0), math.cos(0.01), -math.sin(0.01)],
                               rtol=0, atol=1e-15)


def test_inverse_rope_undoes_the_forward_rotation_and_keeps_nope_dims():
    rng = np.random.default_rng(2)
    o = rng.standard_normal((5, 3, 512))
    pos = np.array([0, 1, 77, 131071, 1 << 20])
    fwd = np.stack([_forward_rope(o[i], pos[i], 10000.0, 448, 64) for i in range(5)])
    back = oracle.inverse_rope(fwd, pos, 10000.0)
    np.testing.assert_allclose(back, o, rtol=0, atol=1e-9)
    assert np.array_equal(back[..., :448], o[..., :448])


def test_inverse_rope_position_zero_is_identity_and_rotations_compose():
    rng = np.random.default_rng(3)
    o = rng.standard_normal((1, 512))
    assert np.array_equal(oracle.inverse_rope(o, [0], 10000.0), o)
    two = oracle.inverse_rope(oracle.inverse_rope(o, [300], 5e5), [4000], 5e5)
    once = oracle.inverse_rope(o, [4300], 5e5)
    np.testing.assert_allclose(two, once, rtol=0, atol=1e-9)
    # each pair keeps its length
    pr = lambda a: np.hypot(a[0, 448::2], a[0, 449::2])
    np.testing.assert_allclose(pr(once), pr(o), rtol=1e-13)
