"""Pins for the oracle's number-format decoding (E4M3, BF16)."""
import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_all_codes_match_torch_cast():
    # library special case: torch's float8_e4m3fn -> float64 conversion
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), hex(c)
        else:
            assert got == ref[c] and math.copysign(1, got) == math.copysign(1, ref[c]), hex(c)


def test_e4m3_spec_values():
    spec = json.load(open(os.path.join(GOLDEN, "e4m3_spec_values.json")))
    for code, val in spec["values"].items():
        got = oracle.e4m3_value(int(code, 16))
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    for code in spec["nan_codes"]:
        assert math.isnan(oracle.e4m3_value(int(code, 16)))


def test_bf16_all_codes_match_torch_cast():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
