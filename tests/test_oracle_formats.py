"""Pins of the oracle's storage-format decoders and bf16 rounding against the
published format tables and library routines."""
import numpy as np
import torch

from oracle import api as O

# OCP Microscaling Formats (MX) v1.0, E2M1 element: the eight magnitudes the
# spec lists for codes 0..7 (sign bit is bit 3).
OCP_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_all_codes_match_spec_table():
    for code in range(16):
        mag = OCP_E2M1[code & 7]
        want = -mag if code & 8 else mag
        assert O.e2m1_value(code) == want


def test_e4m3_all_codes_match_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = O.e4m3_value(c)
        if np.isnan(ref[c]):
            assert np.isnan(got), c
        else:
            assert got == ref[c], (c, got, ref[c])
    # the format's landmarks: max normal 448, min subnormal 2^-9, NaN only at S.1111.111
    assert O.e4m3_value(0x7E) == 448.0 and O.e4m3_value(0x01) == 2.0 ** -9
    assert sum(np.isnan(O.e4m3_value(c)) for c in range(256)) == 2


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                         [0.0, -0.0, 1.0, 3.0e38, -1e-40, 1.00390625, 1.01171875]])
    for x in xs:
        want = torch.tensor(float(np.float32(x)), dtype=torch.float32).to(torch.bfloat16)
        want = int(want.view(torch.int16).item()) & 0xFFFF
        assert O.double_to_bf16(float(x)) == want, x


def test_n_visible_boundaries():
    # m = 2: entry j (tokens 2j, 2j+1) becomes visible at t = 2j + 1
    for j in range(6):
        assert O.n_visible(2 * j, 2) == j
        assert O.n_visible(2 * j + 1, 2) == j + 1
    # m = 1: entry j visible once j <= t
    for t in range(6):
        assert O.n_visible(t, 1) == t + 1
