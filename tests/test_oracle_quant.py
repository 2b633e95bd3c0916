"""Pins of the oracle's quantise-and-write (cache rows in the three storage
formats of the "DeepSeek V4.1 Flash 建模" mixed-precision card), against an
independent float8 implementation, closed forms per binade and round trips.

Reading pinned here: the group scale is an fp32 value (amax / 448 for FP8
block-32; E4M3(amax / 6) for the FP4 main-KV layout; 2^(floor(log2 amax) - 2)
for MXFP4), x / scale is taken in fp32, and the element rounds to nearest,
ties to even, saturating at the largest finite value.
"""
import numpy as np
import pytest
import torch

from oracle import api as O


def _e4m3_table():
    return np.array([O.e4m3_value(c) for c in range(127)])


def test_e4m3_encode_matches_torch_float8():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.normal(0, s, 2000) for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    t = _e4m3_table()
    mids = (t[:-1] + t[1:]) / 2                       # every tie between neighbours
    vals = np.concatenate([vals, t, -t, mids, -mids, [0.0, -0.0]])
    vals = vals[np.abs(vals) <= 448.0].astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.encode_e4m3(float(v)) for v in vals], np.uint8)
    assert (got == ref).all(), vals[got != ref][:5]


def test_e4m3_saturates():
    for v in (448.0, 449.0, 464.0, 1e9, np.inf):
        assert O.encode_e4m3(v) == 0x7E
        assert O.encode_e4m3(-v) == 0xFE


def _e2m1_by_binade(x):
    """E2M1 rounding written per binade: step 0.5 below 2, 1 in [2, 4), 2 in
    [4, 6], ties to even steps (numpy rounds half to even), saturating at 6."""
    a = min(abs(x), 6.0)
    if a < 2.0:
        m = np.round(a * 2.0) / 2.0
    elif a < 4.0:
        m = np.round(a)
    else:
        m = np.round(a / 2.0) * 2.0
    return -m if np.signbit(x) else m


def test_e2m1_encode_per_binade():
    rng = np.random.default_rng(1)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    mids = (grid[:-1] + grid[1:]) / 2
    vals = np.concatenate([rng.uniform(-7, 7, 3000), grid, -grid, mids, -mids, [6.5, 100.0]])
    for v in vals:
        c = O.encode_e2m1(float(v))
        assert O.e2m1_value(c) == _e2m1_by_binade(float(v)), (v, c)
    assert O.encode_e2m1(-0.1) == 0x8            # rounds to zero, keeps the sign


def _decode_rows(fmt, codes, scales, dim):
    n = codes.shape[0]
    out = np.zeros((n, dim))
    for r in range(n):
        for d in range(dim):
            if fmt == O.FMT_FP8_B32:
                out[r, d] = O.e4m3_value(int(codes[r, d])) * scales[r, d // 32]
            else:
                b = int(codes[r, d // 2])
                nib = (b >> 4) if d & 1 else (b & 15)
                s = O.e4m3_value(int(scales[r, d // 16])) if fmt == O.FMT_FP4KV \
                    else scales[r, d // 32]
                out[r, d] = O.e2m1_value(nib) * s
    return out


@pytest.mark.parametrize("fmt,dim", [(O.FMT_FP8_B32, 512), (O.FMT_FP4KV, 512), (O.FMT_MXFP4, 128)])
def test_encode_rows_round_trip_and_scales(fmt, dim):
    rng = np.random.default_rng(fmt)
    n = 6
    x = (rng.normal(0, 1, (n, dim)) * rng.choice([1e-3, 1.0, 50.0], (n, 1))).astype(np.float32)
    x[2, :32] = 0.0                                    # an all-zero group
    cw = dim if fmt == O.FMT_FP8_B32 else dim // 2
    sw, st = (dim // 16, np.uint8) if fmt == O.FMT_FP4KV else (dim // 32, np.float32)
    codes, scales, err = O.encode_rows(fmt, x, np.arange(n), np.zeros((n, cw), np.uint8),
                                       np.zeros((n, sw), st))
    assert err == 0
    y = _decode_rows(fmt, codes, scales, dim)
    gs = 16 if fmt == O.FMT_FP4KV else 32
    for r in range(n):
        for g in range(dim // gs):
            xs = x[r, g * gs:(g + 1) * gs].astype(np.float64)
            amax = np.abs(xs).max()
            if fmt == O.FMT_FP8_B32:
                s = np.float32(amax) / np.float32(448.0) if amax > 0 else 1.0
                assert scales[r, g] == np.float32(s)
                # half a step of the coarsest E4M3 binade below 448 (32), scaled
                assert np.abs(y[r, g * gs:(g + 1) * gs] - xs).max() <= 16 * s + 1e-30
            elif fmt == O.FMT_MXFP4:
                s = 2.0 ** (np.floor(np.log2(amax)) - 2) if amax > 0 else 1.0
                assert scales[r, g] == s
                # half a step below 6*s, saturation above (amax/s < 8)
                assert np.abs(y[r, g * gs:(g + 1) * gs] - xs).max() <= \
                    max(1.0 * s, amax - 6 * s) + 1e-30
            else:
                s = O.e4m3_value(int(scales[r, g]))
                assert int(scales[r, g]) == O.encode_e4m3(float(np.float32(amax) / np.float32(6)))
                if s > 0:
                    # below 6*s: half a step (1*s); above: saturation at 6*s
                    err_max = np.abs(y[r, g * gs:(g + 1) * gs] - xs).max()
                    assert err_max <= max(1.0 * s, amax - 6 * s) + 1e-30
    assert (y[2, :32] == 0).all()


def test_encode_rows_exact_values_and_flags():
    # values on the grids come back exactly
    x = np.zeros((3, 512), np.float32)
    t = _e4m3_table()
    x[0, :32] = np.concatenate([[448.0], t[:31]]).astype(np.float32)   # amax 448: scale 1
    x[1, :] = np.nan
    x[2, :] = 1.0
    codes, scales, err = O.encode_rows(O.FMT_FP8_B32, x, np.array([2, 0, 9]),
                                       np.full((4, 512), 0x55, np.uint8),
                                       np.full((4, 16), -1.0, np.float32))
    assert err == 256 | 512                     # row 9 past 4 rows; the NaN row
    assert scales[2, 0] == 1.0 and codes[2, 0] == 0x7E
    assert [O.e4m3_value(int(c)) for c in codes[2, 1:32]] == list(t[:31])
    assert (codes[0] == 0).all() and (scales[0] == 1.0).all()      # the NaN row, zeroed
    assert (codes[1] == 0x55).all() and (codes[3] == 0x55).all()   # rows not written
    # negative destination rows are skipped without a flag
    _, _, err = O.encode_rows(O.FMT_FP8_B32, x[2:], np.array([-1]), codes, scales)
    assert err == 0
