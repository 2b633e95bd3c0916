"""Pins of the oracle's index-key projection from the compressed main KV
("DeepSeek V4.1 Flash 建模", CSA2 card, compressor paragraph; SGLang/Miles
day-0 article sec. 5: BF16 weights, FP32 accumulation), followed by the MXFP4
cache write: against numpy's float64 matrix product of the decoded bf16
values, a channel-selection closed form, power-of-two homogeneity of the
MXFP4 recipe, a hand-worked group, and the row-skip / range flags."""
import numpy as np
import torch

from oracle import api as O

ERR_RANGE_ROW = 256


def _bf16(a):
    """float array -> (bf16 bit patterns uint16, their exact values float64)."""
    t = torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16), t.double().numpy()


def _dst(n, rows=None):
    rows = rows or n
    codes = np.zeros((rows, 64), np.uint8)
    scales = np.zeros((rows, 4), np.float32)
    return np.arange(n, dtype=np.int64), codes, scales


def test_projection_equals_float64_matmul_of_the_bf16_values():
    rng = np.random.default_rng(0)
    xb, xv = _bf16(rng.standard_normal((37, 512)))
    wb, wv = _bf16(rng.standard_normal((128, 512)) / np.sqrt(512))
    dst, c0, s0 = _dst(37)
    codes, scales, y, err = O.index_k_project(xb, wb, dst, c0, s0)
    assert err == 0
    want = (xv @ wv.T).astype(np.float32)     # exact sums (narrow exponent range) rounded once
    assert np.array_equal(y, want)
    # the cache rows are exactly the MXFP4 encoding of y
    c2, s2, err2 = O.encode_rows(3, y, dst, c0, s0)
    assert err2 == 0 and np.array_equal(codes, c2) and np.array_equal(scales, s2)


def test_channel_selection_gives_the_input_columns():
    rng = np.random.default_rng(1)
    xb, xv = _bf16(rng.standard_normal((9, 512)))
    perm = rng.permutation(512)[:128]
    w = np.zeros((128, 512))
    w[np.arange(128), perm] = 1.0
    wb, _ = _bf16(w)
    dst, c0, s0 = _dst(9)
    codes, scales, y, err = O.index_k_project(xb, wb, dst, c0, s0)
    assert err == 0 and np.array_equal(y, xv[:, perm].astype(np.float32))


def test_power_of_two_weights_scale_outputs_and_mxfp4_scales_only():
    rng = np.random.default_rng(2)
    xb, _ = _bf16(rng.standard_normal((11, 512)))
    w = rng.standard_normal((128, 512)) / 16
    wb1, _ = _bf16(w)
    wb2, _ = _bf16(w * 8.0)
    dst, c0, s0 = _dst(11)
    c1, s1, y1, _ = O.index_k_project(xb, wb1, dst, c0, s0)
    c2, s2, y2, _ = O.index_k_project(xb, wb2, dst, c0, s0)
    assert np.array_equal(y2, y1 * 8.0)
    assert np.array_equal(c1, c2) and np.array_equal(s2, s1 * 8.0)


def test_hand_worked_group():
    """x = e_0 (one-hot), so y[o] = w[o][0]: group 0 holds 6, 3, -1.5, 0.5 and
    zeros: amax 6 -> scale 2^(floor(log2 6) - 2) = 1; E2M1 codes 7, 5, 8|3,
    1, 0 ...; element 2i in the low nibble of byte i."""
    x = np.zeros((1, 512))
    x[0, 0] = 1.0
    xb, _ = _bf16(x)
    w = np.zeros((128, 512))
    w[0:4, 0] = [6.0, 3.0, -1.5, 0.5]
    w[32, 0] = 0.75     # group 1: amax 0.75 -> scale 2^-3, 0.75 / 2^-3 = 6 -> code 7
    wb, _ = _bf16(w)
    dst, c0, s0 = _dst(1)
    codes, scales, y, err = O.index_k_project(xb, wb, dst, c0, s0)
    assert err == 0
    assert codes[0, 0] == (7 | (5 << 4)) and codes[0, 1] == (11 | (1 << 4))
    assert (codes[0, 2:16] == 0).all()
    assert scales[0, 0] == 1.0 and scales[0, 1] == 2.0 ** -3 and codes[0, 16] == 7
    assert scales[0, 2] == 1.0 and scales[0, 3] == 1.0      # all-zero groups


def test_skipped_and_out_of_range_rows():
    rng = np.random.default_rng(3)
    xb, _ = _bf16(rng.standard_normal((3, 512)))
    wb, _ = _bf16(rng.standard_normal((128, 512)) / 32)
    codes = np.full((2, 64), 0x5A, np.uint8)
    scales = np.full((2, 4), 7.0, np.float32)
    dst = np.array([-1, 5, 1], np.int64)
    c, s, y, err = O.index_k_project(xb, wb, dst, codes, scales)
    assert err == ERR_RANGE_ROW
    assert (c[0] == 0x5A).all() and (s[0] == 7.0).all()       # untouched
    c_ref, s_ref, _ = O.encode_rows(3, y[2:3], np.array([1]), codes, scales)
    assert np.array_equal(c[1], c_ref[1]) and np.array_equal(s[1], s_ref[1])
