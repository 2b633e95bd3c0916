"""Pins of the oracle's sparse + sliding-window attention: dense equivalence
against torch's scaled_dot_product_attention in float64, closed forms and
special cases named on the pages."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import api as O
from sparse_attention_prefill_gb300 import synth


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(b.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def _decode_rows(codes, scales):
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
    return (v * torch.from_numpy(scales).double().repeat_interleave(32, -1)).numpy()


def _setup(n_entries, t, n_heads, seed, swa_lo=None):
    torch.manual_seed(seed)
    kv, kvs = synth.encode_fp8_block32(torch.randn(n_entries, 512))
    swa_lo = max(0, t - 200) if swa_lo is None else swa_lo
    swa, swas = synth.encode_fp8_block32(torch.randn(t - swa_lo + 1, 512))
    q = torch.randn(1, n_heads, 512)
    b = dict(num_q=1, num_req=1, ratio=1, q_req=[0], q_pos=[t], kv_start=[0],
             kv_len=[n_entries], swa_start=[0], swa_pos0=[swa_lo], swa_len=[t - swa_lo + 1])
    return b, _bf16_bits(q), kv.numpy(), kvs.numpy(), swa.numpy(), swas.numpy()


def _sdpa(qbits, rows, scale, mask=None):
    q = torch.from_numpy(_bits_to_f64(qbits))                   # [1, H, D]
    r = torch.from_numpy(rows)[None, None]                      # [1, 1, N, D]
    o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], r, r, attn_mask=mask, scale=scale)
    return o[0].transpose(0, 1).numpy()                         # [1, H, D]


def test_dense_equivalence_when_k_covers_all_visible():
    t, n_heads = 60, 4
    b, q, kv, kvs, swa, swas = _setup(64, t, n_heads, 0)
    n_vis = t + 1
    idx = np.arange(512, dtype=np.int32)[None] % 10 ** 9
    idx[0, n_vis:] = -1                                         # K = 512 >= n_vis
    out, lse, err = O.sparse_swa_attn(b, q, kv, kvs, idx, swa, swas, None, 128)
    assert err == 0
    rows = np.concatenate([_decode_rows(kv[:n_vis], kvs[:n_vis]),
                           _decode_rows(swa[:t + 1 - b["swa_pos0"][0]], swas[:t + 1 - b["swa_pos0"][0]])])
    ref = _sdpa(q, rows, 1 / math.sqrt(512))
    want = _bf16_bits(torch.from_numpy(ref))
    got = _bits_to_f64(out)
    # the oracle rounds once from double; allow the reference's own bf16 tie flips
    assert np.abs(got - _bits_to_f64(want)).max() <= 2 ** -8 * np.abs(ref).max()
    lq = torch.from_numpy(_bits_to_f64(q))[0] @ torch.from_numpy(rows).T / math.sqrt(512)
    np.testing.assert_allclose(lse[0], torch.logsumexp(lq, -1).numpy(), rtol=1e-6, atol=1e-6)


def test_window_only_is_sliding_window_attention():
    t, n_heads = 300, 2
    b, q, kv, kvs, swa, swas = _setup(16, t, n_heads, 1, swa_lo=0)
    idx = np.full((1, 8), -1, np.int32)
    out, lse, err = O.sparse_swa_attn(b, q, kv, kvs, idx, swa, swas, None, 128)
    rows = _decode_rows(swa, swas)                              # positions 0..300
    mask = torch.zeros(1, 1, 1, t + 1, dtype=torch.bool)
    mask[..., t - 127:] = True                                  # [t-127, t]
    ref = _sdpa(q, rows, 1 / math.sqrt(512), mask)
    assert np.abs(_bits_to_f64(out) - ref).max() <= 2 ** -8 * np.abs(ref).max()


def test_single_row_and_equal_logits():
    t = 40
    b, q, kv, kvs, swa, swas = _setup(8, t, 3, 2)
    one_row = swa[t - b["swa_pos0"][0]:][:1]
    # win_lo = t: the window is only the row at t (pages: 8064 "reads only itself")
    out, lse, err = O.sparse_swa_attn(b, q, kv, kvs, None, swa, swas, np.array([t]), 128)
    row = _decode_rows(one_row, swas[t - b["swa_pos0"][0]:][:1])[0]
    for h in range(3):
        assert (_bits_to_f64(out[0, h]) == _bits_to_f64(_bf16_bits(torch.from_numpy(row)))).all()
    # a zero query gives equal logits: the output is the mean of the rows
    qz = np.zeros_like(q)
    idx = np.array([[0, 3, 5, -1]], np.int32)
    out, lse, _ = O.sparse_swa_attn(b, qz, kv, kvs, idx, swa, swas, np.array([t - 9]), 128)
    rows = np.concatenate([_decode_rows(kv[[0, 3, 5]], kvs[[0, 3, 5]]),
                           _decode_rows(swa[t - 9 - b["swa_pos0"][0]:], swas[t - 9 - b["swa_pos0"][0]:])])
    mean = rows.mean(0)
    assert np.abs(_bits_to_f64(out[0, 0]) - mean).max() <= 2 ** -8 * np.abs(mean).max()
    assert abs(lse[0, 0] - math.log(13)) < 1e-6


def test_sink_closed_form():
    t = 5
    b, q, kv, kvs, swa, swas = _setup(8, t, 1, 3, swa_lo=0)
    sink = np.array([0.7], np.float32)
    out, lse, _ = O.sparse_swa_attn(b, q, kv, kvs, None, swa, swas, np.array([t]), 128,
                                    sink=sink)
    row = _decode_rows(swa[t:t + 1], swas[t:t + 1])[0]
    ell = float(_bits_to_f64(q)[0, 0] @ row) / math.sqrt(512)
    p = math.exp(ell) / (math.exp(ell) + math.exp(0.7))
    ref = p * row
    assert np.abs(_bits_to_f64(out[0, 0]) - ref).max() <= 2 ** -8 * np.abs(ref).max()
    assert abs(lse[0, 0] - math.log(math.exp(ell) + math.exp(0.7))) < 1e-6


def test_invalid_rows_are_flagged_and_skipped():
    t = 20
    b, q, kv, kvs, swa, swas = _setup(30, t, 2, 4)
    good = np.array([[1, 2, -1, -1]], np.int32)
    bad = np.array([[1, 2, 21, 29]], np.int32)                 # 21, 29 are not visible at t=20
    o1, l1, e1 = O.sparse_swa_attn(b, q, kv, kvs, good, swa, swas, None, 128)
    o2, l2, e2 = O.sparse_swa_attn(b, q, kv, kvs, bad, swa, swas, None, 128)
    assert e1 == 0 and e2 == 1
    assert (o1 == o2).all() and (l1 == l2).all()
    # window reaching below the stored SWA rows
    b2 = dict(b, swa_pos0=[t - 3], swa_len=[4])
    _, _, e3 = O.sparse_swa_attn(b2, q, kv, kvs, good, swa[-4:], swas[-4:], None, 128)
    assert e3 == 2
