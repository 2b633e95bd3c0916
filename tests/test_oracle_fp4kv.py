"""Pins of the oracle's FP4 main-KV attention ("DeepSeek V4.1 Flash 建模",
mixed-precision card: E2M1 data, one E4M3 scale per 16 channels, no global
scale): the row decode against the format's value table and torch's E4M3
conversion, the encoder's error bound, dense equivalence against torch's
scaled_dot_product_attention, and agreement with the FP8 path on rows exact
in both formats."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import api as O
from sparse_attention_prefill_gb300 import synth

# OCP MX E2M1 magnitudes for codes 0..7 (sign in bit 3)
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1(code):
    return (-1.0 if code & 8 else 1.0) * E2M1[code & 7]


def _ref_decode(codes, sf):
    """codes uint8 [..., D/2], sf uint8 [..., D/16] -> float64 [..., D]."""
    lo, hi = codes & 15, codes >> 4
    nib = np.stack([lo, hi], -1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    vals = np.vectorize(_e2m1)(nib)
    sc = torch.from_numpy(sf).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * np.repeat(sc, 16, -1)


def _bf16_bits(x):
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b):
    return torch.from_numpy(b.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def test_row_decode_every_code_and_scale():
    rng = np.random.default_rng(0)
    # every E2M1 pair and every finite E4M3 scale code appear
    codes = np.arange(256, dtype=np.uint8)
    sfs = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    for rep in range(4):
        sf = rng.choice(sfs, 32).astype(np.uint8)
        got = O.decode_fp4kv_row(codes, sf)
        assert np.array_equal(got, _ref_decode(codes, sf))


def test_encoder_error_bound():
    x = torch.randn(64, 512)
    codes, sf = synth.encode_fp4kv(x)
    dec = _ref_decode(codes.numpy(), sf.numpy())
    amax = x.abs().reshape(64, 32, 16).amax(-1).repeat_interleave(16, -1).double().numpy()
    # half the widest E2M1 gap (2 between 4 and 6) over the scale amax/6, with
    # the scale itself rounded to E4M3 (relative error <= 2^-4)
    assert (np.abs(dec - x.double().numpy()) <= amax * (1 / 6) * (1 + 2 ** -4) + 1e-12).all()


def _setup(n_entries, t, n_heads, seed):
    torch.manual_seed(seed)
    kv4, sf = synth.encode_fp4kv(torch.randn(n_entries, 512))
    swa_lo = max(0, t - 200)
    swa, swas = synth.encode_fp8_block32(torch.randn(t - swa_lo + 1, 512))
    q = torch.randn(1, n_heads, 512)
    b = dict(num_q=1, num_req=1, ratio=1, q_req=[0], q_pos=[t], kv_start=[0],
             kv_len=[n_entries], swa_start=[0], swa_pos0=[swa_lo], swa_len=[t - swa_lo + 1])
    return b, _bf16_bits(q), kv4.numpy(), sf.numpy(), swa.numpy(), swas.numpy()


def test_dense_equivalence_when_k_covers_all_visible():
    t, n_heads = 60, 4
    b, q, kv4, sf, swa, swas = _setup(64, t, n_heads, 1)
    n_vis = t + 1
    idx = np.arange(512, dtype=np.int32)[None]
    idx[0, n_vis:] = -1
    out, lse, err = O.sparse_swa_attn_fp4kv(b, q, kv4, sf, idx, swa, swas, None, 128)
    assert err == 0
    win = t + 1 - b["swa_pos0"][0]
    fp8 = torch.from_numpy(swa[:win]).view(torch.float8_e4m3fn).to(torch.float64)
    fp8 = (fp8 * torch.from_numpy(swas[:win]).double().repeat_interleave(32, -1)).numpy()
    rows = np.concatenate([_ref_decode(kv4[:n_vis], sf[:n_vis]), fp8])
    qq = torch.from_numpy(_bits_to_f64(q))
    r = torch.from_numpy(rows)[None, None]
    ref = F.scaled_dot_product_attention(qq.transpose(0, 1)[None], r, r,
                                         scale=1 / math.sqrt(512))[0].transpose(0, 1).numpy()
    got = _bits_to_f64(out)
    assert np.abs(got - ref).max() <= 2 ** -8 * np.abs(ref).max()


def test_agrees_with_fp8_path_on_rows_exact_in_both():
    """Rows whose values are E2M1 grid points times a power of two are exact in
    both layouts, so the two oracle entry points must return identical bits."""
    rng = np.random.default_rng(3)
    n, t, n_heads = 40, 39, 4
    nib = rng.integers(0, 16, (n, 512)).astype(np.uint8)
    kv4 = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    sf = np.full((n, 32), 0x38, np.uint8)                   # E4M3 1.0
    vals = _ref_decode(kv4, sf)                             # grid values, |v| <= 6
    kv8 = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    kvs = np.ones((n, 16), np.float32)
    assert np.array_equal(torch.from_numpy(kv8).view(torch.float8_e4m3fn).double().numpy(), vals)
    b, q, _, _, swa, swas = _setup(n, t, n_heads, 4)
    idx = rng.permutation(n).astype(np.int32)[None, :32]
    o8, l8, e8 = O.sparse_swa_attn(b, q, kv8, kvs, idx, swa, swas, None, 128)
    o4, l4, e4 = O.sparse_swa_attn_fp4kv(b, q, kv4, sf, idx, swa, swas, None, 128)
    assert e8 == e4 == 0
    assert np.array_equal(o8, o4) and np.array_equal(l8, l4)
