"""Pins of the oracle's index scoring (MXFP4 operands, ReLU head-weighted sum,
causal visibility over compressed positions, pool slots)."""
import numpy as np
import pytest
import torch

from oracle import api as O
from sparse_attention_prefill_gb300 import synth

OCP_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0,
                     -4.0, -6.0])


def _dense_decode(codes, scales):
    """Library-style decode: spec table lookup, numpy reshapes."""
    lo = codes & 15
    hi = codes >> 4
    nib = np.stack([lo, hi], -1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    vals = OCP_E2M1[nib]
    return vals * np.repeat(scales.astype(np.float64), 32, axis=-1)


def _batch(nq, q_pos, ratio, kv_len, q_req=None, kv_start=None):
    R = len(kv_len)
    return dict(num_q=nq, num_req=R, ratio=ratio,
                q_req=np.zeros(nq, np.int32) if q_req is None else np.asarray(q_req),
                q_pos=np.asarray(q_pos, np.int64),
                kv_start=np.zeros(R, np.int64) if kv_start is None else np.asarray(kv_start),
                kv_len=np.asarray(kv_len, np.int64), swa_start=np.zeros(R, np.int64),
                swa_pos0=np.zeros(R, np.int64), swa_len=np.zeros(R, np.int64))


def test_nibble_order_and_group_scales():
    # key row: element 1 = 1.0 (high nibble of byte 0), element 33 = 1.0 (group 1)
    k = np.zeros((1, 64), np.uint8)
    k[0, 0] = 0x20
    k[0, 16] = 0x20
    ks = np.array([[1.0, 4.0, 1.0, 1.0]], np.float32)
    # query head: element 0 = 2.0 (low nibble of byte 0), element 1 = 1.0 (high),
    # element 33 = 3.0; group scales 1, 0.5
    q = np.zeros((1, 1, 64), np.uint8)
    q[0, 0, 0] = 0x24
    q[0, 0, 16] = 0x50
    qs = np.array([[[1.0, 0.5, 1.0, 1.0]]], np.float32)
    b = _batch(1, [0], 1, [1])
    s, err = O.index_score(b, q, qs, None, k, ks, ld=1)
    assert err == 0
    # <q,k> = 1.0*1.0*(1*1) + 3.0*1.0*(0.5*4)
    assert s[0, 0] == 1.0 + 6.0


def test_closed_form_all_ones():
    # every element 1.0 (code 2 in both nibbles); head h of query q has scales
    # 2^-(h) in every group, key scales 2^g per group g, weights w_h
    hi = 4
    q = np.full((1, hi, 64), 0x22, np.uint8)
    qs = np.array([[[2.0 ** -h] * 4 for h in range(hi)]], np.float32)
    k = np.full((3, 64), 0x22, np.uint8)
    ks = np.array([[2.0 ** g for g in range(4)]] * 3, np.float32)
    w = np.array([[1.0, -2.0, 0.5, 3.0]], np.float32)
    b = _batch(1, [2], 1, [3])
    s, err = O.index_score(b, q, qs, w, k, ks, ld=3)
    dot = [32 * sum(2.0 ** g for g in range(4)) * 2.0 ** -h for h in range(hi)]
    want = sum(w[0, h] * dot[h] for h in range(hi))
    assert err == 0 and (s[0] == np.float32(want)).all()


def test_relu_drops_negative_heads():
    q = np.zeros((1, 2, 64), np.uint8)
    q[0, 0, 0] = 0x02          # head 0: +1.0 at element 0
    q[0, 1, 0] = 0x0A          # head 1: -1.0 at element 0
    qs = np.ones((1, 2, 4), np.float32)
    k = np.zeros((1, 64), np.uint8)
    k[0, 0] = 0x04             # key: 2.0 at element 0
    ks = np.ones((1, 4), np.float32)
    b = _batch(1, [0], 1, [1])
    s, _ = O.index_score(b, q, qs, np.array([[1.0, 5.0]], np.float32), k, ks, ld=1)
    assert s[0, 0] == 2.0      # head 1's dot is -2 -> ReLU -> 0
    s, _ = O.index_score(b, q, qs, np.array([[-1.5, 5.0]], np.float32), k, ks, ld=1)
    assert s[0, 0] == -3.0     # negative weight on a positive head stays negative


@pytest.mark.parametrize("ratio", [1, 2])
def test_brute_force_random_with_visibility(ratio):
    torch.manual_seed(0)
    R, hi, per_req = 2, 3, 13
    entries = [per_req, per_req - 4]
    kv_start = [0, per_req]
    qk, qs = synth.encode_mxfp4(torch.randn(7, hi, 128))
    kk, ks = synth.encode_mxfp4(torch.randn(sum(entries), 128))
    w = (torch.randn(7, hi) / 2).numpy()
    q_req = np.array([0, 0, 0, 1, 1, 1, 0], np.int32)
    q_pos = np.array([0, 1, 2 * per_req // ratio - 1, 3, 4, 17 // ratio, 5], np.int64)
    b = _batch(7, q_pos, ratio, entries, q_req, kv_start)
    ld = per_req
    s, err = O.index_score(b, qk.numpy(), qs.numpy(), w, kk.numpy(), ks.numpy(), ld)
    Qd = _dense_decode(qk.numpy(), qs.numpy())          # [nq, hi, 128]
    Kd = _dense_decode(kk.numpy(), ks.numpy())          # [N, 128]
    dots = np.einsum("qhd,nd->qhn", Qd, Kd)
    full = np.einsum("qh,qhn->qn", w.astype(np.float64), np.maximum(dots, 0.0))
    over = False
    for q in range(7):
        r = q_req[q]
        nv = (q_pos[q] + 1) // ratio           # entries whose last token is <= t
        if nv > entries[r]:
            over = True
            nv = entries[r]
        want = full[q, kv_start[r]:kv_start[r] + nv]
        np.testing.assert_allclose(s[q, :nv], want, rtol=1e-6, atol=1e-6)
        assert np.isnan(s[q, nv:]).all()      # columns past the row are not written
    assert bool(err & 4) == over


def test_pool_slots_map_to_entries():
    torch.manual_seed(1)
    hi, n = 2, 40
    qk, qs = synth.encode_mxfp4(torch.randn(2, hi, 128))
    kk, ks = synth.encode_mxfp4(torch.randn(n, 128))
    b = _batch(2, [37, 20], 1, [n])
    full, _ = O.index_score(b, qk.numpy(), qs.numpy(), None, kk.numpy(), ks.numpy(), ld=n)
    blocks = np.array([[0, 2, 4, -1], [1, 2, -1, -1]], np.int32)
    pool, err = O.index_score(b, qk.numpy(), qs.numpy(), None, kk.numpy(), ks.numpy(), ld=32,
                              cand_blocks=blocks, block=8)
    assert err == 0
    for q in range(2):
        nv = [38, 21][q]
        nb = int((blocks[q] >= 0).sum())
        for slot in range(nb * 8):
            e = blocks[q, slot // 8] * 8 + slot % 8
            if e < nv:
                assert pool[q, slot] == full[q, e]
            else:
                assert pool[q, slot] == -np.inf
        assert np.isnan(pool[q, nb * 8:]).all()


def test_mxfp4_row_decode_order_and_scales():
    """Element 2i in the low nibble of byte i, one scale per 32 elements (the
    layout a quantiser writes; dot products alone cannot see the nibble order)."""
    codes = np.zeros(64, np.uint8)
    codes[0] = 0x21        # element 0 = 0.5 (code 1), element 1 = 1.0 (code 2)
    codes[17] = 0xF7       # element 34 = 6.0 (code 7), element 35 = -6.0 (code 15)
    scales = np.array([2.0, 0.25, 1.0, 1.0], np.float32)
    row = O.decode_mxfp4_row(codes, scales)
    expect = np.zeros(128)
    expect[0], expect[1] = 1.0, 2.0
    expect[34], expect[35] = 1.5, -1.5
    assert (row == expect).all()
    # round trip through the oracle's own quantiser
    x = np.linspace(-3, 3, 128).astype(np.float32)[None, :]
    c, s, err = O.encode_rows(O.FMT_MXFP4, x, np.array([0]), np.zeros((1, 64), np.uint8),
                              np.zeros((1, 4), np.float32))
    assert err == 0
    y = O.decode_mxfp4_row(c[0], s[0])
    # E2M1's widest gap is 2 units (between 4 and 6): at most 1 unit x scale off
    assert np.abs(y - x[0]).max() <= s.max()
