"""GPU parity of the quantise-and-write of cache rows (csa2_quantize_rows),
bit-exact against the oracle, and the encoder-replay write protocol.

"DeepSeek V4.1 Flash 建模", mixed-precision card (the three storage formats)
and Encoder Bounded Replay card (replayed tokens rewrite SWA only; the cached
global KV is read, never rewritten); SGLang/Miles day-0 article sec. 5 (a
fused quantise-and-write keeps the unfused rounding sequence).
"""
import numpy as np
import pytest
import torch

import sparse_attention_prefill_gb300 as S
from oracle import api as O
from tests.helpers import npy

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _shapes(fmt, rows, dim):
    if fmt == S.FMT_FP8_B32:
        return (rows, dim), np.uint8, (rows, dim // 32), np.float32
    if fmt == S.FMT_FP4KV:
        return (rows, dim // 2), np.uint8, (rows, dim // 16), np.uint8
    return (rows, dim // 2), np.uint8, (rows, dim // 32), np.float32


def _run(fmt, x, dst, rows, fill=0x5A):
    n, dim = x.shape
    cs, ct, ss, stp = _shapes(fmt, rows, dim)
    codes0 = np.full(cs, fill, ct)
    scales0 = np.full(ss, 7, stp) if stp == np.uint8 else np.full(ss, -3.0, stp)
    d_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    codes = torch.from_numpy(codes0).to(DEV)
    scales = torch.from_numpy(scales0).to(DEV)
    S.quantize_rows(fmt, torch.from_numpy(x).to(DEV), torch.from_numpy(dst).to(DEV), codes,
                    scales, d_err)
    torch.cuda.synchronize()
    rc, rs, rerr = O.encode_rows(fmt, x, dst, codes0, scales0)
    return npy(codes), npy(scales), int(d_err.item()), rc, rs, rerr


@pytest.mark.parametrize("fmt,dim", [(S.FMT_FP8_B32, 512), (S.FMT_FP4KV, 512),
                                     (S.FMT_MXFP4, 128), (S.FMT_FP8_B32, 96),
                                     (S.FMT_FP4KV, 1040), (S.FMT_MXFP4, 1536),
                                     (S.FMT_MXFP4, 64), (S.FMT_FP8_B32, 32), (S.FMT_FP4KV, 16)])
def test_quantize_rows_bit_exact(fmt, dim):
    rng = np.random.default_rng(fmt * 1000 + dim)
    n = 300
    mag = rng.choice([1e-40, 1e-30, 1e-6, 1e-2, 1.0, 3e2, 1e30], (n, 1))
    x = (rng.normal(0, 1, (n, dim)) * mag).astype(np.float32)
    x[5, :40] = 0.0
    x[6, :] = -0.0
    x[7, 3] = np.nan
    x[8, 100 % dim] = np.inf
    # exact ties of the element grids after scaling (amax pins the scale)
    x[9, :8] = np.array([448, 0.75, 1.25, 2.5, 3.5, 5.0, -0.25, -1.75], np.float32)
    x[10, :16] = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -5, -3.5, -2.5,
                           -1.75, -1.25, -0.75, -0.25, 7], np.float32)
    dst = rng.permutation(n + 20)[:n].astype(np.int64)
    dst[11] = -1
    dst[12] = n + 50                 # past the cache rows
    g_c, g_s, g_e, r_c, r_s, r_e = _run(fmt, x, dst, n + 20)
    assert g_e == r_e
    assert (g_c == r_c).all(), np.argwhere(g_c != r_c)[:5]
    assert (g_s.view(np.uint8) == r_s.view(np.uint8)).all(), np.argwhere(g_s != r_s)[:5]


def test_encoder_replay_write_protocol():
    """Rows of an encoder replay: every processed row rewrites its SWA row;
    global entries are written only in [entry_range); the cached ones keep
    their bytes."""
    p = np.array([300, 61, 0], np.int64)
    e = np.array([40, 20, 10], np.int32)
    lay, err = O.encoder_replay_layout(p, e, 128, 2)
    assert err == 0
    dim = 512
    rng = np.random.default_rng(7)
    # SWA cache: one row per position 0 .. S_r - 1 of each request
    seq = p + e
    swa_start = np.concatenate([[0], np.cumsum(seq)[:-1]])
    swa_dst = (swa_start[lay["row_req"]] + lay["pos"]).astype(np.int64)
    xs = rng.normal(0, 1, (len(swa_dst), dim)).astype(np.float32)
    # global pool: floor(S_r / 2) entries per request; new entries only
    ents = seq // 2
    kv_start = np.concatenate([[0], np.cumsum(ents)[:-1]])
    g_dst = np.concatenate([kv_start[r] + np.arange(*lay["entry_range"][r])
                            for r in range(len(p))]).astype(np.int64)
    xg = rng.normal(0, 1, (len(g_dst), dim)).astype(np.float32)
    for dst, x, rows in ((swa_dst, xs, int(seq.sum())), (g_dst, xg, int(ents.sum()))):
        g_c, g_s, g_e, r_c, r_s, r_e = _run(S.FMT_FP8_B32, x, dst, rows, fill=0x33)
        assert g_e == r_e == 0
        assert (g_c == r_c).all() and (g_s == r_s).all()
        untouched = np.setdiff1d(np.arange(rows), dst)
        assert (g_c[untouched] == 0x33).all()
    # the cached entries (below each request's range) are among the untouched rows
    cached = np.concatenate([kv_start[r] + np.arange(lay["entry_range"][r][0])
                             for r in range(len(p))])
    assert len(np.intersect1d(cached, g_dst)) == 0 and len(cached) == 150 + 30
