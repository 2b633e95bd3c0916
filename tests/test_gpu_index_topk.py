"""The index score streamed into the top-K (csa2_index_topk) against the
unstreamed path on the same inputs (csa2_index_score + csa2_topk: the same
tensor-core scores, so the sets must be equal exactly) and against the oracle
(index score and top-K, sets equal except swaps among near-ties of the k-th
score).  Rows short enough to list everything, rows that take the threshold,
and rows built to defeat the threshold guess (which must go through the exact
fallback) are all covered."""
import numpy as np
import pytest
import torch

import sparse_attention_prefill_gb300 as S
from oracle import api as O
from sparse_attention_prefill_gb300 import synth
from tests.helpers import np_batch, npy, topk_near_tie_ok, topk_sets_match

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _derr():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _run(w, k, max_len=None):
    """(streamed idx, count, fallback rows), (dense idx, count), oracle (idx,
    count, scores)."""
    b, L = w.batch("full"), w.layers["full"]
    max_len = max_len or w.ld
    need = S.csa2_index_topk_workspace(w.num_q, max_len)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device=DEV)   # contents must not matter
    d0 = _derr()
    si, sc = S.index_topk(b, L.q_fp4, L.q_scale, L.head_w, w.pool.k_fp4, w.pool.k_scale, max_len,
                          k, workspace=ws, d_err=d0)
    torch.cuda.synchronize()
    # white-box: the first word of the workspace counts the rows the fallback took
    n_fb = int(ws[:4].view(torch.int32).item())
    d1 = _derr()
    s = S.index_score(b, L.q_fp4, L.q_scale, L.head_w, w.pool.k_fp4, w.pool.k_scale, max_len,
                      d_err=d1)
    di, dc = S.topk(b, s, k, d_err=d1)
    torch.cuda.synchronize()
    assert int(d0.item()) == int(d1.item())
    nb = np_batch(b)
    rs, _ = O.index_score(nb, npy(L.q_fp4), npy(L.q_scale), npy(L.head_w), npy(w.pool.k_fp4),
                          npy(w.pool.k_scale), max_len)
    ri, rc, _ = O.topk(nb, np.nan_to_num(rs, nan=-np.inf), k)
    return (si, sc, n_fb), (di, dc), (ri, rc, rs), int(d0.item())


def _check(w, k, expect_fallback=None, max_len=None):
    (si, sc, n_fb), (di, dc), (ri, rc, rs), derr = _run(w, k, max_len)
    topk_sets_match(si, sc, npy(di), npy(dc))
    ties = topk_near_tie_ok(si, sc, ri, rc, rs)
    if expect_fallback is not None:
        assert (n_fb > 0) == expect_fallback, n_fb
    print("index_topk: %d rows, k %d, fallback rows %d, near-tie rows vs oracle %d"
          % (w.num_q, k, n_fb, len(ties)))
    return n_fb, derr


@pytest.mark.parametrize("hi,k", [(8, 512), (16, 100), (32, 512), (64, 2048)])
def test_short_rows_list_everything(hi, k):
    """At most 4096 visible entries: every entry is listed, no threshold."""
    qpos = [0, 1, 5, 511, 512, 513, 2000, 2999, 4095] + list(range(3000, 4096, 97))
    w = synth.full_layer(4096, 1, qpos, 16, hi, seed=hi + k, device=DEV, tag="streamshort")
    n_fb, _ = _check(w, k, expect_fallback=False)


@pytest.mark.parametrize("ratio,hi,k", [(2, 32, 512), (1, 32, 512), (2, 64, 2048), (1, 16, 300)])
def test_long_rows_take_the_threshold(ratio, hi, k):
    """Rows of 4097 .. 20000 visible entries (C3-like at m = 2): the sample
    pass, the threshold, the appending scoring pass and the list selection."""
    ctx = 40000 if ratio == 2 else 20000
    g = torch.Generator().manual_seed(ratio * 100 + hi)
    qpos = sorted(set((torch.randint(8194 * ratio, ctx, (40,), generator=g)).tolist() +
                      [8192 * ratio, ctx - 1]))
    w = synth.full_layer(ctx, ratio, qpos, 16, hi, seed=ratio + hi + k, device=DEV,
                         tag="streamlong")
    _check(w, k)


def _defeat(kind):
    """A workload whose sampled key tiles (every 8th tile of 128 entries)
    mislead the threshold: all keys equal (every score tied), sampled tiles
    scaled down (too many listed) or up (too few listed)."""
    qpos = [9000, 12000, 15555, 19999]
    w = synth.full_layer(20000, 1, qpos, 16, 32, seed=7, device=DEV, tag="streamdefeat")
    p = w.pool
    j = torch.arange(p.k_scale.shape[0], device=DEV)
    sampled = ((j // 128) % 8 == 0)[:, None]
    if kind == "tied":
        p.k_fp4.fill_(0x22)           # every element 1.0
        p.k_scale.fill_(1.0)
    elif kind == "sample_low":
        p.k_scale.copy_(torch.where(sampled, p.k_scale * 2.0 ** -6, p.k_scale))
    else:
        p.k_scale.copy_(torch.where(sampled, p.k_scale * 2.0 ** 3, p.k_scale))
    return w


@pytest.mark.parametrize("kind", ["tied", "sample_low", "sample_high"])
def test_rows_that_defeat_the_guess_take_the_exact_fallback(kind):
    w = _defeat(kind)
    n_fb, derr = _check(w, 512, expect_fallback=True)
    assert derr == 0


def test_rows_longer_than_max_len_are_cut_and_flagged():
    qpos = [3000, 9000, 9999]
    w = synth.full_layer(10000, 1, qpos, 16, 32, seed=3, device=DEV, tag="streamcut")
    _, derr = _check(w, 512, max_len=6000)
    assert derr & S.DERR_LD


def test_workspace_too_small_is_rejected():
    w = synth.full_layer(5000, 1, [4999], 16, 32, seed=4, device=DEV, tag="streamws")
    b, L = w.batch("full"), w.layers["full"]
    need = S.csa2_index_topk_workspace(1, w.ld)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    idx = torch.empty((1, 512), dtype=torch.int32, device=DEV)
    cnt = torch.empty(1, dtype=torch.int32, device=DEV)
    st = S.csa2_index_topk(b, 32, 128, L.q_fp4, L.q_scale, L.head_w, w.pool.k_fp4,
                           w.pool.k_scale, w.ld, 512, idx, cnt, ws, ws.numel(), None)
    assert st == S.ERR_INVALID_ARG
