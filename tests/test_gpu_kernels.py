"""GPU parity of each C-ABI entry point against the oracle on seeded inputs
that span several tiles with ragged tails, plus edge cases."""
import numpy as np
import pytest
import torch

import sparse_attention_prefill_gb300 as S
from oracle import api as O
from sparse_attention_prefill_gb300 import synth
from tests.helpers import (assert_attn_close, np_batch, npy, topk_near_tie_ok, topk_sets_match)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _to(w_batch, dev=DEV):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in w_batch.items()}


def _derr():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


# ---------------------------------------------------------------------------
# a1 tail layout: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(3))
def test_tail_layout_random_batches(seed):
    g = torch.Generator().manual_seed(seed)
    r = [1, 7, 1500, 3000][seed]
    e = torch.randint(0, 400, (r,), generator=g, dtype=torch.int32)
    e[torch.rand(r, generator=g) < 0.2] = 128
    s = e.to(torch.int64) + torch.randint(0, 10 ** 6, (r,), generator=g)
    ref, rerr = O.tail_layout(e.numpy(), s.numpy(), 128)
    d_err = _derr()
    got = S.tail_layout(e.to(DEV), s.to(DEV), 128, d_err=d_err)
    n = int(ref["cu_tail"][-1])
    for k in ("tail_len", "cu_tail"):
        assert (npy(got[k]) == ref[k]).all(), k
    for k in ("src_row", "pos", "win_lo", "row_req"):
        assert (npy(got[k])[:n] == ref[k]).all(), k
    assert int(d_err.item()) == rerr


def test_tail_layout_pages_examples_and_flags():
    e = torch.tensor([8192, 64, 8192, 8192, 8192, 8192, 0, 1], dtype=torch.int32)
    s = torch.tensor([8192, 8256, 8192, 16384, 24576, 32768, 5, 1], dtype=torch.int64)
    got = S.tail_layout(e.to(DEV), s.to(DEV), 128)
    pos = npy(got["pos"])
    cu = npy(got["cu_tail"])
    assert pos[cu[0]] == 8064 and pos[cu[1] - 1] == 8191
    assert pos[cu[1]] == 8192 and pos[cu[2] - 1] == 8255 and npy(got["win_lo"])[cu[1]] == 8192
    assert [int(pos[cu[i]]) for i in range(2, 6)] == [8064, 16256, 24448, 32640]
    assert npy(got["tail_len"]).tolist() == [128, 64, 128, 128, 128, 128, 0, 1]
    # bad extends and a short capacity raise data-error bits, never fault
    d_err = _derr()
    e2 = torch.tensor([5, -1, 300], dtype=torch.int32, device=DEV)
    s2 = torch.tensor([3, 10, 300], dtype=torch.int64, device=DEV)
    tl = torch.empty(3, dtype=torch.int32, device=DEV)
    cu2 = torch.empty(4, dtype=torch.int32, device=DEV)
    buf32 = torch.empty(100, dtype=torch.int32, device=DEV)
    buf64 = torch.empty(100, dtype=torch.int64, device=DEV)
    buf64b = torch.empty(100, dtype=torch.int64, device=DEV)
    st = S.csa2_tail_layout(3, e2, s2, 128, tl, cu2, buf32, buf64, buf64b, None, 100, d_err)
    torch.cuda.synchronize()
    assert st == 0 and int(d_err.item()) == (S.DERR_BAD_EXTEND | S.DERR_CAPACITY)
    assert npy(tl).tolist() == [0, 0, 128]


# ---------------------------------------------------------------------------
# a2-a4, a7 index scores
# ---------------------------------------------------------------------------

def _score_tol(b, wl, layer, ref, cand=None):
    """|d| <= 1e-5 * sum_h |w_h| relu(dot_h): the oracle with |w| gives the bound."""
    L = wl.layers[layer]
    absw = None if L.head_w is None else L.head_w.abs()
    bound, _ = O.index_score(b, npy(L.q_fp4), npy(L.q_scale), npy(absw), npy(wl.pool.k_fp4),
                             npy(wl.pool.k_scale), ref.shape[1], cand_blocks=cand,
                             block=wl.block)
    return 1e-5 * np.nan_to_num(np.abs(bound), nan=0.0, posinf=0.0) + 1e-30


@pytest.mark.parametrize("ratio,hi", [(2, 8), (1, 32), (2, 64), (1, 16)])
def test_index_score_full_mode(ratio, hi):
    ctx = 2 * 1500 + 7
    qpos = [0, 1, 2, 5, 300, 301, 1499, 2999, 3000, ctx - 1, 2 * 128 * ratio - 1, 2 * 128 * ratio]
    w = synth.full_layer(ctx, ratio, qpos, 16, hi, seed=11, tag="iscore%d" % hi)
    b = w.batch("full")
    L = w.layers["full"]
    ref, rerr = O.index_score(np_batch(b), npy(L.q_fp4), npy(L.q_scale), npy(L.head_w),
                              npy(w.pool.k_fp4), npy(w.pool.k_scale), w.ld)
    d_err = _derr()
    got = torch.full((w.num_q, w.ld), float("nan"), device=DEV)
    S.index_score(_to(b), L.q_fp4.to(DEV), L.q_scale.to(DEV), L.head_w.to(DEV),
                  w.pool.k_fp4.to(DEV), w.pool.k_scale.to(DEV), w.ld, scores=got, d_err=d_err)
    g = npy(got)
    tol = _score_tol(np_batch(b), w, "full", ref)
    written = ~np.isnan(ref)
    assert (np.isnan(g) == ~written).all()          # exactly the visible columns written
    assert (np.abs(g[written] - ref[written]) <= tol[written]).all()
    assert int(d_err.item()) == rerr


@pytest.mark.parametrize("ctx", [16384, 16385])
def test_index_score_chunk_sizes(ctx):
    """Rows at the key-tile chunk boundaries: a CTA covers 128 key tiles when
    the longest row fits them (16384 entries) and 64 otherwise (16385); rows of
    8192/8193 and 16384/16385 entries end at or just past a chunk."""
    qpos = [8191, 8192, 8193, 16383, ctx - 1, 100]
    w = synth.full_layer(ctx, 1, qpos, 16, 32, seed=13, tag="ichunk%d" % ctx)
    b = w.batch("full")
    L = w.layers["full"]
    ref, rerr = O.index_score(np_batch(b), npy(L.q_fp4), npy(L.q_scale), npy(L.head_w),
                              npy(w.pool.k_fp4), npy(w.pool.k_scale), w.ld)
    d_err = _derr()
    got = torch.full((w.num_q, w.ld), float("nan"), device=DEV)
    S.index_score(_to(b), L.q_fp4.to(DEV), L.q_scale.to(DEV), L.head_w.to(DEV),
                  w.pool.k_fp4.to(DEV), w.pool.k_scale.to(DEV), w.ld, scores=got, d_err=d_err)
    g = npy(got)
    tol = _score_tol(np_batch(b), w, "full", ref)
    written = ~np.isnan(ref)
    assert (np.isnan(g) == ~written).all()
    assert (np.abs(g[written] - ref[written]) <= tol[written]).all()
    assert int(d_err.item()) == rerr


@pytest.mark.parametrize("hi", [32, 16, 8])
def test_index_score_pool_mode_and_ctx_flag(hi):
    # hi = 32 keeps a CTA's candidate blocks in shared memory; 16 and 8 (more
    # queries per tile) read them from global memory
    ctx = 5000
    qpos = [4999, 4000, 17, 2048, 2049]
    w = synth.full_layer(ctx, 1, qpos, 16, hi, seed=5, tag="ipool%d" % hi)
    b = w.batch("full")
    L = w.layers["full"]
    g = torch.Generator().manual_seed(3)
    nb = [100, 37, 3, 256, 1]
    cand = np.full((5, 300), -1, np.int32)
    for q in range(5):
        n_blocks_vis = (qpos[q] + 1 + 7) // 8
        pick = torch.randperm(n_blocks_vis + 2, generator=g)[:nb[q]].sort().values
        cand[q, :nb[q]] = pick.numpy()
    ref, rerr = O.index_score(np_batch(b), npy(L.q_fp4), npy(L.q_scale), npy(L.head_w),
                              npy(w.pool.k_fp4), npy(w.pool.k_scale), 2400, cand_blocks=cand)
    got = torch.full((5, 2400), float("nan"), device=DEV)
    d_err = _derr()
    S.index_score(_to(b), L.q_fp4.to(DEV), L.q_scale.to(DEV), L.head_w.to(DEV),
                  w.pool.k_fp4.to(DEV), w.pool.k_scale.to(DEV), 2400,
                  cand_blocks=torch.from_numpy(cand).to(DEV), scores=got, d_err=d_err)
    gg = npy(got)
    tol = _score_tol(np_batch(b), w, "full", ref, cand)
    same_nan = np.isnan(gg) == np.isnan(ref)
    assert same_nan.all()
    fin = np.isfinite(ref)
    assert (np.isinf(gg) == np.isinf(ref)).all()
    assert (np.abs(gg[fin] - ref[fin]) <= tol[fin]).all()
    assert int(d_err.item()) == rerr
    # a query whose visible count exceeds the stored entries raises RANGE_CTX
    b2 = dict(b, kv_len=torch.tensor([1000], dtype=torch.int64))
    d_err2 = _derr()
    S.index_score(_to(b2), L.q_fp4.to(DEV), L.q_scale.to(DEV), L.head_w.to(DEV),
                  w.pool.k_fp4.to(DEV), w.pool.k_scale.to(DEV), w.ld, d_err=d_err2)
    torch.cuda.synchronize()
    assert int(d_err2.item()) & S.DERR_RANGE_CTX


# ---------------------------------------------------------------------------
# a5-a7 selection: bit-exact on identical score input
# ---------------------------------------------------------------------------

def _sel_batch(q_pos, kv_len, ratio=1):
    nq = len(q_pos)
    return dict(num_q=nq, num_req=1, ratio=ratio, q_req=torch.zeros(nq, dtype=torch.int32),
                q_pos=torch.tensor(q_pos, dtype=torch.int64),
                kv_start=torch.zeros(1, dtype=torch.int64),
                kv_len=torch.tensor([kv_len], dtype=torch.int64),
                swa_start=torch.zeros(1, dtype=torch.int64), swa_pos0=torch.zeros(1, dtype=torch.int64),
                swa_len=torch.zeros(1, dtype=torch.int64))


@pytest.mark.parametrize("n,k", [(700, 512), (50000, 512), (200000, 2048), (3000, 1), (20000, 37),
                                 # row strides that are not a multiple of four scores: the
                                 # listing sweep's 16-byte loads start past a scalar head
                                 (5003, 512), (9001, 100), (20001, 512), (50001, 2048)])
def test_topk_full_mode_bit_exact(n, k):
    rng = np.random.default_rng(n + k)
    q_pos = sorted(set([n - 1, n // 2, k - 1, k, k + 1, 0, 7, n - 2]))
    s = (np.round(rng.standard_normal((len(q_pos), n)) * 64) / 64).astype(np.float32)
    s[rng.random(s.shape) < 0.01] = np.nan
    s[rng.random(s.shape) < 0.01] = -np.inf
    s[rng.random(s.shape) < 0.001] = np.inf
    b = _sel_batch(q_pos, n)
    ref_idx, ref_cnt, _ = O.topk(np_batch(b), s, k)
    idx, cnt = S.topk(_to(b), torch.from_numpy(s).to(DEV), k)
    topk_sets_match(idx, cnt, ref_idx, ref_cnt)


@pytest.mark.parametrize("n,k", [(1024, 512), (2048, 512), (4000, 512), (8192, 512), (16384, 512),
                                 (16384, 2048), (6000, 1)])
def test_topk_special_rows_bit_exact(n, k):
    """Rows of every register-path size with degenerate contents: all keys
    equal, ties straddling the k-th key, fewer than k eligible entries, one
    eligible entry, dense coarse-grid scores, -0/+0 (equal scores, so entry
    order decides) at the k-th key, and rows that defeat the threshold guess."""
    rng = np.random.default_rng(7 * n + k)
    q_pos = [n - 1] * 7 + [k - 1, n // 3, n - 1, n - 1, n - 1]
    s = (np.round(rng.standard_normal((len(q_pos), n)) * 4) / 4).astype(np.float32)
    s[0, :] = 1.5                                         # all equal
    s[1, :] = np.where(rng.random(n) < 0.5, 2.0, -1.0)    # two values
    s[2, :] = np.nan
    s[2, rng.choice(n, min(n, k // 2 + 1), replace=False)] = 3.0  # few eligible, tied
    s[3, :] = -np.inf
    s[3, n // 2] = 0.0                                    # one eligible
    s[4, :] = rng.standard_normal(n).astype(np.float32)   # continuous
    s[5, :] = -np.abs(s[5, :]) - 1e-3                     # negative keys only
    s[6, :] = np.float32(1e-40)                           # subnormal, all equal
    s[9, :] = np.where(rng.random(n) < 0.5, np.float32(-0.0), np.float32(0.0))
    s[9, rng.choice(n, k // 2, replace=False)] = 1.0      # -0 and +0 tie at the k-th key
    # rows whose moments mislead a normal-quantile threshold guess: a few far
    # outliers inflate the deviation (too few keys listed), or a tight cluster
    # sits just above a long left tail (too many)
    s[10, :] = (rng.standard_normal(n) * 0.01).astype(np.float32)
    s[10, rng.choice(n, max(1, n // 64), replace=False)] = 100.0
    s[11, :] = (5.0 + rng.standard_normal(n) * 1e-3).astype(np.float32)
    s[11, rng.choice(n, max(1, n // 5), replace=False)] = -1000.0
    b = _sel_batch(q_pos, n)
    ref_idx, ref_cnt, _ = O.topk(np_batch(b), s, k)
    idx, cnt = S.topk(_to(b), torch.from_numpy(s).to(DEV), k)
    topk_sets_match(idx, cnt, ref_idx, ref_cnt)


def test_topk_pool_mode_bit_exact():
    rng = np.random.default_rng(9)
    q_pos = [16383, 9000, 100, 16390]
    nbv = [(p + 1 + 7) // 8 for p in q_pos]
    cand = np.full((4, 2048), -1, np.int32)
    for q in range(4):
        m = min(2048, nbv[q] + 1)
        cand[q, :m] = np.sort(rng.choice(nbv[q] + 1, m, replace=False))
    s = (np.round(rng.standard_normal((4, 16384)) * 16) / 16).astype(np.float32)
    b = _sel_batch(q_pos, 20000)
    ref_idx, ref_cnt, _ = O.topk(np_batch(b), s, 512, cand_blocks=cand)
    idx, cnt = S.topk(_to(b), torch.from_numpy(s).to(DEV), 512,
                      cand_blocks=torch.from_numpy(cand).to(DEV))
    topk_sets_match(idx, cnt, ref_idx, ref_cnt)


@pytest.mark.parametrize("n_vis_list,bsz,nb_max", [
    ([16383, 16384, 16385, 16393, 131072, 130561, 9, 1, 0], 8, 2048),
    ([23, 22, 9, 8, 7, 3], 2, 4),
    ([50000, 400001], 8, 4096),
    # one- and two-block budgets: only the latest block, or it and the best
    # other block (rows longer than the 4096-block ranking buffer included)
    ([40000, 33000, 17, 9, 8, 1, 0], 8, 1),
    ([40000, 33000, 17, 9, 8, 1, 0], 8, 2),
])
def test_candidates_bit_exact(n_vis_list, bsz, nb_max):
    rng = np.random.default_rng(len(n_vis_list) + bsz)
    n = max(max(n_vis_list), 1)
    q_pos = [v - 1 for v in n_vis_list]
    s = (np.round(rng.standard_normal((len(q_pos), n)) * 8) / 8).astype(np.float32)
    b = _sel_batch(q_pos, n)
    ref = O.topk_candidates(np_batch(b), s, k=512, block=bsz, max_blocks=nb_max)
    idx, cnt, blocks, nblocks = S.topk_candidates(_to(b), torch.from_numpy(s).to(DEV), 512,
                                                  block=bsz, max_blocks=nb_max)
    topk_sets_match(idx, cnt, ref[0], ref[1])
    assert (npy(nblocks) == ref[3]).all()
    assert (npy(blocks) == ref[2]).all()


# ---------------------------------------------------------------------------
# a8-a10 attention
# ---------------------------------------------------------------------------

def _attn_case(n_heads, k, nq=9, ctx=3000, seed=0, win=None, sink=False, bad_idx=False):
    qpos = list(range(ctx - nq, ctx))
    w = synth.full_layer(ctx, 1, qpos, n_heads, 8, seed=seed, tag="attn%d" % n_heads,
                         tail_win_lo=win)
    b = w.batch("full")
    L = w.layers["full"]
    g = torch.Generator().manual_seed(seed)
    idx = torch.full((nq, max(k, 1)), -1, dtype=torch.int32)
    for q in range(nq):
        nv = qpos[q] + 1
        take = min(k, nv) - (q % 3 == 1) * 5           # some rows not full
        if take > 0:
            idx[q, :take] = torch.randperm(nv, generator=g)[:take].to(torch.int32)
    if bad_idx:
        idx[0, 0] = ctx + 5
        idx[1, 3] = qpos[1] + 1
    sk = torch.randn(n_heads, generator=g) if sink else None
    return w, b, L, idx[:, :k] if k else None, sk


@pytest.mark.parametrize("n_heads,k", [(64, 512), (16, 512), (32, 300), (64, 0), (64, 2048)])
def test_attention_parity(n_heads, k):
    w, b, L, idx, sk = _attn_case(n_heads, k, seed=n_heads + k)
    ref_o, ref_l, rerr = O.sparse_swa_attn(np_batch(b), npy(L.q), npy(w.pool.kv_fp8),
                                           npy(w.pool.kv_scale), npy(idx), npy(L.swa_fp8),
                                           npy(L.swa_scale), None, 128, w.sm_scale)
    d_err = _derr()
    o, l = S.sparse_swa_attn(_to(b), L.q.to(DEV), w.pool.kv_fp8.to(DEV), w.pool.kv_scale.to(DEV),
                             None if idx is None else idx.to(DEV), L.swa_fp8.to(DEV),
                             L.swa_scale.to(DEV), None, 128, w.sm_scale, d_err=d_err)
    assert_attn_close(o, l, ref_o, ref_l)
    assert int(d_err.item()) == rerr == 0


def test_attention_tail_window_sink_and_bad_indices():
    w, b, L, idx, sk = _attn_case(64, 512, nq=12, ctx=2500, seed=4, win=2495, sink=True,
                                  bad_idx=True)
    wl = L.win_lo
    ref_o, ref_l, rerr = O.sparse_swa_attn(np_batch(b), npy(L.q), npy(w.pool.kv_fp8),
                                           npy(w.pool.kv_scale), npy(idx), npy(L.swa_fp8),
                                           npy(L.swa_scale), npy(wl), 128, w.sm_scale,
                                           sink=npy(sk))
    d_err = _derr()
    o, l = S.sparse_swa_attn(_to(b), L.q.to(DEV), w.pool.kv_fp8.to(DEV), w.pool.kv_scale.to(DEV),
                             idx.to(DEV), L.swa_fp8.to(DEV), L.swa_scale.to(DEV), wl.to(DEV), 128,
                             w.sm_scale, sink=sk.to(DEV), d_err=d_err)
    assert_attn_close(o, l, ref_o, ref_l)
    assert rerr == S.DERR_RANGE_IDX and int(d_err.item()) == rerr


def test_attention_window_outside_swa_rows_and_empty_rows():
    w, b, L, idx, sk = _attn_case(16, 64, nq=4, ctx=600, seed=8)
    b2 = dict(b, swa_pos0=b["swa_pos0"] + 50, swa_len=b["swa_len"] - 50)
    ref_o, ref_l, rerr = O.sparse_swa_attn(np_batch(b2), npy(L.q), npy(w.pool.kv_fp8),
                                           npy(w.pool.kv_scale), npy(idx), npy(L.swa_fp8),
                                           npy(L.swa_scale), None, 128, w.sm_scale)
    d_err = _derr()
    o, l = S.sparse_swa_attn(_to(b2), L.q.to(DEV), w.pool.kv_fp8.to(DEV), w.pool.kv_scale.to(DEV),
                             idx.to(DEV), L.swa_fp8.to(DEV), L.swa_scale.to(DEV), None, 128,
                             w.sm_scale, d_err=d_err)
    assert_attn_close(o, l, ref_o, ref_l)
    assert rerr & S.DERR_RANGE_WINDOW and int(d_err.item()) == rerr
    # a query with no row at all: out = 0, lse = -inf
    b3 = dict(b, swa_len=torch.zeros_like(b["swa_len"]))
    none_idx = torch.full_like(idx, -1).to(DEV)
    o3, l3 = S.sparse_swa_attn(_to(b3), L.q.to(DEV), w.pool.kv_fp8.to(DEV),
                               w.pool.kv_scale.to(DEV), none_idx, L.swa_fp8.to(DEV),
                               L.swa_scale.to(DEV), None, 128, w.sm_scale)
    assert (o3.float() == 0).all() and torch.isneginf(l3).all()


def test_host_argument_checks():
    b = _sel_batch([5], 10)
    s = torch.zeros((1, 10), device=DEV)
    idx = torch.empty((1, 4), dtype=torch.int32, device=DEV)
    cnt = torch.empty(1, dtype=torch.int32, device=DEV)
    assert S.csa2_topk(_to(b), s, 10, 4096, None, 8, 2048, idx, cnt, None) == S.ERR_UNSUPPORTED
    assert S.csa2_topk(_to(b), s, 10, 0, None, 8, 2048, idx, cnt, None) == S.ERR_INVALID_ARG
    bb = dict(_to(b), ratio=3)
    assert S.csa2_topk(bb, s, 10, 4, None, 8, 2048, idx, cnt, None) == S.ERR_INVALID_ARG


def test_attention_reference_moves_mid_query():
    """Window rows 64 times larger than the selected rows: their logits jump
    far past the reference set by the first chunks, so the softmax moves the
    per-head reference in a later chunk and rescales the O accumulator and
    the row sums already gathered."""
    w, b, L, idx, sk = _attn_case(64, 512, nq=9, ctx=3000, seed=21)
    swa_scale = (L.swa_scale * 64.0).contiguous()
    ref_o, ref_l, rerr = O.sparse_swa_attn(np_batch(b), npy(L.q), npy(w.pool.kv_fp8),
                                           npy(w.pool.kv_scale), npy(idx), npy(L.swa_fp8),
                                           npy(swa_scale), None, 128, w.sm_scale)
    d_err = _derr()
    o, l = S.sparse_swa_attn(_to(b), L.q.to(DEV), w.pool.kv_fp8.to(DEV), w.pool.kv_scale.to(DEV),
                             idx.to(DEV), L.swa_fp8.to(DEV), swa_scale.to(DEV), None, 128,
                             w.sm_scale, d_err=d_err)
    assert int(d_err.item()) == rerr == 0
    assert_attn_close(o, None, ref_o, None)
    # lse: its error is at most the largest logit error, and a logit errs by at
    # most sm_scale * 2^-10 * sum_d |q_d r_d| (f16 rows: the f16 scale and the
    # f16 product each round once).  The logits here are ~64x the unit-variance
    # ones, and so is that bound.
    tab = np.array([O.e4m3_value(c) for c in range(256)])
    rows_of = lambda codes, sc: tab[codes.astype(np.int64)] * np.repeat(   # noqa: E731
        sc.astype(np.float64), 32, axis=1)
    kv = rows_of(npy(w.pool.kv_fp8), npy(w.pool.kv_scale))
    sw = rows_of(npy(L.swa_fp8), npy(swa_scale))
    nb = np_batch(b)
    q = L.q.float().numpy().astype(np.float64)
    bound = np.zeros(ref_l.shape)
    for i in range(ref_l.shape[0]):
        t, r = int(nb["q_pos"][i]), int(nb["q_req"][i])
        rows = [kv[int(nb["kv_start"][r]) + int(j)] for j in npy(idx)[i] if j >= 0]
        rows += [sw[int(nb["swa_start"][r]) + p - int(nb["swa_pos0"][r])]
                 for p in range(max(0, t - 127), t + 1)]
        bound[i] = w.sm_scale * 2.0 ** -10 * (np.abs(q[i]) @ np.abs(np.stack(rows)).T).max(1)
    d = np.abs(npy(l).astype(np.float64) - ref_l)
    assert (d <= bound + 1e-5 * np.abs(ref_l)).all(), (d.max(), bound.min())
