"""GPU parity on the five named workloads at full size.

The GPU runs every query row of each workload through the layer call sequence
(the same launches bench.py times).  The oracle runs its own chain on a seeded
sample of rows, from the same inputs, and the two are compared:
  * tail layout: bit-exact;
  * index scores: |d| <= 1e-5 * sum_h |w_h| relu(dot_h) per element;
  * top-K / candidate blocks: bit-exact when the GPU selects from the oracle's
    fp32 scores; end to end, sets equal except swaps among near-ties
    (within 1e-3 relative of the k-th score);
  * attention: with the oracle's indices as input, max|d|/max|r| <= 2e-2 and
    mean|d|/mean|r| <= 1e-3 per layer; lse within 1e-4.
"""
import numpy as np
import pytest
import torch

import sparse_attention_prefill_gb300 as S
from oracle import api as O
from sparse_attention_prefill_gb300 import synth
from sparse_attention_prefill_gb300.layer import LayerRunner
from tests.helpers import (assert_attn_close, np_batch, npy, pool_near_tie_rows, topk_near_tie_ok,
                           topk_sets_match)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _sub(b, rows):
    """Oracle batch restricted to rows (host arrays)."""
    nb = np_batch(b)
    r = rows.cpu().numpy()
    nb["q_req"] = nb["q_req"][r]
    nb["q_pos"] = nb["q_pos"][r]
    nb["num_q"] = len(r)
    return nb


def _lt(w, layer, attr, rows):
    t = getattr(w.layers[layer], attr)
    return None if t is None else npy(t[rows])


def _oracle_scores(w, layer, b, rows, ld, cand=None):
    s, err = O.index_score(b, _lt(w, layer, "q_fp4", rows), _lt(w, layer, "q_scale", rows),
                           _lt(w, layer, "head_w", rows), npy(w.pool.k_fp4),
                           npy(w.pool.k_scale), ld, cand_blocks=cand, block=w.block)
    hw = w.layers[layer].head_w
    bound, _ = O.index_score(b, _lt(w, layer, "q_fp4", rows), _lt(w, layer, "q_scale", rows),
                             None if hw is None else npy(hw[rows].abs()), npy(w.pool.k_fp4),
                             npy(w.pool.k_scale), ld, cand_blocks=cand, block=w.block)
    return s, 1e-5 * np.nan_to_num(np.abs(bound), nan=0.0, posinf=0.0) + 1e-30, err


def _check_scores(gpu_scores, rows, ref, tol):
    g = npy(gpu_scores[rows])[:, :ref.shape[1]]
    written = ~np.isnan(ref)
    fin = np.isfinite(ref)
    assert (np.isneginf(g[written]) == np.isneginf(ref[written])).all()
    assert (np.abs(g[fin] - ref[fin]) <= tol[fin]).all(), np.abs(g[fin] - ref[fin]).max()


def _gpu_select_on(ref_scores, batch_dev_rows, w, cand=None, candidates=False):
    s = torch.from_numpy(np.nan_to_num(ref_scores, nan=-np.inf)).to(DEV)
    if candidates:
        return S.topk_candidates(batch_dev_rows, s, w.topk, w.block, w.max_blocks)
    return S.topk(batch_dev_rows, s, w.topk, cand_blocks=None if cand is None else
                  torch.from_numpy(cand).to(DEV), block=w.block)


def _gpu_attend_on(w, layer, batch_dev_rows, rows, ref_idx, win_lo=None):
    L = w.layers[layer]
    return S.sparse_swa_attn(batch_dev_rows, L.q[rows].contiguous(), w.pool.kv_fp8,
                             w.pool.kv_scale, torch.from_numpy(ref_idx).to(DEV), L.swa_fp8,
                             L.swa_scale, None if win_lo is None else win_lo, w.window,
                             w.sm_scale)


def _oracle_attend(w, layer, b, rows, idx, win_lo=None):
    L = w.layers[layer]
    return O.sparse_swa_attn(b, _lt(w, layer, "q", rows), npy(w.pool.kv_fp8),
                             npy(w.pool.kv_scale), idx, npy(L.swa_fp8), npy(L.swa_scale),
                             None if win_lo is None else npy(win_lo), w.window, w.sm_scale)


def _dev_batch(b, rows):
    d = dict(b)
    d["q_req"] = b["q_req"][rows].contiguous()
    d["q_pos"] = b["q_pos"][rows].contiguous()
    d["num_q"] = int(rows.numel())
    return d


def _layer_parity(w, runner, layer, rows, mode, pool=None, given_idx=None, win_lo=None,
                  chain_idx=None, justified=(), label=None):
    """Compare one layer of the GPU chain with the oracle chain on `rows`.

    `pool` is the ORACLE's candidate pool for these rows (pool-restricted
    Reindex).  `justified` lists the positions (in `rows`) whose inputs to
    this layer already differ from the oracle's for a reason an earlier check
    accepted: a candidate pool that differs only by near-ties of block maxima,
    or a selection that differs only by near-tie swaps.  Every other row must
    match end to end.  Returns (oracle indices, oracle blocks of a source
    layer, the positions whose outputs may differ downstream: the pool's
    near-tie rows for a source layer, else the rows whose selection may)."""
    b_dev = runner.batches[layer]
    b_or = _sub(b_dev, rows)
    bd_rows = _dev_batch(b_dev, rows)
    wl = None if win_lo is None else win_lo[rows].contiguous()
    just = set(int(q) for q in justified)
    ref_idx, ref_blocks = given_idx, None
    sel_ok = set(just)          # rows whose chain selection may differ from the oracle's
    downstream = set(just)
    n_pool_ties = n_sel_ties = 0
    if mode in ("full", "source", "reindex"):
        keep = np.array([q not in just for q in range(len(rows))], bool)
        if pool is not None:
            # rows in `just` scored a different (near-tie) pool: they are held
            # to the rule that accepted that pool, not compared score by score
            ld = runner.pool_scores.shape[1]
            ref_s, tol, oerr = _oracle_scores(w, layer, b_or, rows, ld, cand=pool)
            assert oerr & 16 == 0     # no row longer than the stride (the LD flag)
            kt = torch.from_numpy(np.nonzero(keep)[0]).to(DEV)
            _check_scores(runner.pool_scores[rows][kt], torch.arange(len(kt), device=DEV),
                          ref_s[keep], tol[keep])
        else:
            assert not just
            ld = runner.scores.shape[1]
            ref_s, tol, _ = _oracle_scores(w, layer, b_or, rows, ld)
            _check_scores(runner.scores, rows, ref_s, tol)
        # selection: bit-exact on the oracle's fp32 scores
        if mode == "source":
            ri, rc, rb, rn, _ = O.topk_candidates(b_or, np.nan_to_num(ref_s, nan=-np.inf),
                                                  w.topk, w.block, w.max_blocks)
            gi, gc, gb, gn = _gpu_select_on(ref_s, bd_rows, w, candidates=True)
            assert (npy(gb) == rb).all() and (npy(gn) == rn).all()
            ref_blocks = rb
            # the chain's own pool: bit-exact, near-ties of block maxima excepted
            pool_rows = pool_near_tie_rows(runner.blocks[rows], runner.nblocks[rows], rb, rn,
                                           ref_s, w.block)
            n_pool_ties = len(pool_rows)
            downstream = set(pool_rows)
        else:
            ri, rc, _ = O.topk(b_or, np.nan_to_num(ref_s, nan=-np.inf), w.topk,
                               cand_blocks=pool, block=w.block)
            gi, gc = _gpu_select_on(ref_s, bd_rows, w, cand=pool)
        topk_sets_match(gi, gc, ri, rc)
        ref_idx = ri
        # end to end: the chain's own selection, near-ties allowed
        k_rows = np.nonzero(keep)[0]
        sel = torch.from_numpy(k_rows).to(DEV)
        c_idx = runner.idx[layer][rows][sel]
        c_cnt = runner.count[layer][rows][sel]
        entry_of_col = None
        if pool is not None:
            entry_of_col = [{int(pool[q, c // w.block]) * w.block + c % w.block: c
                             for c in range(int((pool[q] >= 0).sum()) * w.block)} for q in k_rows]
        tie_rows = topk_near_tie_ok(c_idx, c_cnt, ri[k_rows], rc[k_rows], ref_s[k_rows],
                                    entry_of_col)
        n_sel_ties = len(tie_rows)
        sel_ok |= set(int(k_rows[t]) for t in tie_rows)
        if mode != "source":
            downstream = set(sel_ok)
    # attention on the oracle's indices
    ro, rl, _ = _oracle_attend(w, layer, b_or, rows, ref_idx, wl)
    go, gl = _gpu_attend_on(w, layer, bd_rows, rows, ref_idx, wl)
    assert_attn_close(go, gl, ro, rl)
    # end to end: every row whose chain indices equal the oracle's; a row may
    # differ only if a check above (or upstream) accepted the difference
    if mode != "reuse":
        chain = npy(runner.idx[layer][rows])
    else:   # the indices the GPU chain actually used (its own earlier layer)
        chain = npy(chain_idx[rows]) if chain_idx is not None else np.asarray(given_idx)
    same = np.array([sorted(chain[q].tolist()) == sorted(ref_idx[q].tolist())
                     for q in range(len(rows))])
    differ = set(np.nonzero(~same)[0].tolist())
    assert differ <= sel_ok, sorted(differ - sel_ok)[:10]
    sel = np.nonzero(same)[0]
    if len(sel):
        st = torch.from_numpy(sel).to(DEV)
        assert_attn_close(runner.out[layer][rows][st], runner.lse[layer][rows][st], ro[sel],
                          rl[sel])
    print("%s %s: %d rows; pool near-tie rows %d; selection near-tie rows %d; "
          "rows with upstream differences %d; end-to-end attention compared on %d rows"
          % (label or "", layer, len(rows), n_pool_ties, n_sel_ties, len(just), len(sel)))
    return ref_idx, ref_blocks, sorted(downstream)


@pytest.fixture(scope="module")
def seed():
    return 0


def test_c1_tiny_full(seed):
    w = synth.config("c1_tiny_full", DEV, seed)
    run = LayerRunner(w)
    run.full_layer("full")
    torch.cuda.synchronize()
    rows = torch.arange(w.num_q, device=DEV)
    ref_idx, _, tie_rows = _layer_parity(w, run, "full", rows, "full", label="C1")
    assert int(run.d_err.item()) == 0
    # the bounded-window variant of the same layer (tail lower bound 3968)
    win = torch.full((w.num_q,), 3968, dtype=torch.int64, device=DEV)
    run.attend("full", run.idx["full"], win)
    _layer_parity(w, run, "full", rows, "reuse", given_idx=ref_idx, win_lo=win,
                  chain_idx=run.idx["full"], justified=tie_rows, label="C1 bounded")


def test_c2_decoder_replay(seed):
    w = synth.config("c2_decoder_replay", DEV, seed)
    run = LayerRunner(w)
    run.decoder_tail_step()
    torch.cuda.synchronize()
    assert int(run.d_err.item()) == 0
    tail, terr = O.tail_layout(npy(w.extend_len), npy(w.seq_len), w.replay)
    n = int(tail["cu_tail"][-1])
    assert terr == 0 and n == w.num_q
    for k in ("pos", "win_lo", "src_row", "row_req"):
        assert (npy(run.tail[k])[:n] == tail[k]).all(), k
    assert (tail["pos"] == npy(w.q_pos)).all()
    rows = torch.arange(w.num_q, device=DEV)
    win = run.tail_win_lo
    _, blocks, pool_rows = _layer_parity(w, run, "L20", rows, "source", label="C2")
    idx21, _, just21 = _layer_parity(w, run, "L21", rows, "reindex", pool=blocks, win_lo=win,
                                     justified=pool_rows, label="C2")
    _layer_parity(w, run, "L22", rows, "reuse", given_idx=idx21, win_lo=win,
                  chain_idx=run.idx["L21"], justified=just21, label="C2")


def test_c3_encoder_prefill(seed):
    w = synth.config("c3_encoder_prefill", DEV, seed)
    run = LayerRunner(w)
    run.full_layer("full")
    torch.cuda.synchronize()
    assert int(run.d_err.item()) == 0
    g = torch.Generator().manual_seed(seed)
    rows = torch.arange(0, w.num_q, 64) + torch.randint(0, 64, (w.num_q // 64,), generator=g)
    rows = torch.cat([rows, torch.tensor([0, 1, 2, 1023, 1024, w.num_q - 1])]).unique().to(DEV)
    _layer_parity(w, run, "full", rows, "full", label="C3")


def test_c4_hierarchical(seed):
    w = synth.config("c4_hierarchical", DEV, seed)
    run = LayerRunner(w)
    blocks = run.source_layer("L20")
    run.reindex_layer("L21", blocks)
    torch.cuda.synchronize()
    assert int(run.d_err.item()) == 0
    nb = npy(run.nblocks)
    assert (nb == 2048).all()
    last = (npy(w.q_pos) + 1 + 7) // 8 - 1
    assert (npy(run.blocks)[np.arange(w.num_q), 2047] == last).all()   # latest block kept
    # every one of the 512 query rows, in both layers
    rows = torch.arange(w.num_q, device=DEV)
    _, ref_blocks, pool_rows = _layer_parity(w, run, "L20", rows, "source", label="C4")
    _layer_parity(w, run, "L21", rows, "reindex", pool=ref_blocks, justified=pool_rows,
                  label="C4")


def test_c5_ragged_mixed(seed):
    w = synth.config("c5_ragged_mixed", DEV, seed)
    req = w.q_req.cpu()
    reindex = torch.nonzero(req % 2 == 0).flatten()
    reuse = torch.nonzero(req % 2 == 1).flatten()
    run_ri = LayerRunner(w, reindex.to(DEV))
    run_ru = LayerRunner(w, reuse.to(DEV))
    run_ri.reindex_layer("mixed", None)
    given = w.layers["mixed"].given_idx[reuse.to(DEV)].contiguous()
    run_ru.reuse_layer("mixed", given)
    torch.cuda.synchronize()
    assert int(run_ri.d_err.item()) == 0 and int(run_ru.d_err.item()) == 0
    # every extend row (16 extends x 64 rows) and 64 seeded decode rows of each mode
    n_dec = 256
    g = torch.Generator().manual_seed(seed)
    ri_list, ru_list = reindex.tolist(), reuse.tolist()
    dec_ri = [i for i, r in enumerate(ri_list) if r < n_dec]
    dec_ru = [i for i, r in enumerate(ru_list) if r < n_dec]
    pick_ri = sorted(dec_ri[j] for j in torch.randperm(len(dec_ri), generator=g)[:64].tolist()) + \
        [i for i, r in enumerate(ri_list) if r >= n_dec]
    pick_ru = sorted(dec_ru[j] for j in torch.randperm(len(dec_ru), generator=g)[:64].tolist()) + \
        [i for i, r in enumerate(ru_list) if r >= n_dec]
    assert len(pick_ri) + len(pick_ru) == 128 + 16 * 64
    wl_all = w.layers["mixed"].win_lo
    wri = wl_all[reindex.to(DEV)].contiguous()
    wru = wl_all[reuse.to(DEV)].contiguous()
    # parity helpers index layer tensors by absolute row; map runner rows back
    _layer_parity_rows(w, run_ri, reindex, pick_ri, "reindex", wri)
    _layer_parity_rows(w, run_ru, reuse, pick_ru, "reuse", wru,
                       given=npy(w.layers["mixed"].given_idx[reuse[pick_ru].to(DEV)]))


def _layer_parity_rows(w, runner, abs_rows, pick, mode, win_lo, given=None):
    """Parity for a runner built on a row subset: `pick` indexes the subset.
    Reindex rows: scores, selection bit-exact on the oracle's scores, the
    chain's selection with near-ties only, and the chain's attention output on
    every row whose selection equals the oracle's.  Reuse rows: the chain's
    output on the given indices."""
    pick_t = torch.tensor(pick, device=DEV)
    abs_pick = abs_rows.to(DEV)[pick_t]
    layer = "mixed"
    b_or = _sub(w.batch(layer), abs_pick)
    bd_rows = _dev_batch(w.batch(layer), abs_pick)
    wl = win_lo[pick_t].contiguous()
    if mode == "reindex":
        ld = runner.scores.shape[1]
        ref_s, tol, _ = _oracle_scores(w, layer, b_or, abs_pick, ld)
        _check_scores(runner.scores, pick_t, ref_s, tol)
        ri, rc, _ = O.topk(b_or, np.nan_to_num(ref_s, nan=-np.inf), w.topk)
        gi, gc = _gpu_select_on(ref_s, bd_rows, w)
        topk_sets_match(gi, gc, ri, rc)
        tie_rows = set(topk_near_tie_ok(runner.idx[layer][pick_t], runner.count[layer][pick_t],
                                        ri, rc, ref_s))
        idx = ri
    else:
        idx = given
        tie_rows = set()
    ro, rl, _ = _oracle_attend(w, layer, b_or, abs_pick, idx, wl)
    go, gl = _gpu_attend_on(w, layer, bd_rows, abs_pick, idx, wl)
    assert_attn_close(go, gl, ro, rl)
    chain = npy(runner.idx[layer][pick_t]) if mode == "reindex" else np.asarray(given)
    same = np.array([sorted(chain[q].tolist()) == sorted(idx[q].tolist())
                     for q in range(len(pick))])
    differ = set(np.nonzero(~same)[0].tolist())
    assert differ <= tie_rows, sorted(differ - tie_rows)[:10]
    sel = np.nonzero(same)[0]
    st = torch.from_numpy(sel).to(DEV)
    assert_attn_close(runner.out[layer][pick_t][st], runner.lse[layer][pick_t][st], ro[sel],
                      rl[sel])
    print("C5 %s: %d rows; selection near-tie rows %d; end-to-end attention compared on %d rows"
          % (mode, len(pick), len(tie_rows), len(sel)))
