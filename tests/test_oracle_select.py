"""Pins of the oracle's top-K and hierarchical candidate-block selection:
brute force by full sort on small rows and the pages' invariants."""
import numpy as np
import pytest

from oracle import api as O


def _batch(q_pos, ratio=1, kv_len=None):
    nq = len(q_pos)
    kv_len = kv_len or [10 ** 9]
    return dict(num_q=nq, num_req=1, ratio=ratio, q_req=np.zeros(nq, np.int32),
                q_pos=np.asarray(q_pos, np.int64), kv_start=np.zeros(1, np.int64),
                kv_len=np.asarray(kv_len, np.int64), swa_start=np.zeros(1, np.int64),
                swa_pos0=np.zeros(1, np.int64), swa_len=np.zeros(1, np.int64))


def _brute_topk(row, k):
    elig = [(float(v), j) for j, v in enumerate(row) if not np.isnan(v) and v != -np.inf]
    elig.sort(key=lambda p: (-p[0], p[1]))
    return [j for _, j in elig[:k]]


@pytest.mark.parametrize("seed", range(4))
def test_topk_brute_force_with_ties_nan_inf(seed):
    rng = np.random.default_rng(seed)
    n, k = 300, 37
    s = np.round(rng.standard_normal((5, n)) * 4) / 4          # many exact ties
    s[rng.random((5, n)) < 0.05] = np.nan
    s[rng.random((5, n)) < 0.05] = -np.inf
    s[rng.random((5, n)) < 0.02] = np.inf
    s = s.astype(np.float32)
    q_pos = [n - 1, 10, 36, 37, 150]
    idx, count, err = O.topk(_batch(q_pos), s, k)
    assert err == 0
    for q, t in enumerate(q_pos):
        want = _brute_topk(s[q, :t + 1], k)
        assert count[q] == len(want)
        assert idx[q, :count[q]].tolist() == want
        assert (idx[q, count[q]:] == -1).all()


def test_topk_signed_zeros_tie_by_entry():
    """-0 and +0 are equal scores, so the entry id orders them."""
    row = np.array([-0.0, 1.0, 0.0, -0.0, 0.0, -1.0], np.float32)
    idx, count, err = O.topk(_batch([5]), row[None, :], 3)
    assert err == 0 and count[0] == 3
    assert idx[0].tolist() == [1, 0, 2]


def test_topk_invariants_and_short_rows():
    rng = np.random.default_rng(7)
    s = rng.standard_normal((3, 2000)).astype(np.float32)
    idx, count, _ = O.topk(_batch([1999, 511, 99], ratio=1), s, 512)
    assert count.tolist() == [512, 512, 100]
    sel = idx[0, :512]
    kth = s[0, sel].min()
    rest = np.setdiff1d(np.arange(2000), sel)
    assert (s[0, rest] <= kth).all()
    # K >= n_vis: every visible entry is selected (dense case)
    assert sorted(idx[2, :100].tolist()) == list(range(100))


def test_topk_pool_mode_maps_slots():
    rng = np.random.default_rng(3)
    blocks = np.array([[1, 3, 6, -1]], np.int32)
    s = rng.standard_normal((1, 32)).astype(np.float32)
    idx, count, _ = O.topk(_batch([50]), s, 5, cand_blocks=blocks, block=8)
    slots = list(range(24))
    entry = [blocks[0, sl // 8] * 8 + sl % 8 for sl in slots]
    vis = [(float(s[0, sl]), entry[sl]) for sl in slots if entry[sl] <= 50]
    vis.sort(key=lambda p: (-p[0], p[1]))
    assert idx[0].tolist() == [e for _, e in vis[:5]]
    assert count[0] == 5


def _brute_blocks(row, n_vis, bsz, nb_max):
    nb = -(-n_vis // bsz)
    if nb <= nb_max:
        return list(range(nb))
    bm = []
    for b in range(nb - 1):
        vals = [v for v in row[b * bsz:min((b + 1) * bsz, n_vis)] if not np.isnan(v)]
        bm.append((max(vals) if vals else -np.inf, b))
    bm.sort(key=lambda p: (-p[0], p[1]))
    return sorted([b for _, b in bm[:nb_max - 1]] + [nb - 1])


@pytest.mark.parametrize("seed,nb_max", [(s, 4) for s in range(6)] + [(6, 1), (7, 2)])
def test_candidates_brute_force_small_pool(seed, nb_max):
    """A one-block budget keeps only the latest block; two keep it plus the
    best earlier block."""
    rng = np.random.default_rng(seed)
    bsz, n = 2, 23
    s = np.round(rng.standard_normal((n, n)) * 2) / 2
    s = s.astype(np.float32)
    q_pos = list(range(n))
    idx, count, blocks, nblocks, err = O.topk_candidates(_batch(q_pos), s, k=3, block=bsz,
                                                         max_blocks=nb_max)
    assert err == 0
    for q in range(n):
        want = _brute_blocks(s[q], q + 1, bsz, nb_max)
        assert nblocks[q] == len(want)
        assert blocks[q, :len(want)].tolist() == want
        assert (blocks[q, len(want):] == -1).all()
        # the block holding the latest visible position is always kept
        assert q // bsz in want
        assert idx[q, :count[q]].tolist() == _brute_topk(s[q, :q + 1], 3)


@pytest.mark.parametrize("n_vis,n_blocks,kept", [(16383, 2048, 2048), (16384, 2048, 2048),
                                                 (16385, 2049, 2048), (16393, 2050, 2048),
                                                 (9, 2, 2), (1, 1, 1), (0, 0, 0)])
def test_candidates_pool_budget_invariants(n_vis, n_blocks, kept):
    """Pages: <= 2048 blocks of 8 (<= 16384 positions); the latest block is
    always kept; the filter excludes nothing when all reachable positions fit."""
    rng = np.random.default_rng(n_vis)
    s = rng.standard_normal((1, max(n_vis, 1))).astype(np.float32)
    _, _, blocks, nblocks, _ = O.topk_candidates(_batch([n_vis - 1]), s, k=512)
    assert nblocks[0] == kept
    got = blocks[0, :kept]
    if n_blocks <= 2048:
        assert got.tolist() == list(range(n_blocks))
    else:
        assert got[-1] == n_blocks - 1                      # latest block kept
        assert len(set(got.tolist())) == 2048 and (np.diff(got) > 0).all()
        dropped = sorted(set(range(n_blocks)) - set(got.tolist()))
        assert len(dropped) == n_blocks - 2048
        bmax = [s[0, 8 * b:min(8 * b + 8, n_vis)].max() for b in range(n_blocks)]
        worst_kept = min(bmax[b] for b in got[:-1])
        for d in dropped:
            assert bmax[d] <= worst_kept
