"""Pins of the oracle's encoder-side bounded-replay layout and of the row cut /
scatter-back, against the rules the pages state, closed forms and brute force.

Encoder replay: "DeepSeek V4.1 Flash 建模", Encoder Bounded Replay card, and the
SGLang/Miles day-0 article, sec. 4.1 and 4.3: on a prefix hit whose SWA state
was dropped, the last 128 cached tokens are processed again together with the
new suffix; they rebuild SWA only, the cached global entries stay as they are,
and local attention is cut at the rebuild boundary.

Row cut / scatter-back: "SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部
token", sec. 2.2 (the per-row state is cut to the tail rows on entry to the late
layers, and the outer layout is restored afterwards) and sec. 2.7 (the computed
tail rows are scattered back into the full extend layout; the other rows are
not filled in).
"""
import numpy as np
import pytest

from oracle import api as O
from tests.test_oracle_tail import _window_rows_used


def test_prefix_hit_replays_last_128():
    # P = 8192 cached tokens (m = 2: 4096 cached entries), 100 new tokens
    out, err = O.encoder_replay_layout([8192], [100], 128, 2)
    assert err == 0
    assert out["replay_len"].tolist() == [128]
    assert out["cu_rows"].tolist() == [0, 228]
    assert out["pos"].tolist() == list(range(8064, 8292))
    assert (out["win_lo"] == 8064).all()
    assert out["src_row"].tolist() == [-1] * 128 + list(range(100))
    # entries 0..4095 are cached and read only; the extend completes 4096..4145
    assert out["entry_range"].tolist() == [[4096, 4146]]


@pytest.mark.parametrize("p", [0, 1, 50, 127, 128, 129])
def test_short_and_empty_prefix(p):
    out, err = O.encoder_replay_layout([p], [10], 128, 2)
    assert err == 0
    rp = min(128, p)
    assert out["replay_len"].tolist() == [rp]
    assert out["pos"].tolist() == list(range(p - rp, p + 10))
    assert (out["win_lo"] == p - rp).all()
    if p <= 128:
        # the whole prefix is replayed: the bound is 0, i.e. no cut at all
        assert (out["win_lo"] == 0).all()


def test_pending_pair_and_chunk_tiling():
    # m = 2, odd prefix: entry 4095 pairs tokens 8190 (cached, replayed) and 8191 (new)
    out, _ = O.encoder_replay_layout([8191], [1], 128, 2)
    assert out["entry_range"].tolist() == [[4095, 4096]]
    assert 8190 in out["pos"].tolist() and out["src_row"][-1] == 0
    # consecutive extends of one sequence complete every entry exactly once, and
    # no extend's range reaches below the entries its prefix already holds
    rng = np.random.default_rng(0)
    for m in (1, 2):
        cuts = np.sort(rng.choice(np.arange(1, 3000), 12, replace=False))
        bounds = [0] + cuts.tolist() + [3001]
        seen = []
        for a, b in zip(bounds[:-1], bounds[1:]):
            o, err = O.encoder_replay_layout([a], [b - a], 128, m)
            assert err == 0
            lo, hi = o["entry_range"][0]
            assert lo == a // m                  # cached entries are never rewritten
            seen += list(range(lo, hi))
        assert seen == list(range(3001 // m))


def test_brute_force_batch_and_flags():
    rng = np.random.default_rng(1)
    p = rng.integers(0, 400, 40).tolist() + [-1, 5]
    e = rng.integers(0, 200, 40).tolist() + [3, -2]
    out, err = O.encoder_replay_layout(p, e, 128, 2)
    assert err == 64                                  # the two bad requests
    rows_src, rows_pos, rows_lo, rows_req = [], [], [], []
    cu_e = 0
    for r, (a, b) in enumerate(zip(p, e)):
        if a < 0 or b < 0:
            assert out["replay_len"][r] == 0
            continue
        rp = min(128, a)
        for k in range(rp + b):
            rows_pos.append(a - rp + k)
            rows_lo.append(a - rp)
            rows_src.append(-1 if k < rp else cu_e + k - rp)
            rows_req.append(r)
        cu_e += b
    assert out["pos"].tolist() == rows_pos
    assert out["win_lo"].tolist() == rows_lo
    assert out["src_row"].tolist() == rows_src
    assert out["row_req"].tolist() == rows_req
    # capacity cut: rows past it are not written and flagged
    small, err2 = O.encoder_replay_layout(p[:3], e[:3], 128, 2, capacity=10)
    assert err2 & 32 and len(small["pos"]) == 10


def test_new_rows_see_full_windows():
    """With a full 128-token replay, the first new row's window [P-127, P] lies
    inside the rebuilt rows, so no new row is cut; replayed rows are."""
    p = 4096
    lo = p - 128
    for t, expect in [(lo, 1), (lo + 5, 6), (p - 1, 128), (p, 128), (p + 40, 128)]:
        count, _ = _window_rows_used(t, lo)
        assert count == expect, (t, count)


def test_rows_gather_scatter():
    rng = np.random.default_rng(2)
    full = rng.integers(0, 256, (300, 48), dtype=np.uint8)
    t, _ = O.tail_layout(np.array([200, 60, 40], np.int32), np.array([500, 60, 900], np.int64),
                         32)
    cut, err = O.rows_gather(t["src_row"], full, np.zeros((len(t["src_row"]), 48), np.uint8))
    assert err == 0 and (cut == full[t["src_row"]]).all()
    # scatter-back: the tail rows land at their extend rows, all others untouched
    fresh = rng.integers(0, 256, cut.shape, dtype=np.uint8)
    back, err = O.rows_scatter(t["src_row"], fresh, full)
    assert err == 0
    expect = full.copy()
    expect[t["src_row"]] = fresh
    assert (back == expect).all()
    others = np.setdiff1d(np.arange(300), t["src_row"])
    assert (back[others] == full[others]).all()
    # negative indices are skipped; out-of-range ones are skipped and flagged
    idx = np.array([3, -1, 299, 300, 7], np.int32)
    dst = np.full((5, 48), 9, np.uint8)
    g, err = O.rows_gather(idx, full, dst)
    assert err == 256
    assert (g[0] == full[3]).all() and (g[1] == 9).all() and (g[3] == 9).all()
    s, err = O.rows_scatter(idx, dst + 1, full)
    assert err == 256 and (s[3] == 10).all() and (s[299] == 10).all() and (s[0] == full[0]).all()
