"""Pins of the oracle's bounded-replay tail layout against the pages' worked
examples (tests/golden/tail_layout_pages.json, each with its citation) and
brute force."""
import json
import os

import numpy as np
import pytest

from oracle import api as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tail_layout_pages.json")))


def _tail(e, s, window=128):
    out, err = O.tail_layout(np.array(e), np.array(s), window)
    assert err == 0
    return out


@pytest.mark.parametrize("case", ["single_extend_8192", "short_extend"])
def test_single_request_examples(case):
    g = GOLD[case]
    out = _tail(g["extend_len"], g["seq_len"])
    assert out["tail_len"].tolist() == g["tail_len"]
    assert out["pos"][0] == g["first_pos"] and out["pos"][-1] == g["last_pos"]
    assert (out["win_lo"] == g["win_lo"]).all()
    # positions stay absolute: never renumbered from 0
    assert out["pos"].tolist() == list(range(g["first_pos"], g["last_pos"] + 1))
    # the rows kept are the last T rows of the extend
    e = g["extend_len"][0]
    t = g["tail_len"][0]
    assert out["src_row"].tolist() == list(range(e - t, e))


def _window_rows_used(t, win_lo, window=128):
    """Which SWA positions does the oracle's attention read for a query at t?
    Every SWA row p holds the constant value p (code 1.0, scale p) and the query
    is zero, so all logits are equal: lse = log(count) and O = mean(positions)."""
    lo_store = max(0, t - 300)
    n = t - lo_store + 1
    swa_fp8 = np.full((n, 512), 0x38, np.uint8)          # E4M3 code of 1.0
    swa_scale = np.repeat(np.arange(lo_store, t + 1, dtype=np.float32)[:, None], 16, 1)
    b = dict(num_q=1, num_req=1, ratio=1, q_req=[0], q_pos=[t], kv_start=[0], kv_len=[t + 1],
             swa_start=[0], swa_pos0=[lo_store], swa_len=[n])
    q = np.zeros((1, 1, 512), np.uint16)
    out, lse, err = O.sparse_swa_attn(b, q, np.zeros((1, 512), np.uint8),
                                      np.ones((1, 16), np.float32), None, swa_fp8, swa_scale,
                                      None if win_lo is None else np.array([win_lo]), window)
    assert err == 0
    count = int(round(float(np.exp(lse[0, 0]))))
    mean = float(np.frombuffer((out[0, 0, :1].astype(np.uint32) << 16).tobytes(), np.float32)[0])
    return count, mean


@pytest.mark.parametrize("case", ["single_extend_8192", "short_extend"])
def test_visible_window_table(case):
    g = GOLD[case]
    for row in g["visible"]:
        t = row["t"]
        for kind in ("normal", "bounded"):
            if kind not in row:
                continue
            lo, hi = row[kind]
            assert hi == t
            count, mean = _window_rows_used(t, g["win_lo"] if kind == "bounded" else None)
            assert count == hi - lo + 1
            # the mean of the positions is (lo + hi) / 2, exact up to bf16 rounding
            assert abs(mean - (lo + hi) / 2) <= 2 ** -8 * abs(mean)


def test_chunk_tails():
    g = GOLD["chunked_32768"]
    # as one batch of independent extends and as four separate extend calls
    out = _tail(g["extend_len"], g["seq_len"])
    got = [[int(out["pos"][out["cu_tail"][r]]), int(out["pos"][out["cu_tail"][r + 1] - 1])]
           for r in range(4)]
    assert got == g["tails"]
    for r in range(4):
        o = _tail([g["extend_len"][r]], [g["seq_len"][r]])
        assert [int(o["pos"][0]), int(o["pos"][-1])] == g["tails"][r]


def test_token_layer_counts():
    g = GOLD["token_layer_counts"]
    for c in g["cases"]:
        e = c["extend_len"]
        s = np.cumsum(e)  # chunks of one prompt: each extend ends where it ends
        out = _tail(e, s)
        tail = g["layers_full"] * sum(e) + g["layers_tail"] * int(out["tail_len"].sum())
        assert tail == c["tail"]
        assert 40 * sum(e) == c["full"]
        if "reduction_pct" in c:
            assert abs((c["full"] - tail) / c["full"] * 100 - c["reduction_pct"]) < 1e-12


@pytest.mark.parametrize("e", [0, 1, 63, 127, 128, 129, 4097])
def test_boundary_lengths_and_per_request(e):
    # heterogeneous batch: each request keeps its own tail (never one cut of the batch)
    es = [e, 8192, 1, e]
    ss = [e + 10, 8192 + 7, 1, e]
    out = _tail(es, ss)
    assert out["tail_len"].tolist() == [min(128, x) for x in es]
    assert out["cu_tail"].tolist() == list(np.concatenate([[0], np.cumsum(out["tail_len"])]))
    # brute force: enumerate the rows of each extend and keep the last T
    cu_e = np.concatenate([[0], np.cumsum(es)])
    rows, pos, lo = [], [], []
    for r, (x, s) in enumerate(zip(es, ss)):
        keep = list(range(x))[-min(128, x):] if x else []
        rows += [int(cu_e[r]) + k for k in keep]
        pos += [s - x + k for k in keep]          # extend row k sits at s - x + k
        lo += [s - min(128, x)] * len(keep)
    assert out["src_row"].tolist() == rows
    assert out["pos"].tolist() == pos
    assert out["win_lo"].tolist() == lo


def test_bad_extend_and_capacity_flags():
    _, err = O.tail_layout(np.array([5, -1]), np.array([3, 10]), 128)
    assert err & 64
    out, err = O.tail_layout(np.array([200, 200]), np.array([200, 300]), 128, capacity=150)
    assert err & 32
    assert out["cu_tail"].tolist() == [0, 128, 256]


@pytest.mark.parametrize("R", [64, 256, 512])
def test_replay_budget_sweep(R):
    """"SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部 token", sec. 3.5: the
    rows kept (R) are swept while the SWA width stays 128.  The layout keeps
    T = min(R, E) rows per request with lower bound S - T, and a kept row at t
    reads the positions [max(S - T, t - 127), t]: for R > 128 the first 127
    rows of a tail are cut by the bound, the rest see a full window."""
    es, ss = [8192, 100, 1000], [8192, 600, 5000]
    out = _tail(es, ss, R)
    ts = [min(R, e) for e in es]
    assert out["tail_len"].tolist() == ts
    cu_e = np.concatenate([[0], np.cumsum(es)])
    rows, pos, lo = [], [], []
    for r, (e, s, t) in enumerate(zip(es, ss, ts)):
        rows += [int(cu_e[r]) + e - t + k for k in range(t)]
        pos += [s - t + k for k in range(t)]
        lo += [s - t] * t
    assert out["src_row"].tolist() == rows
    assert out["pos"].tolist() == pos
    assert out["win_lo"].tolist() == lo
    # windows of the first request's rows (S = E = 8192)
    s, t = 8192, ts[0]
    for k in sorted({0, 1, 126, 127, 128, t - 1} & set(range(t))):
        q = s - t + k
        count, mean = _window_rows_used(q, s - t)
        first = max(s - t, q - 127)
        assert count == q - first + 1 == min(k + 1, 128)
        assert abs(mean - (first + q) / 2) <= 2 ** -8 * abs(mean)
