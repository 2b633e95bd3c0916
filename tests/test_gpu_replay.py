"""GPU parity of the encoder-side bounded replay layout, the row cut /
scatter-back, and attention over an encoder replay's rows.

Encoder replay: "DeepSeek V4.1 Flash 建模", Encoder Bounded Replay card; the
SGLang/Miles day-0 article sec. 4.1 and 4.3.  Row cut / scatter-back: "SGLang
如何让 DeepSeek V4.1 Flash 的后半层只处理尾部 token", sec. 2.2 and 2.7.
Layouts and row copies are integer / byte work: bit-exact against the oracle.
"""
import numpy as np
import pytest
import torch

import sparse_attention_prefill_gb300 as S
from oracle import api as O
from sparse_attention_prefill_gb300 import synth
from sparse_attention_prefill_gb300.layer import LayerRunner
from tests.helpers import npy
from tests.test_gpu_configs import _layer_parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _layout_case(p, e, window, ratio, capacity=None):
    p_t = torch.tensor(p, dtype=torch.int64, device=DEV)
    e_t = torch.tensor(e, dtype=torch.int32, device=DEV)
    ref, rerr = O.encoder_replay_layout(np.array(p, np.int64), np.array(e, np.int32), window,
                                        ratio, capacity)
    cap = capacity if capacity is not None else max(1, int(ref["cu_rows"][-1]))
    d_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = S.encoder_replay_layout(p_t, e_t, cap, window, ratio, d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) == rerr
    n = len(ref["pos"])
    for k in ("replay_len", "cu_rows"):
        assert (npy(out[k]) == ref[k]).all(), k
    for k in ("src_row", "pos", "win_lo", "row_req"):
        assert (npy(out[k])[:n] == ref[k]).all(), k
    assert (npy(out["entry_range"])[:len(p)] == ref["entry_range"]).all()
    return out, ref


@pytest.mark.parametrize("ratio", [1, 2])
def test_encoder_replay_layout_bit_exact(ratio):
    rng = np.random.default_rng(ratio)
    # more than one 1024-request chunk, empty prefixes, short prefixes, empty extends
    p = rng.integers(0, 600, 2500).tolist()
    e = rng.integers(0, 300, 2500).tolist()
    p[:4] = [0, 1, 127, 8191]
    e[:4] = [5, 0, 1, 1]
    _layout_case(p, e, 128, ratio)
    _layout_case([8192], [100], 128, ratio)


def test_encoder_replay_layout_flags():
    # bad requests and a capacity cut
    _layout_case([10, -1, 300, 5], [4, 2, -3, 9], 128, 2)
    _layout_case([400, 400, 400], [50, 50, 50], 128, 2, capacity=200)


@pytest.mark.parametrize("row_bytes", [16, 48, 2048, 8208])
def test_rows_gather_scatter_bit_exact(row_bytes):
    g = torch.Generator().manual_seed(row_bytes)
    # the cut / scatter-back of a decoder extend batch's tail rows
    ext = torch.tensor([3000, 60, 129, 1000], dtype=torch.int32)
    seq = torch.tensor([3000, 900, 5000, 1200], dtype=torch.int64)
    tail = S.tail_layout(ext.to(DEV), seq.to(DEV), 128)
    n_full = int(ext.sum())
    full = torch.randint(0, 256, (n_full, row_bytes), dtype=torch.uint8, generator=g)
    full_d = full.to(DEV)
    count = tail["cu_tail"][-1:]                     # device scalar: no host sync
    cap = tail["src_row"].shape[0]
    cut = torch.full((cap, row_bytes), 7, dtype=torch.uint8, device=DEV)
    d_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    S.rows_gather(tail["src_row"], full_d, cut, count=count, d_err=d_err)
    fresh = torch.randint(0, 256, (cap, row_bytes), dtype=torch.uint8, generator=g)
    back = full_d.clone()
    S.rows_scatter(tail["src_row"], fresh.to(DEV), back, count=count, d_err=d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) == 0
    n = int(tail["cu_tail"][-1].item())
    src_row = npy(tail["src_row"])[:n]
    ref_cut, e1 = O.rows_gather(src_row, full.numpy(), np.full((n, row_bytes), 7, np.uint8))
    ref_back, e2 = O.rows_scatter(src_row, fresh.numpy()[:n], full.numpy())
    assert e1 == 0 and e2 == 0
    assert (npy(cut)[:n] == ref_cut).all()
    assert (npy(cut)[n:] == 7).all()                 # rows past the device count untouched
    assert (npy(back) == ref_back).all()


def test_rows_skip_and_range_flag():
    full = torch.arange(40 * 32, dtype=torch.int32).reshape(40, 32).to(DEV)   # 128-byte rows
    idx = torch.tensor([3, -1, 39, 40, 7, 1000], dtype=torch.int32, device=DEV)
    dst = torch.full((6, 32), -5, dtype=torch.int32, device=DEV)
    d_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    S.rows_gather(idx, full, dst, d_err=d_err)
    torch.cuda.synchronize()
    ref, rerr = O.rows_gather(npy(idx), npy(full), np.full((6, 32), -5, np.int32))
    assert int(d_err.item()) == rerr == S.DERR_RANGE_ROW
    assert (npy(dst) == ref).all()
    d_err.zero_()
    tgt = full.clone()
    S.rows_scatter(idx, dst, tgt, d_err=d_err)
    torch.cuda.synchronize()
    ref2, rerr2 = O.rows_scatter(npy(idx), npy(dst), npy(full))
    assert int(d_err.item()) == rerr2 == S.DERR_RANGE_ROW
    assert (npy(tgt) == ref2).all()


@pytest.mark.parametrize("prefix,extend", [(4096, 200), (60, 200), (4097, 33)])
def test_encoder_replay_attention(prefix, extend):
    """A Full encoder layer (m = 2) over the rows of an encoder replay: the
    layout's positions and lower bound drive the GPU chain (score, top-K,
    attention) and the oracle chain on the same rows."""
    out, ref = _layout_case([prefix], [extend], 128, 2)
    rp = int(ref["replay_len"][0])
    pos = ref["pos"].tolist()
    w = synth.full_layer(prefix + extend, 2, pos, 16, 8, seed=5, device=DEV,
                         tail_win_lo=prefix - rp, tag=f"encreplay{prefix}")
    assert (npy(w.layers["full"].win_lo) == ref["win_lo"]).all()
    run = LayerRunner(w)
    run.full_layer("full")
    torch.cuda.synchronize()
    assert int(run.d_err.item()) == 0
    rows = torch.arange(w.num_q, device=DEV)
    _layer_parity(w, run, "full", rows, "full", win_lo=w.layers["full"].win_lo)
