"""GPU parity of csa2_sparse_swa_attn_fp4kv (selected rows from the FP4 main-KV
pool, window rows FP8) against the oracle: several chunks with ragged tails,
chunks that mix FP4 selected rows and FP8 window rows in one step, tail
windows with a sink and invalid indices, and a decoder-replay sized case."""
import types

import numpy as np
import pytest
import torch

import sparse_attention_prefill_gb300 as S
from oracle import api as O
from sparse_attention_prefill_gb300 import synth
from tests.helpers import assert_attn_close, np_batch, npy

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _to(w_batch, dev=DEV):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in w_batch.items()}


def _case(n_heads, k, nq=9, ctx=3000, seed=0, win=None, sink=False, bad_idx=False):
    qpos = list(range(ctx - nq, ctx))
    w = synth.full_layer(ctx, 1, qpos, n_heads, 8, seed=seed, tag="fp4kv%d" % n_heads,
                         tail_win_lo=win)
    synth.with_fp4kv(w, seed)
    b = w.batch("full")
    L = w.layers["full"]
    g = torch.Generator().manual_seed(seed)
    idx = torch.full((nq, max(k, 1)), -1, dtype=torch.int32)
    for q in range(nq):
        nv = qpos[q] + 1
        take = min(k, nv) - (q % 3 == 1) * 5
        if take > 0:
            idx[q, :take] = torch.randperm(nv, generator=g)[:take].to(torch.int32)
    if bad_idx:
        idx[0, 0] = ctx + 5
        idx[1, 3] = qpos[1] + 1
    sk = torch.randn(n_heads, generator=g) if sink else None
    return w, b, L, idx[:, :k] if k else None, sk


def _run(w, b, L, idx, sk, wl=None):
    ref_o, ref_l, rerr = O.sparse_swa_attn_fp4kv(np_batch(b), npy(L.q), npy(w.pool.kv_fp4),
                                                 npy(w.pool.kv_sf), npy(idx), npy(L.swa_fp8),
                                                 npy(L.swa_scale), npy(wl), 128, w.sm_scale,
                                                 sink=npy(sk))
    d_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o, l = S.sparse_swa_attn_fp4kv(_to(b), L.q.to(DEV), w.pool.kv_fp4.to(DEV),
                                   w.pool.kv_sf.to(DEV), None if idx is None else idx.to(DEV),
                                   L.swa_fp8.to(DEV), L.swa_scale.to(DEV),
                                   None if wl is None else wl.to(DEV), 128, w.sm_scale,
                                   sink=None if sk is None else sk.to(DEV), d_err=d_err)
    assert_attn_close(o, l, ref_o, ref_l)
    assert int(d_err.item()) == rerr
    return rerr


@pytest.mark.parametrize("n_heads,k", [(64, 512), (16, 512), (32, 300), (64, 0), (64, 2048),
                                       (64, 37)])
def test_fp4kv_attention_parity(n_heads, k):
    w, b, L, idx, sk = _case(n_heads, k, seed=n_heads + k)
    assert _run(w, b, L, idx, sk) == 0


def test_fp4kv_tail_window_sink_and_bad_indices():
    w, b, L, idx, sk = _case(64, 512, nq=12, ctx=2500, seed=4, win=2495, sink=True, bad_idx=True)
    assert _run(w, b, L, idx, sk, L.win_lo) & S.DERR_RANGE_IDX


def test_fp4kv_decoder_replay_rows():
    """Two 8192-token requests of the decoder-replay shape, 64 tail rows each,
    with 512 uniformly sampled visible entries per row."""
    w = synth.decoder_replay([8192, 8192], [0, 0], 64, 32, seed=5, device="cpu", tag="fp4kvdr")
    synth.with_fp4kv(w, 5)
    rows = torch.cat([torch.arange(64, 128), torch.arange(192, 256)])
    b = w.batch("L22", rows)
    L = w.layers["L22"]
    g = torch.Generator().manual_seed(5)
    idx = torch.stack([torch.randperm(int(p) + 1, generator=g)[:512] for p in b["q_pos"]])
    idx = idx.to(torch.int32)
    Lr = types.SimpleNamespace(q=L.q[rows].contiguous(), swa_fp8=L.swa_fp8,
                               swa_scale=L.swa_scale)
    assert _run(w, b, Lr, idx, None, L.win_lo[rows].contiguous()) == 0
