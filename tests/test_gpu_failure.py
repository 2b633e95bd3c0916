"""Failure paths of the tensor-core kernels on the GPU, made without a fault:
the pipeline-wait bound is shortened to 1 ns, so every wait that is not
satisfied at once runs out.  The kernel must report CSA2_DERR_TIMEOUT through
the host-read flag and return with its tensor memory freed and the context
usable: a following call at the default bound gives the oracle's result.
(Negative cases reported without taking the serving process down:
"SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部 token", sec. 2.7.)"""
import numpy as np
import pytest
import torch

import sparse_attention_prefill_gb300 as S
from oracle import api as O
from sparse_attention_prefill_gb300 import synth
from tests.helpers import assert_attn_close, np_batch, npy

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _derr():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _case():
    nq, ctx = 40, 3000
    qpos = list(range(ctx - nq, ctx))
    w = synth.full_layer(ctx, 1, qpos, 64, 32, seed=31, device=DEV, tag="waits")
    g = torch.Generator().manual_seed(31)
    idx = torch.stack([torch.randperm(p + 1, generator=g)[:512] for p in qpos]).to(torch.int32)
    return w, w.batch("full"), w.layers["full"], idx.to(DEV)


def _attend(w, b, L, idx, d_err):
    return S.sparse_swa_attn(b, L.q, w.pool.kv_fp8, w.pool.kv_scale, idx, L.swa_fp8,
                             L.swa_scale, None, w.window, w.sm_scale, d_err=d_err)


def _score(w, b, L, d_err):
    return S.index_score(b, L.q_fp4, L.q_scale, L.head_w, w.pool.k_fp4, w.pool.k_scale, w.ld,
                         d_err=d_err)


def test_attention_wait_runs_out_then_recovers():
    w, b, L, idx = _case()
    S.set_wait_limit_ns(1)
    try:
        d0 = _derr()
        for _ in range(3):
            _attend(w, b, L, idx, d0)
        torch.cuda.synchronize()
    finally:
        S.set_wait_limit_ns(0)
    assert int(d0.item()) & S.DERR_TIMEOUT
    d1 = _derr()
    out, lse = _attend(w, b, L, idx, d1)
    torch.cuda.synchronize()
    assert int(d1.item()) == 0
    ro, rl, _ = O.sparse_swa_attn(np_batch(b), npy(L.q), npy(w.pool.kv_fp8),
                                  npy(w.pool.kv_scale), npy(idx), npy(L.swa_fp8),
                                  npy(L.swa_scale), None, w.window, w.sm_scale)
    assert_attn_close(out, lse, ro, rl)


def test_index_score_wait_runs_out_then_recovers():
    w, b, L, _ = _case()
    S.set_wait_limit_ns(1)
    try:
        d0 = _derr()
        for _ in range(3):
            _score(w, b, L, d0)
        torch.cuda.synchronize()
    finally:
        S.set_wait_limit_ns(0)
    assert int(d0.item()) & S.DERR_TIMEOUT
    d1 = _derr()
    got = _score(w, b, L, d1)
    torch.cuda.synchronize()
    assert int(d1.item()) == 0
    nb = np_batch(b)
    ref, _ = O.index_score(nb, npy(L.q_fp4), npy(L.q_scale), npy(L.head_w), npy(w.pool.k_fp4),
                           npy(w.pool.k_scale), w.ld)
    bound, _ = O.index_score(nb, npy(L.q_fp4), npy(L.q_scale), np.abs(npy(L.head_w)),
                             npy(w.pool.k_fp4), npy(w.pool.k_scale), w.ld)
    g = npy(got)[:, :ref.shape[1]]
    fin = np.isfinite(ref)
    tol = 1e-5 * np.nan_to_num(np.abs(bound), nan=0.0) + 1e-30
    assert (np.abs(g[fin] - ref[fin]) <= tol[fin]).all()
