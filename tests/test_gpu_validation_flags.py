"""Device data-error flags the other GPU tests do not reach: MXFP4 scales that
are not in-range powers of two, and score rows longer than the stride ld.
Both are reported without faulting; the cut rows match the oracle."""
import numpy as np
import pytest
import torch

import sparse_attention_prefill_gb300 as S
from oracle import api as O
from sparse_attention_prefill_gb300 import synth
from tests.helpers import np_batch, npy

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _to(b):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in b.items()}


def _derr():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _score(w, b, L, q_scale, k_scale, ld, d_err, scores=None):
    return S.index_score(_to(b), L.q_fp4.to(DEV), q_scale.to(DEV), L.head_w.to(DEV),
                         w.pool.k_fp4.to(DEV), k_scale.to(DEV), ld, scores=scores, d_err=d_err)


def test_index_scale_not_a_power_of_two_is_flagged():
    w = synth.full_layer(3000, 1, [2999, 1500, 200], 16, 32, seed=21, tag="flagscale")
    b, L = w.batch("full"), w.layers["full"]
    d0 = _derr()
    _score(w, b, L, L.q_scale, w.pool.k_scale, w.ld, d0)
    torch.cuda.synchronize()
    assert int(d0.item()) == 0
    # a key scale of 3 on entry 100 (visible to every query)
    ks = w.pool.k_scale.clone()
    ks[100, 1] = 3.0
    d1 = _derr()
    _score(w, b, L, L.q_scale, ks, w.ld, d1)
    torch.cuda.synchronize()
    assert int(d1.item()) & S.DERR_SCALE
    # a query scale of 0.75
    qs = L.q_scale.clone()
    qs[0, 0, 0] = 0.75
    d2 = _derr()
    _score(w, b, L, qs, w.pool.k_scale, w.ld, d2)
    torch.cuda.synchronize()
    assert int(d2.item()) & S.DERR_SCALE


def test_index_rows_longer_than_ld_are_cut_and_flagged():
    w = synth.full_layer(3000, 1, [2999, 1000, 10], 16, 32, seed=22, tag="flagld")
    b, L = w.batch("full"), w.layers["full"]
    ld = 1024
    ref, rerr = O.index_score(np_batch(b), npy(L.q_fp4), npy(L.q_scale), npy(L.head_w),
                              npy(w.pool.k_fp4), npy(w.pool.k_scale), ld)
    assert rerr & S.DERR_LD
    bound, _ = O.index_score(np_batch(b), npy(L.q_fp4), npy(L.q_scale), np.abs(npy(L.head_w)),
                             npy(w.pool.k_fp4), npy(w.pool.k_scale), ld)
    got = torch.full((3, ld), float("nan"), device=DEV)
    d_err = _derr()
    _score(w, b, L, L.q_scale, w.pool.k_scale, ld, d_err, scores=got)
    torch.cuda.synchronize()
    assert int(d_err.item()) == rerr
    g = npy(got)
    written = ~np.isnan(ref)
    assert (np.isnan(g) == ~written).all()
    tol = 1e-5 * np.nan_to_num(np.abs(bound), nan=0.0) + 1e-30
    assert (np.abs(g[written] - ref[written]) <= tol[written]).all()
