"""csa2_index_topk_static: the streamed index score -> top-K for callers that
cannot allocate device memory (code running under CUDA graph capture, a
memory pool's own set-up, runtimes that forbid cudaMalloc after start-up).
It uses the library's fixed scratch array instead of a workspace.  Called
through the C ABI twice in a row on different inputs (the array keeps the
first call's contents), each result must equal csa2_index_topk's with a
caller-allocated workspace on the same inputs; a request larger than the
array is rejected.  This file is collected last, so a run that stops at the
first failure has run every other test before it."""
import pytest
import torch

import sparse_attention_prefill_gb300 as S
from sparse_attention_prefill_gb300 import synth
from tests.helpers import npy, topk_sets_match

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _layer(seed, qpos, ctx, ratio, hi):
    w = synth.full_layer(ctx, ratio, qpos, 16, hi, seed=seed, device=DEV, tag="noalloc%d" % seed)
    return w, w.batch("full"), w.layers["full"]


def _with_workspace(w, b, L, k):
    need = S.csa2_index_topk_workspace(w.num_q, w.ld)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    idx = torch.empty((w.num_q, k), dtype=torch.int32, device=DEV)
    cnt = torch.empty(w.num_q, dtype=torch.int32, device=DEV)
    d_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = S.csa2_index_topk(b, L.q_fp4.shape[1], 128, L.q_fp4, L.q_scale, L.head_w, w.pool.k_fp4,
                           w.pool.k_scale, w.ld, k, idx, cnt, ws, need, d_err)
    assert st == S.OK
    return idx, cnt, d_err


def _static(w, b, L, k):
    idx = torch.empty((w.num_q, k), dtype=torch.int32, device=DEV)
    cnt = torch.empty(w.num_q, dtype=torch.int32, device=DEV)
    d_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = S.csa2_index_topk_static(b, L.q_fp4.shape[1], 128, L.q_fp4, L.q_scale, L.head_w,
                                  w.pool.k_fp4, w.pool.k_scale, w.ld, k, idx, cnt, d_err)
    return st, idx, cnt, d_err


def test_static_scratch_matches_workspace_path_on_two_calls():
    # rows long enough for the sample and list passes, plus short ones
    cases = [_layer(11, [100, 5000, 9000, 12345, 19999], 20000, 1, 32),
             _layer(12, [8192 + 3 * i for i in range(40)] + [50], 40000, 2, 64)]
    for w, b, L in cases:
        for k in (512, 100):
            st, si, sc, sd = _static(w, b, L, k)
            assert st == S.OK
            ri, rc, rd = _with_workspace(w, b, L, k)
            torch.cuda.synchronize()
            topk_sets_match(si, sc, npy(ri), npy(rc))
            assert int(sd.item()) == int(rd.item()) == 0


def test_static_scratch_rejects_requests_larger_than_the_array():
    cap = S.csa2_index_topk_static_capacity()
    assert cap == 64 << 20
    w, b, L = _layer(13, [30000], 40000, 1, 32)
    rows = cap // S.csa2_index_topk_workspace(1, w.ld)
    while S.csa2_index_topk_workspace(rows, w.ld) <= cap:   # the smallest batch that exceeds it
        rows += 1
    b = dict(b, num_q=rows, q_req=torch.zeros(rows, dtype=torch.int32, device=DEV),
             q_pos=torch.full((rows,), 30000, dtype=torch.int64, device=DEV))
    idx = torch.empty((rows, 512), dtype=torch.int32, device=DEV)
    cnt = torch.empty(rows, dtype=torch.int32, device=DEV)
    q_fp4 = L.q_fp4.expand(rows, -1, -1).contiguous()
    q_scale = L.q_scale.expand(rows, -1, -1).contiguous()
    st = S.csa2_index_topk_static(b, 32, 128, q_fp4, q_scale, None, w.pool.k_fp4,
                                  w.pool.k_scale, w.ld, 512, idx, cnt, None)
    assert st == S.ERR_TOO_LARGE
    assert "scratch" in S.status_string(st)
