"""GPU parity of the decoder tail step under other replay budgets R.

"SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部 token", sec. 3.5 proposes
sweeping the number of rows the late layers keep (R = 64, 128, 256, 512) while
the model's SWA width stays 128.  The tail layout keeps T = min(R, E) rows per
request with window lower bound S - T; attention still reads at most the last
128 positions, so for R > 128 the first rows of each tail see a truncated
window and the later ones a full one.  Each case runs the whole GPU chain
(tail layout, L20-style source, L21-style pool Reindex, L22-style Reuse) and
compares it with the oracle chain under the same tolerances as the named
workloads.
"""
import numpy as np
import pytest
import torch

from oracle import api as O
from sparse_attention_prefill_gb300 import synth
from sparse_attention_prefill_gb300.layer import LayerRunner
from tests.helpers import npy
from tests.test_gpu_configs import _layer_parity

pytestmark = pytest.mark.gpu
DEV = "cuda"

# extends mix long, medium and shorter-than-R requests over cached prefixes
EXTENDS = [700, 300, 64, 1000]
PREFIXES = [0, 1500, 600, 200]


@pytest.mark.parametrize("replay", [64, 256, 512])
def test_decoder_tail_step_replay_budget(replay):
    w = synth.decoder_replay(EXTENDS, PREFIXES, 16, 8, seed=3, device=DEV,
                             tag=f"replay{replay}", replay=replay)
    assert w.window == 128 and w.replay == replay
    run = LayerRunner(w)
    run.decoder_tail_step()
    torch.cuda.synchronize()
    assert int(run.d_err.item()) == 0
    tail, terr = O.tail_layout(npy(w.extend_len), npy(w.seq_len), replay)
    n = int(tail["cu_tail"][-1])
    assert terr == 0 and n == w.num_q == sum(min(replay, e) for e in EXTENDS)
    for k in ("tail_len", "cu_tail"):
        assert (npy(run.tail[k]) == tail[k]).all(), k
    for k in ("pos", "win_lo", "src_row", "row_req"):
        assert (npy(run.tail[k])[:n] == tail[k]).all(), k
    # some rows have a window cut by the bound, and (R > 128) some a full one
    pos, lo = tail["pos"], tail["win_lo"]
    assert (pos - lo < 127).any()
    if replay > 128:
        assert (pos - lo >= 127).any()
    rows = torch.arange(w.num_q, device=DEV)
    win = run.tail_win_lo
    _, blocks, pool_rows = _layer_parity(w, run, "L20", rows, "source", label="R=%d" % replay)
    idx21, _, just21 = _layer_parity(w, run, "L21", rows, "reindex", pool=blocks, win_lo=win,
                                     justified=pool_rows, label="R=%d" % replay)
    _layer_parity(w, run, "L22", rows, "reuse", given_idx=idx21, win_lo=win, justified=just21,
                  chain_idx=run.idx["L21"])
