"""CSA2 layer call sequences over the C ABI (host orchestration only).

Mode -> calls ("DeepSeek V4.1 Flash 建模", CSA2 path table; SGLang/Miles day-0
article sec. 2):
  Full      csa2_index_score (all visible) -> csa2_topk -> csa2_sparse_swa_attn
  Source    csa2_index_score (all visible) -> csa2_topk_candidates -> attention
            (the L20-style layer that publishes the candidate pool)
  Reindex   csa2_index_score (restricted to the pool, or all visible) ->
            csa2_topk -> attention
  Reuse     attention with the indices another index source produced
Tail layers first run csa2_tail_layout and use its positions and window lower
bounds ("SGLang 如何让 DeepSeek V4.1 Flash 的后半层只处理尾部 token", sec. 2.1-2.2).
All buffers are allocated once per runner; the calls only enqueue kernels.
"""
from __future__ import annotations

from typing import Dict, Optional

import torch

from . import (csa2_index_score, csa2_sparse_swa_attn, csa2_tail_layout, csa2_topk,
               csa2_topk_candidates)
from .synth import Workload


def _check(st, what):
    from . import _check as chk
    chk(st, what)


class LayerRunner:
    """Pre-allocated buffers and call sequences for one workload on one device."""

    def __init__(self, w: Workload, rows: Optional[torch.Tensor] = None):
        self.w = w
        dev = w.q_pos.device
        self.dev = dev
        self.rows = rows
        nq = w.num_q if rows is None else int(rows.numel())
        self.nq = nq
        self.d_err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.scores = torch.empty((nq, max(1, w.ld)), dtype=torch.float32, device=dev)
        # pool rows hold at most min(max_blocks, ceil(ld / block)) blocks: the
        # candidate blocks are distinct blocks of a visible range of <= ld entries
        pool_len = min(w.max_blocks, -(-max(1, w.ld) // w.block)) * w.block
        self.pool_scores = torch.empty((nq, pool_len), dtype=torch.float32, device=dev)
        self.idx: Dict[str, torch.Tensor] = {}
        self.count: Dict[str, torch.Tensor] = {}
        self.out: Dict[str, torch.Tensor] = {}
        self.lse: Dict[str, torch.Tensor] = {}
        for name in w.layers:
            self.idx[name] = torch.empty((nq, w.topk), dtype=torch.int32, device=dev)
            self.count[name] = torch.empty(nq, dtype=torch.int32, device=dev)
            self.out[name] = torch.empty((nq, w.n_heads, 512), dtype=torch.bfloat16, device=dev)
            self.lse[name] = torch.empty((nq, w.n_heads), dtype=torch.float32, device=dev)
        self.blocks = torch.empty((nq, w.max_blocks), dtype=torch.int32, device=dev)
        self.nblocks = torch.empty(nq, dtype=torch.int32, device=dev)
        self.tail = None
        self.batches = {name: w.batch(name, rows) for name in w.layers}
        # per-layer per-row tensors restricted to the runner's rows, gathered
        # once here so that the call sequences launch only the library's kernels
        self._rows_t = {}
        if rows is not None:
            for name, L in w.layers.items():
                for attr in ("q", "q_fp4", "q_scale", "head_w", "win_lo", "given_idx"):
                    t = getattr(L, attr, None)
                    if t is not None:
                        self._rows_t[(name, attr)] = t[rows].contiguous()

    # ---- per-layer tensors restricted to the runner's rows -------------------
    def _lt(self, layer: str, attr: str):
        t = getattr(self.w.layers[layer], attr)
        if t is None or self.rows is None:
            return t
        got = self._rows_t.get((layer, attr))
        return got if got is not None else t[self.rows].contiguous()

    # ---- a1 -------------------------------------------------------------------
    def tail_layout(self):
        w = self.w
        r = w.num_req
        if self.tail is None:
            cap = r * w.replay
            self.tail = dict(tail_len=torch.empty(r, dtype=torch.int32, device=self.dev),
                             cu_tail=torch.empty(r + 1, dtype=torch.int32, device=self.dev),
                             src_row=torch.empty(cap, dtype=torch.int32, device=self.dev),
                             pos=torch.empty(cap, dtype=torch.int64, device=self.dev),
                             win_lo=torch.empty(cap, dtype=torch.int64, device=self.dev),
                             row_req=torch.empty(cap, dtype=torch.int32, device=self.dev))
        t = self.tail
        # the tail keeps R = w.replay rows per request; attention keeps the SWA
        # width w.window
        _check(csa2_tail_layout(r, w.extend_len, w.seq_len, w.replay, t["tail_len"], t["cu_tail"],
                                t["src_row"], t["pos"], t["win_lo"], t["row_req"], r * w.replay,
                                self.d_err), "csa2_tail_layout")
        return t

    def use_tail_rows(self):
        """Point every layer's batch at the tail layout's rows (positions and
        requests straight from csa2_tail_layout, nothing renumbered)."""
        t = self.tail
        for name, b in self.batches.items():
            b["q_pos"] = t["pos"][:self.nq]
            b["q_req"] = t["row_req"][:self.nq]
        self.tail_win_lo = t["win_lo"][:self.nq]

    # ---- a2-a7 ----------------------------------------------------------------
    def score_full(self, layer: str):
        w = self.w
        _check(csa2_index_score(self.batches[layer], w.n_idx_heads, 128, self._lt(layer, "q_fp4"),
                                self._lt(layer, "q_scale"), self._lt(layer, "head_w"),
                                w.pool.k_fp4, w.pool.k_scale, None, w.block, w.max_blocks,
                                self.scores, self.scores.shape[1], self.d_err),
               "csa2_index_score")
        return self.scores

    def score_pool(self, layer: str, blocks: torch.Tensor):
        w = self.w
        _check(csa2_index_score(self.batches[layer], w.n_idx_heads, 128, self._lt(layer, "q_fp4"),
                                self._lt(layer, "q_scale"), self._lt(layer, "head_w"),
                                w.pool.k_fp4, w.pool.k_scale, blocks, w.block, blocks.shape[1],
                                self.pool_scores, self.pool_scores.shape[1], self.d_err),
               "csa2_index_score")
        return self.pool_scores

    def select(self, layer: str, scores: torch.Tensor, blocks: Optional[torch.Tensor] = None):
        w = self.w
        _check(csa2_topk(self.batches[layer], scores, scores.shape[1], w.topk, blocks, w.block,
                         w.max_blocks if blocks is None else blocks.shape[1], self.idx[layer],
                         self.count[layer], self.d_err), "csa2_topk")
        return self.idx[layer], self.count[layer]

    def select_candidates(self, layer: str, scores: torch.Tensor):
        w = self.w
        _check(csa2_topk_candidates(self.batches[layer], scores, scores.shape[1], w.topk, w.block,
                                    w.max_blocks, self.idx[layer], self.count[layer], self.blocks,
                                    self.nblocks, self.d_err), "csa2_topk_candidates")
        return self.idx[layer], self.count[layer], self.blocks, self.nblocks

    # ---- a8-a10 -----------------------------------------------------------------
    def attend(self, layer: str, idx: Optional[torch.Tensor], win_lo=None, events=None):
        """Attention of `layer`; when `events` is a list, the launch is bracketed
        by CUDA events on the current stream and the pair is appended."""
        w = self.w
        L = w.layers[layer]
        if win_lo is None and L.win_lo is not None:
            win_lo = self._lt(layer, "win_lo")
        if events is not None:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
        _check(csa2_sparse_swa_attn(self.batches[layer], w.n_heads, 512, self._lt(layer, "q"),
                                    w.pool.kv_fp8, w.pool.kv_scale, idx,
                                    0 if idx is None else idx.shape[1], L.swa_fp8, L.swa_scale,
                                    win_lo, w.window, w.sm_scale, None, self.out[layer],
                                    self.lse[layer], self.d_err), "csa2_sparse_swa_attn")
        if events is not None:
            e1.record()
            events.append((e0, e1))
        return self.out[layer], self.lse[layer]

    # ---- whole layers -------------------------------------------------------------
    def full_layer(self, layer: str, events=None):
        """Score, select and attend.  When `events` is a dict, each launch is
        bracketed by CUDA events on the current stream, appended under
        "score", "select" and "attend"."""
        def timed(kind, fn):
            if events is None:
                return fn()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            r = fn()
            e1.record()
            events.setdefault(kind, []).append((e0, e1))
            return r
        s = timed("score", lambda: self.score_full(layer))
        idx, _ = timed("select", lambda: self.select(layer, s))
        return timed("attend", lambda: self.attend(layer, idx))

    def source_layer(self, layer: str, win_lo=None, events=None):
        s = self.score_full(layer)
        idx, _, blocks, _ = self.select_candidates(layer, s)
        self.attend(layer, idx, win_lo, events)
        return blocks

    def reindex_layer(self, layer: str, blocks: Optional[torch.Tensor], win_lo=None, events=None):
        s = self.score_pool(layer, blocks) if blocks is not None else self.score_full(layer)
        idx, _ = self.select(layer, s, blocks)
        self.attend(layer, idx, win_lo, events)
        return idx

    def reuse_layer(self, layer: str, idx: torch.Tensor, win_lo=None, events=None):
        return self.attend(layer, idx, win_lo, events)

    def decoder_tail_step(self, events=None):
        """Decoder bounded replay over the tail rows: tail layout, then the
        L20-style source pass (normal window), the L21-style Reindex layer in the
        published pool and the L22-style Reuse layer (both with the tail's window
        lower bounds)."""
        self.tail_layout()
        self.use_tail_rows()
        blocks = self.source_layer("L20", None, events)
        idx = self.reindex_layer("L21", blocks, self.tail_win_lo, events)
        self.reuse_layer("L22", idx, self.tail_win_lo, events)
