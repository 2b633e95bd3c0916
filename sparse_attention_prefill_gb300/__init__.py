"""Python binding of libcsa2 -- the CSA2 attention layer on one GB300.

The functions named ``csa2_*`` mirror the C ABI of ``include/csa2.h`` one to
one: they take torch CUDA tensors (or None), pass their data pointers, sizes
and the current CUDA stream to the library, and return its status code.  The
short names (``tail_layout``, ``index_score``, ``topk``, ``topk_candidates``,
``sparse_swa_attn``) only allocate the output tensors with torch and call the
``csa2_*`` function.  Every step of the layer runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback: if the library cannot be loaded
or no GPU is present, the calls raise.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libcsa2.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_TOO_LARGE = 0, 1, 2, 3, 4, 5
DERR_RANGE_IDX, DERR_RANGE_WINDOW, DERR_RANGE_CTX = 1, 2, 4
DERR_SCALE, DERR_LD, DERR_CAPACITY, DERR_BAD_EXTEND = 8, 16, 32, 64
DERR_TIMEOUT, DERR_RANGE_ROW, DERR_NONFINITE = 128, 256, 512
FMT_FP8_B32, FMT_FP4KV, FMT_MXFP4 = 1, 2, 3

EXPORTED = ("csa2_status_string", "csa2_tail_layout", "csa2_index_score", "csa2_topk",
            "csa2_topk_candidates", "csa2_sparse_swa_attn", "csa2_sparse_swa_attn_fp4kv",
            "csa2_encoder_replay_layout", "csa2_rows_gather", "csa2_rows_scatter",
            "csa2_quantize_rows", "csa2_set_wait_limit_ns", "csa2_index_topk_workspace",
            "csa2_index_topk", "csa2_index_k_project", "csa2_index_topk_static_capacity",
            "csa2_index_topk_static")


class Csa2Error(RuntimeError):
    pass


class CBatch(C.Structure):
    _fields_ = [("num_q", C.c_int32), ("num_req", C.c_int32), ("ratio", C.c_int32),
                ("reserved", C.c_int32),
                ("q_req", C.c_void_p), ("q_pos", C.c_void_p),
                ("kv_start", C.c_void_p), ("kv_len", C.c_void_p),
                ("swa_start", C.c_void_p), ("swa_pos0", C.c_void_p), ("swa_len", C.c_void_p)]


_lib = None


def load(path: Optional[str] = None):
    """Load libcsa2.so (built by ``sparse_attention_prefill_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise Csa2Error("libcsa2.so not found at %s: run sparse_attention_prefill_gb300.build.build()"
                        % path)
    lib = C.CDLL(path)
    vp, i32, i64, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_float
    lib.csa2_status_string.restype = C.c_char_p
    lib.csa2_status_string.argtypes = [C.c_int]
    lib.csa2_tail_layout.argtypes = [i32, vp, vp, i32, vp, vp, vp, vp, vp, vp, i64, vp, vp]
    lib.csa2_index_score.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp, i32, i32, vp, i64,
                                     vp, vp]
    lib.csa2_topk.argtypes = [vp, vp, i64, i32, vp, i32, i32, vp, vp, vp, vp]
    lib.csa2_topk_candidates.argtypes = [vp, vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    lib.csa2_sparse_swa_attn.argtypes = [vp, i32, i32, vp, vp, vp, vp, i32, vp, vp, vp, i32, f32,
                                         vp, vp, vp, vp, vp]
    lib.csa2_sparse_swa_attn_fp4kv.argtypes = lib.csa2_sparse_swa_attn.argtypes
    lib.csa2_encoder_replay_layout.argtypes = [i32, vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp,
                                               i64, vp, vp]
    lib.csa2_rows_gather.argtypes = [vp, i64, vp, vp, i64, vp, i64, vp, vp]
    lib.csa2_rows_scatter.argtypes = [vp, i64, vp, vp, vp, i64, i64, vp, vp]
    lib.csa2_quantize_rows.argtypes = [i32, i64, vp, i32, vp, vp, vp, i64, vp, vp]
    lib.csa2_set_wait_limit_ns.argtypes = [C.c_uint64]
    lib.csa2_index_topk_workspace.argtypes = [i32, i64, vp]
    lib.csa2_index_k_project.argtypes = [i64, vp, i32, vp, i32, vp, vp, vp, i64, vp, vp]
    lib.csa2_index_topk_static_capacity.argtypes = [vp]
    lib.csa2_index_topk_static.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, i64, i32, vp, vp,
                                           vp, vp]
    lib.csa2_index_topk.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, i64, i32, vp, vp, vp, i64,
                                    vp, vp]
    for name in EXPORTED[1:]:
        getattr(lib, name).restype = C.c_int
    _lib = lib
    return lib


def csa2_index_topk_workspace(num_q, max_len) -> int:
    """Workspace bytes csa2_index_topk needs for num_q rows of at most max_len
    visible entries."""
    out = C.c_int64(0)
    _check(load().csa2_index_topk_workspace(int(num_q), int(max_len), C.byref(out)),
           "csa2_index_topk_workspace")
    return int(out.value)


def csa2_index_topk(batch, n_heads, head_dim, q_fp4, q_scale, head_w, k_fp4, k_scale, max_len,
                    k, idx, count, workspace, workspace_bytes, d_err, stream=None) -> int:
    st, keep = make_batch(batch)
    return load().csa2_index_topk(C.byref(st), int(n_heads), int(head_dim), _ptr(q_fp4),
                                  _ptr(q_scale), _ptr(head_w), _ptr(k_fp4), _ptr(k_scale),
                                  int(max_len), int(k), _ptr(idx), _ptr(count), _ptr(workspace),
                                  int(workspace_bytes), _ptr(d_err), _stream(stream))


def csa2_index_topk_static_capacity() -> int:
    """Bytes of the fixed scratch array csa2_index_topk_static uses."""
    out = C.c_int64(0)
    _check(load().csa2_index_topk_static_capacity(C.byref(out)), "csa2_index_topk_static_capacity")
    return int(out.value)


def csa2_index_topk_static(batch, n_heads, head_dim, q_fp4, q_scale, head_w, k_fp4, k_scale,
                           max_len, k, idx, count, d_err, stream=None) -> int:
    """csa2_index_topk with the library's fixed scratch array instead of a
    workspace (for callers that cannot allocate device memory)."""
    st, keep = make_batch(batch)
    return load().csa2_index_topk_static(C.byref(st), int(n_heads), int(head_dim), _ptr(q_fp4),
                                         _ptr(q_scale), _ptr(head_w), _ptr(k_fp4), _ptr(k_scale),
                                         int(max_len), int(k), _ptr(idx), _ptr(count),
                                         _ptr(d_err), _stream(stream))


def csa2_index_k_project(n, x_bf16, dim_in, w_bf16, dim_out, dst_row, k_fp4, k_scale, rows,
                         d_err, stream=None) -> int:
    return load().csa2_index_k_project(int(n), _ptr(x_bf16), int(dim_in), _ptr(w_bf16),
                                       int(dim_out), _ptr(dst_row), _ptr(k_fp4), _ptr(k_scale),
                                       int(rows), _ptr(d_err), _stream(stream))


def index_k_project(x, w, dst_row, k_fp4, k_scale, d_err=None, stream=None):
    """Project bf16 rows x [n, 512] by bf16 weights w [128, 512] and write the
    results as MXFP4 index-key rows dst_row of (k_fp4 [rows, 64], k_scale
    [rows, 4]) in place."""
    _check(csa2_index_k_project(x.shape[0], x, x.shape[1], w, w.shape[0], dst_row, k_fp4,
                                k_scale, k_fp4.shape[0], d_err, stream), "csa2_index_k_project")


def csa2_set_wait_limit_ns(ns: int) -> int:
    """Bound on the tensor-core kernels' pipeline waits for later launches
    (0 restores the default, 2 s)."""
    return load().csa2_set_wait_limit_ns(int(ns))


set_wait_limit_ns = csa2_set_wait_limit_ns


def status_string(status: int) -> str:
    return load().csa2_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise Csa2Error("libcsa2 takes device tensors; got a %s tensor" % t.device)
    if not t.is_contiguous():
        raise Csa2Error("libcsa2 takes contiguous tensors")
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _check(status: int, what: str):
    if status != OK:
        raise Csa2Error("%s: %s (status %d)" % (what, status_string(status), status))
    return status


def make_batch(b: dict):
    """Host struct for a batch dict of device tensors (see synth.Workload.batch).
    Returns (struct, keepalive)."""
    keep = {k: b[k] for k in ("q_req", "q_pos", "kv_start", "kv_len", "swa_start", "swa_pos0",
                              "swa_len")}
    st = CBatch(int(b["num_q"]), int(b["num_req"]), int(b["ratio"]), 0,
                *[_ptr(keep[k]) for k in ("q_req", "q_pos", "kv_start", "kv_len", "swa_start",
                                          "swa_pos0", "swa_len")])
    return st, keep


# ---------------------------------------------------------------------------
# one-to-one mirrors of the C ABI
# ---------------------------------------------------------------------------

def csa2_tail_layout(num_req, extend_len, seq_len, window, tail_len, cu_tail, src_row, pos,
                     win_lo, row_req, capacity, d_err, stream=None) -> int:
    return load().csa2_tail_layout(int(num_req), _ptr(extend_len), _ptr(seq_len), int(window),
                                   _ptr(tail_len), _ptr(cu_tail), _ptr(src_row), _ptr(pos),
                                   _ptr(win_lo), _ptr(row_req), int(capacity), _ptr(d_err),
                                   _stream(stream))


def csa2_index_score(batch, n_heads, head_dim, q_fp4, q_scale, head_w, k_fp4, k_scale,
                     cand_blocks, block, max_blocks, scores, ld, d_err, stream=None) -> int:
    st, keep = make_batch(batch)
    return load().csa2_index_score(C.byref(st), int(n_heads), int(head_dim), _ptr(q_fp4),
                                   _ptr(q_scale), _ptr(head_w), _ptr(k_fp4), _ptr(k_scale),
                                   _ptr(cand_blocks), int(block), int(max_blocks), _ptr(scores),
                                   int(ld), _ptr(d_err), _stream(stream))


def csa2_topk(batch, scores, ld, k, cand_blocks, block, max_blocks, idx, count, d_err,
              stream=None) -> int:
    st, keep = make_batch(batch)
    return load().csa2_topk(C.byref(st), _ptr(scores), int(ld), int(k), _ptr(cand_blocks),
                            int(block), int(max_blocks), _ptr(idx), _ptr(count), _ptr(d_err),
                            _stream(stream))


def csa2_topk_candidates(batch, scores, ld, k, block, max_blocks, idx, count, blocks, nblocks,
                         d_err, stream=None) -> int:
    st, keep = make_batch(batch)
    return load().csa2_topk_candidates(C.byref(st), _ptr(scores), int(ld), int(k), int(block),
                                       int(max_blocks), _ptr(idx), _ptr(count), _ptr(blocks),
                                       _ptr(nblocks), _ptr(d_err), _stream(stream))


def csa2_sparse_swa_attn(batch, n_heads, dim, q_bf16, kv_fp8, kv_scale, idx, k, swa_fp8,
                         swa_scale, win_lo, window, sm_scale, sink, out_bf16, lse, d_err,
                         stream=None) -> int:
    st, keep = make_batch(batch)
    return load().csa2_sparse_swa_attn(C.byref(st), int(n_heads), int(dim), _ptr(q_bf16),
                                       _ptr(kv_fp8), _ptr(kv_scale), _ptr(idx), int(k),
                                       _ptr(swa_fp8), _ptr(swa_scale), _ptr(win_lo), int(window),
                                       float(sm_scale), _ptr(sink), _ptr(out_bf16), _ptr(lse),
                                       _ptr(d_err), _stream(stream))


def csa2_sparse_swa_attn_fp4kv(batch, n_heads, dim, q_bf16, kv_fp4, kv_sf, idx, k, swa_fp8,
                               swa_scale, win_lo, window, sm_scale, sink, out_bf16, lse, d_err,
                               stream=None) -> int:
    st, keep = make_batch(batch)
    return load().csa2_sparse_swa_attn_fp4kv(C.byref(st), int(n_heads), int(dim), _ptr(q_bf16),
                                             _ptr(kv_fp4), _ptr(kv_sf), _ptr(idx), int(k),
                                             _ptr(swa_fp8), _ptr(swa_scale), _ptr(win_lo),
                                             int(window), float(sm_scale), _ptr(sink),
                                             _ptr(out_bf16), _ptr(lse), _ptr(d_err),
                                             _stream(stream))


# ---------------------------------------------------------------------------
def csa2_encoder_replay_layout(num_req, prefix_len, extend_len, window, ratio, replay_len,
                               cu_rows, src_row, pos, win_lo, row_req, entry_range, capacity,
                               d_err, stream=None) -> int:
    return load().csa2_encoder_replay_layout(
        int(num_req), _ptr(prefix_len), _ptr(extend_len), int(window), int(ratio),
        _ptr(replay_len), _ptr(cu_rows), _ptr(src_row), _ptr(pos), _ptr(win_lo), _ptr(row_req),
        _ptr(entry_range), int(capacity), _ptr(d_err), _stream(stream))


def csa2_rows_gather(count, capacity, row_idx, src, src_rows, dst, row_bytes, d_err,
                     stream=None) -> int:
    return load().csa2_rows_gather(_ptr(count), int(capacity), _ptr(row_idx), _ptr(src),
                                   int(src_rows), _ptr(dst), int(row_bytes), _ptr(d_err),
                                   _stream(stream))


def csa2_rows_scatter(count, capacity, row_idx, src, dst, dst_rows, row_bytes, d_err,
                      stream=None) -> int:
    return load().csa2_rows_scatter(_ptr(count), int(capacity), _ptr(row_idx), _ptr(src),
                                    _ptr(dst), int(dst_rows), int(row_bytes), _ptr(d_err),
                                    _stream(stream))


def csa2_quantize_rows(fmt, n, src, dim, dst_row, codes, scales, rows, d_err,
                       stream=None) -> int:
    return load().csa2_quantize_rows(int(fmt), int(n), _ptr(src), int(dim), _ptr(dst_row),
                                     _ptr(codes), _ptr(scales), int(rows), _ptr(d_err),
                                     _stream(stream))


# allocating conveniences (torch allocates the outputs; the library computes)
# ---------------------------------------------------------------------------

def tail_layout(extend_len, seq_len, window=128, d_err=None, stream=None):
    r = int(extend_len.shape[0])
    dev = extend_len.device
    cap = max(1, r * window)
    out = dict(tail_len=torch.empty(r, dtype=torch.int32, device=dev),
               cu_tail=torch.empty(r + 1, dtype=torch.int32, device=dev),
               src_row=torch.empty(cap, dtype=torch.int32, device=dev),
               pos=torch.empty(cap, dtype=torch.int64, device=dev),
               win_lo=torch.empty(cap, dtype=torch.int64, device=dev),
               row_req=torch.empty(cap, dtype=torch.int32, device=dev))
    _check(csa2_tail_layout(r, extend_len, seq_len, window, out["tail_len"], out["cu_tail"],
                            out["src_row"], out["pos"], out["win_lo"], out["row_req"], r * window,
                            d_err, stream), "csa2_tail_layout")
    return out


def encoder_replay_layout(prefix_len, extend_len, capacity, window=128, ratio=2, d_err=None,
                          stream=None):
    """Rows of an encoder extend over a cached prefix whose SWA state is gone:
    the last min(window, P) cached positions replayed, then the new ones.
    ``capacity`` bounds the rows written (sum of min(window, P) + E suffices)."""
    r = int(prefix_len.shape[0])
    dev = prefix_len.device
    cap = max(1, int(capacity))
    out = dict(replay_len=torch.empty(r, dtype=torch.int32, device=dev),
               cu_rows=torch.empty(r + 1, dtype=torch.int32, device=dev),
               src_row=torch.empty(cap, dtype=torch.int32, device=dev),
               pos=torch.empty(cap, dtype=torch.int64, device=dev),
               win_lo=torch.empty(cap, dtype=torch.int64, device=dev),
               row_req=torch.empty(cap, dtype=torch.int32, device=dev),
               entry_range=torch.empty((max(r, 1), 2), dtype=torch.int64, device=dev))
    _check(csa2_encoder_replay_layout(r, prefix_len, extend_len, window, ratio,
                                      out["replay_len"], out["cu_rows"], out["src_row"],
                                      out["pos"], out["win_lo"], out["row_req"],
                                      out["entry_range"], int(capacity), d_err, stream),
           "csa2_encoder_replay_layout")
    return out


def rows_gather(row_idx, src, dst, count=None, d_err=None, stream=None):
    """dst[i] = src[row_idx[i]] for i < count (device scalar) or len(row_idx);
    negative indices leave dst[i] as it was."""
    rb = src[0].numel() * src.element_size() if src.shape[0] else 0
    _check(csa2_rows_gather(count, int(row_idx.shape[0]), row_idx, src, int(src.shape[0]), dst,
                            rb, d_err, stream), "csa2_rows_gather")
    return dst


def rows_scatter(row_idx, src, dst, count=None, d_err=None, stream=None):
    """dst[row_idx[i]] = src[i] for i < count or len(row_idx); rows of dst
    that no index names keep their values."""
    rb = dst[0].numel() * dst.element_size() if dst.shape[0] else 0
    _check(csa2_rows_scatter(count, int(row_idx.shape[0]), row_idx, src, dst, int(dst.shape[0]),
                             rb, d_err, stream), "csa2_rows_scatter")
    return dst


def quantize_rows(fmt, src, dst_row, codes, scales, d_err=None, stream=None):
    """Quantise fp32 rows src [n, dim] into rows dst_row of a cache
    (codes, scales) in one of the FMT_* layouts; returns (codes, scales)."""
    n, dim = int(src.shape[0]), int(src.shape[1])
    _check(csa2_quantize_rows(fmt, n, src, dim, dst_row, codes, scales, int(codes.shape[0]),
                              d_err, stream), "csa2_quantize_rows")
    return codes, scales


def index_score(batch, q_fp4, q_scale, head_w, k_fp4, k_scale, ld, cand_blocks=None, block=8,
                max_blocks=2048, scores=None, d_err=None, stream=None):
    nq = int(batch["num_q"])
    if scores is None:
        scores = torch.empty((nq, int(ld)), dtype=torch.float32, device=q_fp4.device)
    if cand_blocks is not None:
        max_blocks = int(cand_blocks.shape[1])
    _check(csa2_index_score(batch, q_fp4.shape[1], q_fp4.shape[2] * 2, q_fp4, q_scale, head_w,
                            k_fp4, k_scale, cand_blocks, block, max_blocks, scores, ld, d_err,
                            stream), "csa2_index_score")
    return scores


def topk(batch, scores, k=512, cand_blocks=None, block=8, max_blocks=2048, d_err=None,
         stream=None):
    nq = int(batch["num_q"])
    dev = scores.device
    idx = torch.empty((nq, k), dtype=torch.int32, device=dev)
    count = torch.empty(nq, dtype=torch.int32, device=dev)
    if cand_blocks is not None:
        max_blocks = int(cand_blocks.shape[1])
    _check(csa2_topk(batch, scores, scores.shape[1], k, cand_blocks, block, max_blocks, idx, count,
                     d_err, stream), "csa2_topk")
    return idx, count


def topk_candidates(batch, scores, k=512, block=8, max_blocks=2048, d_err=None, stream=None):
    nq = int(batch["num_q"])
    dev = scores.device
    idx = torch.empty((nq, k), dtype=torch.int32, device=dev)
    count = torch.empty(nq, dtype=torch.int32, device=dev)
    blocks = torch.empty((nq, max_blocks), dtype=torch.int32, device=dev)
    nblocks = torch.empty(nq, dtype=torch.int32, device=dev)
    _check(csa2_topk_candidates(batch, scores, scores.shape[1], k, block, max_blocks, idx, count,
                                blocks, nblocks, d_err, stream), "csa2_topk_candidates")
    return idx, count, blocks, nblocks


def index_topk(batch, q_fp4, q_scale, head_w, k_fp4, k_scale, max_len, k, idx=None,
               count=None, workspace=None, d_err=None, stream=None):
    """Top-k entries of every query by index score, scored and selected in one
    streamed pass (no score rows).  Allocates the outputs and, if not given,
    the workspace (uint8, csa2_index_topk_workspace bytes)."""
    nq = int(batch["num_q"])
    dev = q_fp4.device
    if idx is None:
        idx = torch.empty((nq, int(k)), dtype=torch.int32, device=dev)
    if count is None:
        count = torch.empty(nq, dtype=torch.int32, device=dev)
    need = csa2_index_topk_workspace(nq, max_len)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check(csa2_index_topk(batch, q_fp4.shape[1], q_fp4.shape[2] * 2, q_fp4, q_scale, head_w,
                           k_fp4, k_scale, max_len, k, idx, count, workspace,
                           workspace.numel() * workspace.element_size(), d_err, stream),
           "csa2_index_topk")
    return idx, count


def sparse_swa_attn(batch, q, kv_fp8, kv_scale, idx, swa_fp8, swa_scale, win_lo=None, window=128,
                    sm_scale=None, sink=None, out=None, lse=None, want_lse=True, d_err=None,
                    stream=None):
    nq, n_heads, dim = q.shape
    if sm_scale is None:
        sm_scale = dim ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((nq, n_heads), dtype=torch.float32, device=q.device)
    k = 0 if idx is None else int(idx.shape[1])
    _check(csa2_sparse_swa_attn(batch, n_heads, dim, q, kv_fp8, kv_scale, idx, k, swa_fp8,
                                swa_scale, win_lo, window, sm_scale, sink, out, lse, d_err,
                                stream), "csa2_sparse_swa_attn")
    return out, lse


def sparse_swa_attn_fp4kv(batch, q, kv_fp4, kv_sf, idx, swa_fp8, swa_scale, win_lo=None,
                          window=128, sm_scale=None, sink=None, out=None, lse=None,
                          want_lse=True, d_err=None, stream=None):
    """Attention with the selected rows read from the FP4 main-KV pool
    (E2M1 codes [Nkv, 256] and E4M3 scales per 16 channels [Nkv, 32])."""
    nq, n_heads, dim = q.shape
    if sm_scale is None:
        sm_scale = dim ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((nq, n_heads), dtype=torch.float32, device=q.device)
    k = 0 if idx is None else int(idx.shape[1])
    _check(csa2_sparse_swa_attn_fp4kv(batch, n_heads, dim, q, kv_fp4, kv_sf, idx, k, swa_fp8,
                                      swa_scale, win_lo, window, sm_scale, sink, out, lse, d_err,
                                      stream), "csa2_sparse_swa_attn_fp4kv")
    return out, lse
