"""ctypes front end of the C oracle (test infrastructure only).

Every function takes host numpy arrays, allocates its outputs and returns
them together with the OR of the data-error bits the oracle raised.  The
batch description is a plain dict (see ``sparse_attention_prefill_gb300.synth``
for how workloads build it).
"""
import ctypes as C
import os

import numpy as np

from .build import build_oracle

_lib = None


class _Batch(C.Structure):
    _fields_ = [("num_q", C.c_int32), ("num_req", C.c_int32), ("ratio", C.c_int32),
                ("pad_", C.c_int32),
                ("q_req", C.c_void_p), ("q_pos", C.c_void_p),
                ("kv_start", C.c_void_p), ("kv_len", C.c_void_p),
                ("swa_start", C.c_void_p), ("swa_pos0", C.c_void_p),
                ("swa_len", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        # CSA2_ORACLE_LIB points the pins at another build of this file (the
        # mutation tests load deliberately broken copies through it)
        _lib = C.CDLL(os.environ.get("CSA2_ORACLE_LIB") or build_oracle())
        _lib.oracle_e2m1_value.restype = C.c_double
        _lib.oracle_e2m1_value.argtypes = [C.c_int]
        _lib.oracle_e4m3_value.restype = C.c_double
        _lib.oracle_e4m3_value.argtypes = [C.c_int]
        _lib.oracle_double_to_bf16.restype = C.c_uint16
        _lib.oracle_double_to_bf16.argtypes = [C.c_double]
        _lib.oracle_n_visible.restype = C.c_int64
        _lib.oracle_n_visible.argtypes = [C.c_int64, C.c_int]
        for name in ("oracle_tail_layout", "oracle_index_score", "oracle_topk",
                     "oracle_topk_candidates", "oracle_sparse_swa_attn",
                     "oracle_sparse_swa_attn_fp4kv", "oracle_encoder_replay_layout",
                     "oracle_rows_gather", "oracle_rows_scatter", "oracle_encode_rows",
                     "oracle_encode_e4m3", "oracle_encode_e2m1", "oracle_index_k_project"):
            getattr(_lib, name).restype = C.c_int
        _lib.oracle_decode_fp4kv_row.restype = None
        _lib.oracle_decode_mxfp4_row.restype = None
        _lib.oracle_encode_e4m3.argtypes = [C.c_double]
        _lib.oracle_encode_e2m1.argtypes = [C.c_double]
    return _lib


def set_threads(n: int) -> None:
    """Set the OpenMP thread count the oracle uses (``OMP_NUM_THREADS`` semantics)."""
    os.environ["OMP_NUM_THREADS"] = str(int(n))
    try:
        omp = C.CDLL("libgomp.so.1")
        omp.omp_set_num_threads(int(n))
    except OSError:
        pass


def _p(a):
    return None if a is None else C.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _batch(b):
    keep = {
        "q_req": _c(b["q_req"], np.int32), "q_pos": _c(b["q_pos"], np.int64),
        "kv_start": _c(b["kv_start"], np.int64), "kv_len": _c(b["kv_len"], np.int64),
        "swa_start": _c(b["swa_start"], np.int64), "swa_pos0": _c(b["swa_pos0"], np.int64),
        "swa_len": _c(b["swa_len"], np.int64),
    }
    st = _Batch(int(b["num_q"]), int(b["num_req"]), int(b["ratio"]), 0,
                *[_p(keep[k]) for k in ("q_req", "q_pos", "kv_start", "kv_len",
                                        "swa_start", "swa_pos0", "swa_len")])
    return st, keep


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(int(code))


def double_to_bf16(x: float) -> int:
    return int(lib().oracle_double_to_bf16(float(x)))


def n_visible(t: int, m: int) -> int:
    return int(lib().oracle_n_visible(int(t), int(m)))


def tail_layout(extend_len, seq_len, window=128, capacity=None):
    e = _c(extend_len, np.int32)
    s = _c(seq_len, np.int64)
    r = e.shape[0]
    if capacity is None:
        capacity = int(r * window)
    tail_len = np.zeros(r, np.int32)
    cu_tail = np.zeros(r + 1, np.int32)
    cap = max(int(capacity), 1)
    src_row = np.full(cap, -1, np.int32)
    pos = np.full(cap, -1, np.int64)
    win_lo = np.full(cap, -1, np.int64)
    row_req = np.full(cap, -1, np.int32)
    err = lib().oracle_tail_layout(C.c_int32(r), _p(e), _p(s), C.c_int32(window),
                                   _p(tail_len), _p(cu_tail), _p(src_row), _p(pos),
                                   _p(win_lo), _p(row_req), C.c_int64(capacity))
    n = min(int(cu_tail[-1]), int(capacity))
    return dict(tail_len=tail_len, cu_tail=cu_tail, src_row=src_row[:n], pos=pos[:n],
                win_lo=win_lo[:n], row_req=row_req[:n]), err


def encoder_replay_layout(prefix_len, extend_len, window=128, ratio=2, capacity=None):
    p = _c(prefix_len, np.int64)
    e = _c(extend_len, np.int32)
    r = p.shape[0]
    if capacity is None:
        capacity = int(sum(min(window, max(int(a), 0)) + max(int(b), 0) for a, b in zip(p, e)))
    replay_len = np.zeros(r, np.int32)
    cu_rows = np.zeros(r + 1, np.int32)
    cap = max(int(capacity), 1)
    src_row = np.full(cap, -2, np.int32)
    pos = np.full(cap, -1, np.int64)
    win_lo = np.full(cap, -1, np.int64)
    row_req = np.full(cap, -1, np.int32)
    entry_range = np.zeros((max(r, 1), 2), np.int64)
    err = lib().oracle_encoder_replay_layout(C.c_int32(r), _p(p), _p(e), C.c_int32(window),
                                             C.c_int32(ratio), _p(replay_len), _p(cu_rows),
                                             _p(src_row), _p(pos), _p(win_lo), _p(row_req),
                                             _p(entry_range), C.c_int64(capacity))
    n = min(int(cu_rows[-1]), int(capacity))
    return dict(replay_len=replay_len, cu_rows=cu_rows, src_row=src_row[:n], pos=pos[:n],
                win_lo=win_lo[:n], row_req=row_req[:n], entry_range=entry_range[:r]), err


def rows_gather(row_idx, src, dst):
    """dst[i] = src[row_idx[i]] (rows = leading axis); returns (new dst, err)."""
    idx = _c(row_idx, np.int32)
    s = np.ascontiguousarray(src)
    d = np.array(dst, copy=True, order="C")
    rb = int(s[0].nbytes) if s.shape[0] else int(d[0].nbytes)
    err = lib().oracle_rows_gather(C.c_int64(idx.shape[0]), _p(idx), _p(s),
                                   C.c_int64(s.shape[0]), _p(d), C.c_int64(rb))
    return d, err


def rows_scatter(row_idx, src, dst):
    """dst[row_idx[i]] = src[i]; rows not named keep their values."""
    idx = _c(row_idx, np.int32)
    s = np.ascontiguousarray(src)
    d = np.array(dst, copy=True, order="C")
    rb = int(d[0].nbytes) if d.shape[0] else 0
    err = lib().oracle_rows_scatter(C.c_int64(idx.shape[0]), _p(idx), _p(s), _p(d),
                                    C.c_int64(d.shape[0]), C.c_int64(rb))
    return d, err


FMT_FP8_B32, FMT_FP4KV, FMT_MXFP4 = 1, 2, 3


def encode_e4m3(x: float) -> int:
    return int(lib().oracle_encode_e4m3(float(x)))


def encode_e2m1(x: float) -> int:
    return int(lib().oracle_encode_e2m1(float(x)))


def encode_rows(fmt, src, dst_row, codes, scales):
    """Quantise rows of src (fp32 [n, dim]) into rows dst_row of (codes,
    scales) in place of copies; returns (codes, scales, err)."""
    x = _c(src, np.float32)
    n, dim = x.shape
    dr = _c(dst_row, np.int64)
    cd = np.array(codes, copy=True, order="C")
    sc = np.array(scales, copy=True, order="C")
    err = lib().oracle_encode_rows(C.c_int(fmt), C.c_int64(n), _p(x), C.c_int(dim), _p(dr),
                                   _p(cd), _p(sc), C.c_int64(cd.shape[0]))
    return cd, sc, err


def index_k_project(x_bf16, w_bf16, dst_row, codes, scales):
    """Index keys projected from bf16 rows x [n, dim_in] by bf16 weights w
    [dim_out, dim_in], written as MXFP4 rows dst_row of copies of (codes,
    scales).  Inputs are the raw bf16 bit patterns (uint16).  Returns (codes,
    scales, y fp32 [n, dim_out] before quantisation, err)."""
    x = _c(x_bf16, np.uint16)
    w = _c(w_bf16, np.uint16)
    n, dim_in = x.shape
    dim_out = w.shape[0]
    dr = _c(dst_row, np.int64)
    cd = np.array(codes, copy=True, order="C")
    sc = np.array(scales, copy=True, order="C")
    y = np.zeros((n, dim_out), np.float32)
    err = lib().oracle_index_k_project(C.c_int64(n), _p(x), C.c_int(dim_in), _p(w),
                                       C.c_int(dim_out), _p(dr), _p(cd), _p(sc),
                                       C.c_int64(cd.shape[0]), _p(y))
    return cd, sc, y, err


def index_score(b, q_fp4, q_scale, head_w, k_fp4, k_scale, ld,
                cand_blocks=None, block=8, max_blocks=2048, fill=np.nan):
    st, keep = _batch(b)
    qf, qs = _c(q_fp4, np.uint8), _c(q_scale, np.float32)
    kf, ks = _c(k_fp4, np.uint8), _c(k_scale, np.float32)
    hw = _c(head_w, np.float32)
    cb = _c(cand_blocks, np.int32)
    n_heads = qf.shape[1]
    head_dim = qf.shape[2] * 2
    if cb is not None:
        max_blocks = cb.shape[1]
    scores = np.full((int(b["num_q"]), int(ld)), fill, np.float32)
    err = lib().oracle_index_score(C.byref(st), C.c_int(n_heads), C.c_int(head_dim),
                                   _p(qf), _p(qs), _p(hw), _p(kf), _p(ks), _p(cb),
                                   C.c_int(block), C.c_int(max_blocks), _p(scores),
                                   C.c_int64(ld))
    return scores, err


def topk(b, scores, k=512, cand_blocks=None, block=8, max_blocks=2048):
    st, keep = _batch(b)
    sc = _c(scores, np.float32)
    cb = _c(cand_blocks, np.int32)
    if cb is not None:
        max_blocks = cb.shape[1]
    nq = int(b["num_q"])
    idx = np.full((nq, k), -7, np.int32)
    count = np.full(nq, -7, np.int32)
    err = lib().oracle_topk(C.byref(st), _p(sc), C.c_int64(sc.shape[1]), C.c_int(k),
                            _p(cb), C.c_int(block), C.c_int(max_blocks), _p(idx), _p(count))
    return idx, count, err


def topk_candidates(b, scores, k=512, block=8, max_blocks=2048):
    st, keep = _batch(b)
    sc = _c(scores, np.float32)
    nq = int(b["num_q"])
    idx = np.full((nq, k), -7, np.int32)
    count = np.full(nq, -7, np.int32)
    blocks = np.full((nq, max_blocks), -7, np.int32)
    nblocks = np.full(nq, -7, np.int32)
    err = lib().oracle_topk_candidates(C.byref(st), _p(sc), C.c_int64(sc.shape[1]),
                                       C.c_int(k), C.c_int(block), C.c_int(max_blocks),
                                       _p(idx), _p(count), _p(blocks), _p(nblocks))
    return idx, count, blocks, nblocks, err


def sparse_swa_attn(b, q_bf16, kv_fp8, kv_scale, idx, swa_fp8, swa_scale, win_lo=None,
                    window=128, sm_scale=None, sink=None, want_lse=True):
    """``q_bf16`` is a uint16 array of bf16 bit patterns [Nq, H, D]; the
    output is returned the same way."""
    st, keep = _batch(b)
    q = _c(q_bf16, np.uint16)
    nq, n_heads, dim = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(dim)
    kvf, kvs = _c(kv_fp8, np.uint8), _c(kv_scale, np.float32)
    sf, ss = _c(swa_fp8, np.uint8), _c(swa_scale, np.float32)
    ix = _c(idx, np.int32)
    k = 0 if ix is None else ix.shape[1]
    wl = _c(win_lo, np.int64)
    sk = _c(sink, np.float32)
    out = np.zeros((nq, n_heads, dim), np.uint16)
    lse = np.zeros((nq, n_heads), np.float32) if want_lse else None
    err = lib().oracle_sparse_swa_attn(C.byref(st), C.c_int(n_heads), C.c_int(dim), _p(q),
                                       _p(kvf), _p(kvs), _p(ix), C.c_int(k), _p(sf), _p(ss),
                                       _p(wl), C.c_int(window), C.c_double(sm_scale), _p(sk),
                                       _p(out), _p(lse))
    return out, lse, err


def sparse_swa_attn_fp4kv(b, q_bf16, kv_fp4, kv_sf, idx, swa_fp8, swa_scale, win_lo=None,
                          window=128, sm_scale=None, sink=None, want_lse=True):
    """As ``sparse_swa_attn`` with the selected rows taken from the FP4 main-KV
    pool: ``kv_fp4`` uint8 [Nkv, D/2] E2M1 pairs, ``kv_sf`` uint8 [Nkv, D/16]
    E4M3 scales (one per 16 channels)."""
    st, keep = _batch(b)
    q = _c(q_bf16, np.uint16)
    nq, n_heads, dim = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(dim)
    kvf, kvs = _c(kv_fp4, np.uint8), _c(kv_sf, np.uint8)
    sf, ss = _c(swa_fp8, np.uint8), _c(swa_scale, np.float32)
    ix = _c(idx, np.int32)
    k = 0 if ix is None else ix.shape[1]
    wl = _c(win_lo, np.int64)
    sk = _c(sink, np.float32)
    out = np.zeros((nq, n_heads, dim), np.uint16)
    lse = np.zeros((nq, n_heads), np.float32) if want_lse else None
    err = lib().oracle_sparse_swa_attn_fp4kv(C.byref(st), C.c_int(n_heads), C.c_int(dim), _p(q),
                                             _p(kvf), _p(kvs), _p(ix), C.c_int(k), _p(sf),
                                             _p(ss), _p(wl), C.c_int(window),
                                             C.c_double(sm_scale), _p(sk), _p(out), _p(lse))
    return out, lse, err


def decode_mxfp4_row(codes, scales):
    """One MXFP4 row decoded to float64 (codes uint8 [D/2], scales f32 [D/32])."""
    c, f = _c(codes, np.uint8), _c(scales, np.float32)
    dim = c.shape[-1] * 2
    out = np.zeros(dim, np.float64)
    lib().oracle_decode_mxfp4_row(_p(c), _p(f), C.c_int(dim), _p(out))
    return out


def decode_fp4kv_row(codes, sf):
    """One FP4 main-KV row decoded to float64 (codes uint8 [D/2], sf uint8 [D/16])."""
    c, f = _c(codes, np.uint8), _c(sf, np.uint8)
    dim = c.shape[-1] * 2
    out = np.zeros(dim, np.float64)
    lib().oracle_decode_fp4kv_row(_p(c), _p(f), C.c_int(dim), _p(out))
    return out
