"""Dense tensor-core throughput of this GPU for the operand kinds the layer
could contract in: f16 (kind::f16), E4M3 (kind::f8f6f4) and block-scaled
E2M1 (kind::mxf4, one UE8M0 scale per 32 elements).

The probe (`probe/mma_peak.cu`, its own shared library) keeps one M = 128 x
N = 256 operand pair in each SM's shared memory and issues back-to-back MMAs
into TMEM, so the rate measured is the tensor pipe's.  `check()` first runs one
round per kind and compares the accumulator with an exact host product, so a
rate is only reported for an MMA whose results are right.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict

import numpy as np
import torch

from . import build as _build

KINDS = {"f16": 0, "e4m3": 1, "e2m1_mx": 2}
ELEMS_PER_ROUND = {0: 64, 1: 128, 2: 256}     # K elements per round of four MMAs
M, N = 128, 256

# E2M1 magnitudes by code (OCP MX): used to synthesise operands and their values
_E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.PROBE_LIB
        if not os.path.exists(path):
            raise RuntimeError("probe library missing: run __graft_entry__.build() first")
        _lib = ctypes.CDLL(path)
        _lib.csa2probe_mma.restype = ctypes.c_int
        _lib.csa2probe_mma.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p]
    return _lib


def operands(kind: int, seed: int = 0):
    """Host operand bytes ([128][128 B], [256][128 B]) and their exact values
    ([128][K], [256][K] float64), K-major, small enough that every product and
    sum is exact in fp32."""
    rng = np.random.default_rng(seed + kind)
    if kind == 0:
        va = rng.integers(-8, 9, (M, 64)) / 4.0
        vb = rng.integers(-8, 9, (N, 64)) / 4.0
        ba = va.astype(np.float16).view(np.uint8).reshape(M, 128)
        bb = vb.astype(np.float16).view(np.uint8).reshape(N, 128)
        return ba, bb, va, vb
    if kind == 1:
        grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, -0.5, -1.0, -1.5, -2.0, -3.0])
        va = grid[rng.integers(0, len(grid), (M, 128))]
        vb = grid[rng.integers(0, len(grid), (N, 128))]
        ba = torch.from_numpy(va).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        bb = torch.from_numpy(vb).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        return ba, bb, va, vb

    def fp4(rows):
        codes = rng.integers(0, 16, (rows, 256)).astype(np.uint8)
        vals = _E2M1[codes & 7] * np.where(codes & 8, -1.0, 1.0)
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        return packed, vals

    ba, va = fp4(M)
    bb, vb = fp4(N)
    return ba, bb, va, vb


def _run(kind, iters, ctas, a, b, out, err):
    st = lib().csa2probe_mma(kind, iters, ctas, a.data_ptr(), b.data_ptr(),
                             0 if out is None else out.data_ptr(), err.data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    if st != 0:
        raise RuntimeError("probe launch failed (%d)" % st)


def check(kind: int, dev="cuda") -> float:
    """One round of four MMAs; returns the largest |GPU - exact| (0 expected)."""
    ba, bb, va, vb = operands(kind)
    a = torch.from_numpy(np.ascontiguousarray(ba)).to(dev)
    b = torch.from_numpy(np.ascontiguousarray(bb)).to(dev)
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    _run(kind, 1, 1, a, b, out, err)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError("probe wait timed out")
    ref = va @ vb.T
    return float(np.abs(out.cpu().double().numpy() - ref).max())


def measure(kind: int, dev="cuda", target_ms: float = 20.0, reps: int = 5) -> Dict:
    """Burst dense throughput (TFLOP/s) of one kind: every SM, back-to-back MMAs."""
    ba, bb, _, _ = operands(kind)
    a = torch.from_numpy(np.ascontiguousarray(ba)).to(dev)
    b = torch.from_numpy(np.ascontiguousarray(bb)).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    flops_per_round = 2 * M * N * ELEMS_PER_ROUND[kind]
    iters = 2000
    _run(kind, iters, ctas, a, b, None, err)           # warm-up and sizing
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    _run(kind, iters, ctas, a, b, None, err)
    e1.record()
    torch.cuda.synchronize()
    iters = max(2000, int(iters * target_ms / max(e0.elapsed_time(e1), 1e-3)))
    best = 0.0
    for _ in range(reps):
        e0.record()
        _run(kind, iters, ctas, a, b, None, err)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = max(best, ctas * iters * flops_per_round / (ms * 1e-3) / 1e12)
    if int(err.item()) != 0:
        raise RuntimeError("probe wait timed out")
    return {"tflops": round(best, 1), "iters": iters, "ctas": ctas,
            "shape": "M=128 N=256 per MMA, K=%d per round" % ELEMS_PER_ROUND[kind]}


def measure_all(dev="cuda") -> Dict[str, Dict]:
    out = {}
    for name, kind in KINDS.items():
        e = check(kind, dev)
        r = measure(kind, dev)
        r["max_abs_error_vs_exact"] = e
        out[name] = r
    return out


if __name__ == "__main__":
    import json
    torch.cuda.set_device(0)
    print(json.dumps(measure_all()))
