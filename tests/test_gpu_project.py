"""Index keys projected from the compressed main KV and written as MXFP4
cache rows (csa2_index_k_project) against the oracle.

Codes and scales must be bit-exact where the projection is exact whatever the
order of the fp32 accumulation (small-integer operands).  On N(0,1) operands
the tensor core's fp32 accumulation may differ from the once-rounded exact
sum by a few units in the last place; a code or scale may then differ only
where that difference can cross a decision of the MXFP4 recipe: an element
within the accumulation bound of an E2M1 rounding boundary, or a group whose
largest magnitude is within the bound of a power of two (its scale)."""
import numpy as np
import pytest
import torch

import sparse_attention_prefill_gb300 as S
from oracle import api as O

pytestmark = pytest.mark.gpu
DEV = "cuda"
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
MIDS = (E2M1[1:] + E2M1[:-1]) / 2          # rounding boundaries of |x / scale|
ACC_REL = 2.0 ** -17                        # fp32 accumulation bound, relative to sum |x w|


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _run(x, w, dst, rows):
    codes = torch.full((rows, 64), 0x5A, dtype=torch.uint8, device=DEV)
    scales = torch.full((rows, 4), 7.0, dtype=torch.float32, device=DEV)
    ref = O.index_k_project(_bits(x), _bits(w), dst.cpu().numpy(), codes.cpu().numpy(),
                            scales.cpu().numpy())
    d_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    S.index_k_project(x, w, dst, codes, scales, d_err=d_err)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy(), int(d_err.item()), ref


def _nibbles(c):
    return np.stack([c & 15, c >> 4], -1).reshape(c.shape[0], -1)


def test_exact_operands_bit_exact():
    g = torch.Generator().manual_seed(0)
    n = 1000                                      # 7 full tiles and a ragged one
    x = torch.randint(-2, 3, (n, 512), generator=g).to(torch.bfloat16).to(DEV)
    w = (torch.randint(-2, 3, (128, 512), generator=g) / 8).to(torch.bfloat16).to(DEV)
    dst = torch.randperm(n + 24, generator=g)[:n].to(torch.int64).to(DEV)
    codes, scales, err, (rc, rs, _, rerr) = _run(x, w, dst, n + 24)
    assert err == rerr == 0
    assert np.array_equal(codes, rc) and np.array_equal(scales, rs)


@pytest.mark.parametrize("n", [1, 127, 4096 + 77])
def test_normal_operands_exact_but_for_decision_boundaries(n):
    g = torch.Generator().manual_seed(n)
    x = torch.randn((n, 512), generator=g).to(torch.bfloat16).to(DEV)
    w = (torch.randn((128, 512), generator=g) / 512 ** 0.5).to(torch.bfloat16).to(DEV)
    dst = torch.arange(n, dtype=torch.int64, device=DEV)
    codes, scales, err, (rc, rs, y, rerr) = _run(x, w, dst, n)
    assert err == rerr == 0
    xv, wv = x.double().cpu().numpy(), w.double().cpu().numpy()
    tol = ACC_REL * (np.abs(xv) @ np.abs(wv).T)           # per element, [n, 128]
    exceptions = 0
    gn, rn = _nibbles(codes), _nibbles(rc)
    for i in range(n):
        for gi in range(4):
            sl = slice(32 * gi, 32 * gi + 32)
            yv, tv = y[i, sl].astype(np.float64), tol[i, sl]
            amax = np.abs(yv).max()
            if scales[i, gi] != rs[i, gi]:
                # the scale's binade decision: amax within the bound of 2^e
                e = np.floor(np.log2(amax))
                assert min(abs(amax - 2.0 ** e), abs(2.0 ** (e + 1) - amax)) <= tv.max(), (i, gi)
                exceptions += 1
                continue
            diff = np.nonzero(gn[i, sl] != rn[i, sl])[0]
            for d in diff:
                q = abs(yv[d]) / rs[i, gi]
                near = np.abs(MIDS - q).min() <= tv[d] / rs[i, gi]
                near = near or (abs(yv[d]) <= tv[d])               # sign of a near-zero value
                assert near, (i, gi, d, yv[d], rs[i, gi])
                exceptions += 1
    print("index_k_project: %d rows, %d groups, %d boundary exceptions" % (n, 4 * n, exceptions))


def test_skipped_and_flagged_rows():
    g = torch.Generator().manual_seed(5)
    x = torch.randn((300, 512), generator=g).to(torch.bfloat16).to(DEV)
    w = (torch.randn((128, 512), generator=g) / 16).to(torch.bfloat16).to(DEV)
    dst = torch.arange(300, dtype=torch.int64)
    dst[::7] = -1
    dst[5] = 10 ** 6
    codes, scales, err, (rc, rs, _, rerr) = _run(x, w, dst.to(DEV), 300)
    assert err == rerr == S.DERR_RANGE_ROW
    untouched = [int(r) for r in range(300) if r not in set(dst.tolist())]
    assert (codes[untouched] == 0x5A).all() and (scales[untouched] == 7.0).all()
