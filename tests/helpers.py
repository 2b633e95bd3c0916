"""Test helpers: host copies of workloads for the oracle and parity metrics."""
import numpy as np
import torch

from oracle import api as O


def np_batch(b: dict) -> dict:
    out = {}
    for k, v in b.items():
        out[k] = v.detach().cpu().numpy() if torch.is_tensor(v) else v
    return out


def npy(t):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)
    return t.detach().cpu().numpy()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).double().numpy()


def attn_errors(gpu_bf16: torch.Tensor, ref_bits: np.ndarray):
    g = gpu_bf16.detach().float().cpu().double().numpy()
    r = bf16_to_f64(ref_bits)
    d = np.abs(g - r)
    return float(d.max() / max(np.abs(r).max(), 1e-30)), float(d.mean() / max(np.abs(r).mean(), 1e-30))


ATTN_MAX_REL = 2e-2
ATTN_MEAN_REL = 1e-3
# lse = ln sum_i e^{l_i}: its error is the softmax-weighted mean of the logit
# errors.  With f16 operands (dequantised rows and f16 scales: <= 2^-10
# relative per element) one unit-variance logit over 512 channels errs by
# sigma ~ 2^-11 * sm_scale * ||q o r||_2 ~ 5e-4 (less when many rows share the
# weight).  Bounds: 4 sigma for the worst element, sigma / 2 on average.
LSE_ABS_MAX = 2e-3
LSE_ABS_MEAN = 2.5e-4


def assert_attn_close(gpu_out, gpu_lse, ref_out, ref_lse):
    mx, mean = attn_errors(gpu_out, ref_out)
    assert mx <= ATTN_MAX_REL and mean <= ATTN_MEAN_REL, (mx, mean)
    if ref_lse is not None and gpu_lse is not None:
        gl = gpu_lse.detach().cpu().numpy()
        fin = np.isfinite(ref_lse)
        assert (np.isfinite(gl) == fin).all()
        d = np.abs(gl[fin] - ref_lse[fin])
        if d.size:
            assert d.max() <= LSE_ABS_MAX and d.mean() <= LSE_ABS_MEAN, (d.max(), d.mean())


def topk_sets_match(gpu_idx, gpu_count, ref_idx, ref_count):
    """Bit-exact comparison of selected sets (order within a row is free)."""
    gi = gpu_idx.detach().cpu().numpy()
    gc = gpu_count.detach().cpu().numpy()
    assert (gc == ref_count).all(), np.nonzero(gc != ref_count)[0][:10]
    for q in range(gi.shape[0]):
        c = int(ref_count[q])
        assert sorted(gi[q, :c].tolist()) == sorted(ref_idx[q, :c].tolist()), q
        assert (gi[q, c:] == -1).all(), q


def topk_near_tie_ok(gpu_idx, gpu_count, ref_idx, ref_count, ref_scores, entry_of_col=None,
                     rel=1e-3):
    """End-to-end top-K rule: sets equal except for swaps among entries whose
    oracle scores lie within rel * |s_k| of the oracle's k-th score.  Returns
    the positions of the rows whose sets differ (each one checked)."""
    gi = gpu_idx.detach().cpu().numpy()
    gc = gpu_count.detach().cpu().numpy()
    assert (gc == ref_count).all()
    rows = []
    for q in range(gi.shape[0]):
        c = int(ref_count[q])
        a, b = set(gi[q, :c].tolist()), set(ref_idx[q, :c].tolist())
        diff = a ^ b
        if not diff:
            continue
        row = ref_scores[q]
        col = (lambda e: e) if entry_of_col is None else (lambda e: entry_of_col[q][e])
        sk = min(row[col(e)] for e in b)
        for e in diff:
            assert abs(row[col(e)] - sk) <= rel * abs(sk) + 1e-30, (q, e, row[col(e)], sk)
        rows.append(q)
    return rows


def block_maxima(row: np.ndarray, n_vis: int, block: int) -> np.ndarray:
    """Maximum oracle score of each block of `block` entries over the first
    n_vis entries of a full-visible score row (NaN ignored)."""
    nb = -(-n_vis // block)
    r = np.full(nb * block, -np.inf)
    v = row[:n_vis].astype(np.float64)
    r[:n_vis] = np.where(np.isnan(v), -np.inf, v)
    return r.reshape(nb, block).max(1) if nb else r


def pool_near_tie_rows(gpu_blocks, gpu_nblocks, ref_blocks, ref_nblocks, ref_scores, block,
                       rel=1e-3):
    """End-to-end candidate pools: bit-exact per row.  A row may differ only
    when every block in the symmetric difference has an oracle block maximum
    within rel * |m_k| of m_k, the lowest block maximum the oracle kept among
    the ranked blocks (every block but the latest); the latest block must be
    in both pools.  `ref_scores` are the oracle's full-visible scores of the
    same rows (columns = entries; unwritten columns NaN).  Returns the
    positions of the rows that differ."""
    gb = npy(gpu_blocks) if torch.is_tensor(gpu_blocks) else gpu_blocks
    gn = npy(gpu_nblocks) if torch.is_tensor(gpu_nblocks) else gpu_nblocks
    assert (gn == ref_nblocks).all(), np.nonzero(gn != ref_nblocks)[0][:10]
    rows = []
    for q in range(gb.shape[0]):
        if (gb[q] == ref_blocks[q]).all():
            continue
        n = int(ref_nblocks[q])
        assert (gb[q, n:] == -1).all() and (np.diff(gb[q, :n]) > 0).all(), q
        n_vis = int((~np.isnan(ref_scores[q])).sum())
        latest = -(-n_vis // block) - 1
        a, b = set(gb[q, :n].tolist()), set(ref_blocks[q, :n].tolist())
        assert latest in a and latest in b, q
        bm = block_maxima(ref_scores[q], n_vis, block)
        mk = min(bm[x] for x in b if x != latest)
        for x in a ^ b:
            assert abs(bm[x] - mk) <= rel * abs(mk) + 1e-30, (q, x, bm[x], mk)
        rows.append(q)
    return rows
