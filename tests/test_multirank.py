"""The N > 1 bench path on CPU: gloo, world size 2.  Every rank runs its own
replica (no data-path collective); the step time is the max over ranks and the
value counts every rank's rows."""
import os

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]
    agg = bench.max_over_ranks(ms, torch.device("cpu"), world)
    value = bench.layer_queries_per_s(rows=1024, world=world, ms=agg)
    out[rank] = (agg, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_max_time_and_total_rows():
    port = 29000 + os.getpid() % 1000
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for r in range(2):
        agg, value = out[r]
        assert agg == 5.0
        assert abs(value - 3 * 1024 * 2 / 5e-3) < 1e-6


def _rows_out(w, rows):
    """The oracle's Full layer (score, top-K, attention) on query rows `rows`."""
    import numpy as np
    from oracle import api as O
    from tests.helpers import np_batch, npy
    L = w.layers["full"]
    ri = torch.as_tensor(rows, dtype=torch.int64)
    b = np_batch(w.batch("full", ri))
    s, _ = O.index_score(b, npy(L.q_fp4[ri]), npy(L.q_scale[ri]), npy(L.head_w[ri]),
                         npy(w.pool.k_fp4), npy(w.pool.k_scale), w.ld)
    idx, cnt, _ = O.topk(b, np.nan_to_num(s, nan=-np.inf), w.topk)
    o, lse, _ = O.sparse_swa_attn(b, npy(L.q[ri]), npy(w.pool.kv_fp8), npy(w.pool.kv_scale),
                                  idx, npy(L.swa_fp8), npy(L.swa_scale), None, w.window,
                                  w.sm_scale)
    return idx, o, lse


def _split_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from sparse_attention_prefill_gb300 import synth
    w = synth.full_layer(1200, 2, list(range(0, 1200, 9)), 16, 8, seed=4, tag="split")
    rows = bench.partition_rows(w.num_q, rank, world)
    idx, o, lse = _rows_out(w, rows)
    got = [None] * world
    dist.all_gather_object(got, (rows, idx, o, lse))
    if rank == 0:
        out["parts"] = got
        out["num_q"] = w.num_q
    ms = [4.0, 6.0][rank]
    agg = bench.max_over_ranks(ms, torch.device("cpu"), world)
    out[rank] = bench.split_queries_per_s(w.num_q, 1, agg)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_row_split_covers_the_batch_and_matches_one_rank():
    """The headline's N > 1 path: the query rows of one batch split over two
    gloo ranks (row i on rank i mod 2, pool replicated, no data-path
    collective).  Every row is owned by exactly one rank; the per-rank oracle
    results, reassembled, equal a single-rank run over all rows; the value
    counts the batch's rows once over the slowest rank's time."""
    import numpy as np
    from sparse_attention_prefill_gb300 import synth
    port = 29500 + os.getpid() % 1000
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_split_worker, args=(2, port, out), nprocs=2, join=True)
    nq = out["num_q"]
    owner = np.full(nq, -1)
    for r, (rows, _, _, _) in enumerate(out["parts"]):
        assert (owner[rows] == -1).all()
        owner[rows] = r
    assert (owner >= 0).all()
    w = synth.full_layer(1200, 2, list(range(0, 1200, 9)), 16, 8, seed=4, tag="split")
    idx, o, lse = _rows_out(w, list(range(nq)))
    for rows, pi, po, pl in out["parts"]:
        assert (pi == idx[rows]).all()
        assert (po == o[rows]).all()
        assert np.array_equal(pl, lse[rows])
    for r in range(2):
        assert abs(out[r] - nq / 6e-3) < 1e-6
