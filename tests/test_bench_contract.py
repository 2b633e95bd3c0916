"""The bench's reference arm (the oracle on the host cores) and its JSON line,
checked on the CPU: the keys the line must carry, and that under a multi-rank
launch only rank 0 prints."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, **env):
    e = dict(os.environ, **env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          env=e, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_complete_line():
    r = _run(["--impl", "reference", "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "unit", "dtype", "data", "scaling"):
        assert isinstance(d[key], str) and d[key]
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"] and cb["unit"] == d["unit"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_work():
    r = _run(["--impl", "reference", "--steps", "1", "--warmup", "0"], RANK="1", WORLD_SIZE="2",
             LOCAL_RANK="1")
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_cpulist_parsing_and_unknown_locality():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.parse_cpulist("72-143") == set(range(72, 144))
    assert bench.parse_cpulist("") == set()
    # without a GPU the locality is unknown and nothing is bound
    import torch
    if not torch.cuda.is_available():
        assert bench.gpu_local_cpus(0) == set()


def _tiny_batch(rng, nq=40, nreq=3, ratio=2):
    import torch
    kv_len = torch.tensor(rng.integers(0, 300, nreq), dtype=torch.int64)
    swa_pos0 = torch.tensor(rng.integers(0, 200, nreq), dtype=torch.int64)
    swa_len = torch.tensor(rng.integers(0, 300, nreq), dtype=torch.int64)
    q_req = torch.tensor(rng.integers(0, nreq, nq), dtype=torch.int32)
    q_pos = torch.tensor(rng.integers(0, 600, nq), dtype=torch.int64)
    return dict(num_q=nq, num_req=nreq, ratio=ratio, q_req=q_req, q_pos=q_pos,
                kv_start=torch.zeros(nreq, dtype=torch.int64), kv_len=kv_len,
                swa_start=torch.zeros(nreq, dtype=torch.int64), swa_pos0=swa_pos0,
                swa_len=swa_len)


def test_roofline_counts_match_brute_force():
    """The per-launch accounting of `bench.py --configs` (visible entries,
    stored window rows, pool pairs, attention bytes, index flops) against
    plain loops."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import bench
    rng = np.random.default_rng(7)
    for ratio in (1, 2):
        b = _tiny_batch(rng, ratio=ratio)
        nq = b["num_q"]
        win_lo = torch.tensor(rng.integers(0, 500, nq), dtype=torch.int64)
        window, block, k, heads = 128, 8, 16, 4
        blocks = torch.full((nq, 10), -1, dtype=torch.int32)
        idx = torch.tensor(rng.integers(-1, 400, (nq, k)), dtype=torch.int32)
        nv_ref, win_ref, pool_ref, sel_ref = [], [], [], 0
        for q in range(nq):
            r, t = int(b["q_req"][q]), int(b["q_pos"][q])
            nv = min((t + 1) // ratio, int(b["kv_len"][r]))
            nv_ref.append(nv)
            lo = max(int(win_lo[q]), t - window + 1, 0)
            p0, pn = int(b["swa_pos0"][r]), int(b["swa_len"][r])
            win_ref.append(sum(1 for p in range(lo, t + 1) if p0 <= p < p0 + pn))
            nb = int(rng.integers(0, 11))
            chosen = sorted(rng.choice(max(1, (nv + block - 1) // block + 2), size=min(
                nb, max(1, (nv + block - 1) // block + 2)), replace=False).tolist())
            blocks[q, :len(chosen)] = torch.tensor(chosen, dtype=torch.int32)
            pool_ref.append(sum(1 for c in chosen for j in range(c * block, c * block + block)
                                if j < nv))
            sel_ref += sum(1 for j in idx[q].tolist() if 0 <= j < nv)
        assert bench.visible_entries(b).tolist() == nv_ref
        assert bench.window_rows(b, win_lo, window).tolist() == win_ref
        assert bench.pool_pairs(b, blocks, block).tolist() == pool_ref
        want = sel_ref * 576 + sum(win_ref) * 576 + nq * (heads * 512 * 4 + k * 4 + heads * 4)
        assert bench.attn_launch_bytes(b, idx, win_lo, window, heads) == want
        assert bench.attn_launch_bytes(b, None, None, window, heads) == (
            int(bench.window_rows(b, None, window).sum()) * 576 + nq * (heads * 512 * 4 + heads * 4))
    assert bench.index_score_flops(10, 32) == 2 * 10 * 32 * 128


def test_traffic_record_only_for_the_measured_kernel(tmp_path, monkeypatch):
    """The ncu DRAM traffic is reported only when the record was taken on the
    attention source that is built now (the record keys it by a source hash)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    kid = b.run_kernel_id()
    (tmp_path / "profiles").mkdir()
    rec = {"workloads": {"c3_encoder_prefill": {"kernel_id": kid, "traffic_bytes_per_launch": 123},
                         "c2_decoder_replay": {"kernel_id": "0" * 16,
                                               "traffic_bytes_per_launch": 456}}}
    (tmp_path / "profiles" / "attn_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    monkeypatch.setattr(b, "run_kernel_id", lambda: kid)    # the hash of the real source
    assert b.traffic_record("c3_encoder_prefill") == 123
    assert b.traffic_record("c2_decoder_replay") is None      # taken on another source
    assert b.traffic_record("c4_hierarchical") is None        # never measured
