"""The N > 1 host path of bench.py on CPU: two gloo ranks (torch.multiprocessing, spawn) discover
rank and world from the environment, meet at barriers, take the slowest rank's time and report the
whole job's throughput; each rank scores its own sequence (weak scaling, replicas)."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, world, local, pg = bench.dist_init(None)
    assert (r, world, local) == (rank, 2, rank)
    assert pg.get_backend() == "gloo"
    bench.barrier(pg)
    ms = bench.max_over_ranks(pg, 1.0 + 3.0 * rank, None)  # rank 1 is the slow one
    bench.barrier(pg)
    with open(os.path.join(out_dir, f"{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": bench.whole_job_value(1000.0, world, ms)}, f)
    pg.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_ranks(tmp_path):
    mp.spawn(_worker, args=(_free_port(), str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"{r}.json")) for r in range(2)]
    for x in res:
        assert x["ms"] == 4.0
        assert x["value"] == pytest.approx(1000.0 * 2 / 4e-3)


def test_ranks_score_independent_sequences():
    sys.path.insert(0, ROOT)
    from kv_cache_eviction_02_gb300 import synth
    cfg = synth.LOREKV_CONFIGS["tiny"]
    a = synth.lorekv_inputs(cfg, "cpu")
    b = synth.lorekv_inputs(cfg.replace(seed=cfg.seed + 1), "cpu")  # what rank 1 scores
    assert not torch.equal(a["K"], b["K"]) and not torch.equal(a["Q_W"], b["Q_W"])
    assert torch.equal(a["K"], synth.lorekv_inputs(cfg, "cpu")["K"])  # seeded
