"""Multi-rank host logic on CPU ranks (gloo, world size 2): request shards, per-replica noise
streams, the slowest-rank timing every rank agrees on, and a failing rank surfacing as an error
on the others instead of a hang.  No GPU is involved; the per-rank work is the oracle on that
rank's share of a small verification batch."""
import datetime
import os
import socket
import tempfile

import numpy as np
import pytest

from draft_sampling_verification_tcgen05_gb300.replicas import (RankInfo, job_throughput, max_over_ranks, rank_info,
                                                                replica_seed, shard_range)


def test_shard_ranges_cover_every_request_once():
    for n in (0, 1, 7, 64, 1000):
        for world in (1, 2, 3, 8):
            spans = [shard_range(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1


def test_rank_info_and_seeds():
    assert rank_info({}) == RankInfo(0, 1, 0)
    assert rank_info({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}).rank == 1
    with pytest.raises(ValueError):
        rank_info({"RANK": "2", "WORLD_SIZE": "2"})
    assert replica_seed(2, 0) == 2 and replica_seed(2, 1) != replica_seed(2, 0)
    assert job_throughput(8, 2, 1.0) == 16000.0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _verify_batch():
    from workloads import VerifyConfig, verify_inputs
    cfg = VerifyConfig("gloo", B=6, gamma=3, V=257, target_std=1.5, draft_sigmas=(0.5, 2.0),
                       independent_draft=False, data_seed=17)
    return verify_inputs(cfg)


def _rank_main(rank, world, port, out_dir, fail_rank):
    import torch.distributed as dist
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    ri = rank_info()
    dist.init_process_group("gloo", rank=ri.rank, world_size=ri.world, timeout=datetime.timedelta(seconds=10))
    try:
        if rank == fail_rank:
            raise RuntimeError(f"rank {rank} failed before its step")
        inp = _verify_batch()
        lo, hi = shard_range(inp["p_t"].shape[0], world, rank)
        out, nacc, _, _ = oracle.verify(inp["p_t"][lo:hi], inp["p_d"][lo:hi], inp["draft_tokens"][lo:hi], None,
                                        replica_seed(2, rank), 0)
        step_ms = 1.0 + 2.0 * rank                      # the ranks' own step times
        agreed = max_over_ranks(step_ms, dist)
        shards = [None] * world if rank == 0 else None
        dist.gather_object((lo, hi, out.tolist(), nacc.tolist(), agreed), shards, dst=0)
        if rank == 0:
            np.save(os.path.join(out_dir, "shards.npy"), np.array(shards, dtype=object), allow_pickle=True)
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_agree_on_the_slowest_time_and_cover_the_batch():
    import torch.multiprocessing as mp
    import oracle
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(2, _free_port(), d, -1), nprocs=2, join=True, start_method="spawn")
        shards = np.load(os.path.join(d, "shards.npy"), allow_pickle=True)
    inp = _verify_batch()
    covered = []
    for rank, (lo, hi, out, nacc, agreed) in enumerate(shards):
        assert agreed == 3.0                            # both ranks report the slower rank's time
        ref_out, ref_nacc, _, _ = oracle.verify(inp["p_t"][lo:hi], inp["p_d"][lo:hi], inp["draft_tokens"][lo:hi],
                                                None, replica_seed(2, rank), 0)
        np.testing.assert_array_equal(np.array(out), ref_out)
        np.testing.assert_array_equal(np.array(nacc), ref_nacc)
        covered.extend(range(lo, hi))
    assert covered == list(range(inp["p_t"].shape[0]))
    assert job_throughput(sum(h - l for l, h, *_ in shards) / 2, 2, 3.0) > 0


def test_a_failing_rank_surfaces_as_an_error_not_a_hang():
    import torch.multiprocessing as mp
    with tempfile.TemporaryDirectory() as d:
        with pytest.raises(Exception):
            mp.start_processes(_rank_main, args=(2, _free_port(), d, 1), nprocs=2, join=True,
                               start_method="spawn")
