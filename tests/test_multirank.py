"""Host logic of the multi-rank bench run (``bench.py`` under torchrun, one
rank per GPU): each rank draws its own sequences, the job's time is the
largest rank time (an all-reduce MAX), the job's rate counts every rank's
queries, and the reference arm runs on rank 0 alone.  Two ``gloo`` ranks on
the CPU run the same reduction code the NCCL run uses."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 2.0 + 3.0 * rank                     # rank 1 is the slow one
        job_ms = bench._max_over_ranks(torch, tdist, ms, device="cpu")
        rate = bench._job_rate(world, 32 * 10, job_ms)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{job_ms} {rate}")
    finally:
        tdist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    got = [tuple(map(float, (tmp_path / f"rank{r}.txt").read_text().split())) for r in range(world)]
    assert got[0] == got[1]                       # every rank reports the same job time
    job_ms, rate = got[0]
    assert job_ms == 5.0                          # the slowest rank's time, not the mean
    assert rate == pytest.approx(2 * 32 * 10 / 5e-3)   # all ranks' queries over that time


def test_single_rank_needs_no_collective():
    assert bench._max_over_ranks(torch, None, 7.5) == 7.5
    assert bench._job_rate(1, 32, 0.25) == pytest.approx(128000.0)


class _Args:
    batch = 0
    steps = 1
    warmup = 0


def test_each_rank_draws_its_own_sequences():
    from long_context_compressed_18_b300 import inputs
    s0, s1 = bench._decode_shape(_Args, 0), bench._decode_shape(_Args, 1)
    assert s0.seed != s1.seed and (s0.B, s0.N_c, s0.k) == (s1.B, s1.N_c, s1.k)
    small = dict(n=256, q_pos0=255)            # 64 compressed entries a sequence
    a = inputs.make_inputs(type(s0)(**{**s0.__dict__, **small}), device="cpu", batches=[0])
    b = inputs.make_inputs(type(s1)(**{**s1.__dict__, **small}), device="cpu", batches=[0])
    assert not torch.equal(a["idx_q"].float(), b["idx_q"].float())


def test_reference_arm_runs_on_rank_zero_only():
    assert bench.run_reference(_Args, torch, rank=1, world=2) is None
