"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2).

With N GPUs every rank runs its own replica of the pass; the only
cross-rank operations are a barrier and the max / sum of scalars used to
report the job time (the slowest rank) and the total bytes.  The reference
arm runs on rank 0 only; the other ranks exit without work.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    bench.init_dist(world, "gloo")
    bench.barrier(world)
    m = bench.max_over_ranks(1.5 + rank, world)       # rank 1 is the slow one
    s = bench.sum_over_ranks(100.0 * (rank + 1), world)
    bench.barrier(world)
    torch.distributed.destroy_process_group()
    out[rank] = (m, s)


def test_max_and_sum_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        m, s = res[rank]
        assert m == 2.5          # every rank reports the slowest rank's time
        assert s == 300.0        # and the bytes of all ranks


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.sum_over_ranks(7.0, 1) == 7.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_oracle_sample_bytes_scale_with_the_sample():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from transformer_reduce_gb300 import traffic, workloads as W
    sm = W.SoftmaxCase("s", 2, 2, 64, False, (32, 64), 3.0, "bf16", 4)
    ln = W.LayerNormCase("l", 64, 128, 1.0, 2.0, "bf16", 4)
    si = W.softmax_inputs(sm)
    sample = bench.OracleSample(sm, si, [(ln, W.layernorm_inputs(ln))], softmax_frac=4, ln_frac=2)
    full = (traffic.softmax_fw_bytes(2, 2, 64, si["lengths"], False, "bf16")
            + traffic.softmax_bw_bytes(2, 2, 64, "bf16"))
    want = full / 4 + (traffic.layernorm_fw_bytes(32, 128, "bf16")
                       + traffic.layernorm_dinp_bytes(32, 128, "bf16")
                       + traffic.layernorm_dgdb_bytes(32, 128, "bf16"))
    assert sample.bytes == pytest.approx(want)
    sample.run()
    assert sample.time(min_seconds=0.01) > 0
