"""Data-parallel host logic on CPU with two gloo ranks (no GPU).

The layer is independent per token row, so N GPUs run N replicas or row
shards with no data-path collective; the only cross-rank operations are the
barrier and the max over ranks of the timed region.  These tests run that
logic as two processes: row shards that cover the batch once and reproduce the
unsharded result (the oracle stands in for each rank's compute), the job time
as the slowest rank's, the whole-job value, and the reference arm's
rank-0-only output."""
import os
import socket
import types

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import oracle  # noqa: E402


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import synth
        import int8_rotated_quantized_gb300 as cr
        job_ms = bench.max_over_ranks(torch, dist, 10.0 + 5.0 * rank, "cpu")
        value = bench.weak_scaling_value(world, 1e12, 4, job_ms)
        M, K, N, b = 37, 128, 48, 32
        x = synth.activations_bf16(3, M, K, 2, 10.0)
        W = synth.normal_bf16(3, synth.STREAM_W, N, K, 0.02)
        wq, sw = oracle.quantize_weight(W, b)
        start, count = cr.shard_rows(M, world, rank)
        y_part, _, _ = oracle.linear_fwd(np.ascontiguousarray(x[start:start + count]), wq, sw, b)
        parts = [None] * world
        dist.all_gather_object(parts, (start, count, y_part))
        if rank == 0:
            y_full, _, _ = oracle.linear_fwd(x, wq, sw, b)
            parts.sort(key=lambda p: p[0])
            y = np.concatenate([p[2] for p in parts])
            contiguous = all(parts[i][0] + parts[i][1] == parts[i + 1][0] for i in range(world - 1))
            np.save(os.path.join(out_dir, "result.npy"),
                    np.array([job_ms, value, sum(p[1] for p in parts), float(contiguous),
                              float(np.array_equal(y, y_full))]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_rows_and_time_the_job(tmp_path):
    oracle.build()  # compile once, before the ranks load it
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    job_ms, value, covered, contiguous, equal = np.load(tmp_path / "result.npy")
    assert job_ms == 15.0                       # the slowest rank's time
    assert value == pytest.approx(world * 1e12 * 4 / 15e-3 / 1e12)
    assert covered == 37 and contiguous == 1.0  # every row exactly once, in order
    assert equal == 1.0                          # sharded rows give the unsharded result bit for bit


@pytest.mark.parametrize("M,world", [(0, 2), (1, 4), (37, 2), (20480, 8), (7, 3)])
def test_shard_rows_partition(M, world):
    import int8_rotated_quantized_gb300 as cr
    spans = [cr.shard_rows(M, world, r) for r in range(world)]
    assert spans[0][0] == 0
    assert all(spans[i][0] + spans[i][1] == spans[i + 1][0] for i in range(world - 1))
    assert sum(c for _, c in spans) == M
    assert max(c for _, c in spans) - min(c for _, c in spans) <= 1
    with pytest.raises(ValueError):
        cr.shard_rows(M, world, world)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = types.SimpleNamespace(steps=3, warmup=3, ref_rows=4)
    assert bench.run_reference(args) is None
