"""The benchmark's multi-rank host logic on CPU: two gloo ranks (no GPU).

Each rank runs its own shard of independent (b, h) problems (weak scaling): the
shards differ, the timing is the maximum over ranks, the whole-job throughput
counts every rank's work, and only rank 0 runs the CPU reference arm.
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    import bench
    from transformer_scaled_dot_mha_gb300 import workloads as W

    w = W.WORKLOADS["decoder_causal_b16_h8_n512_d64"]
    q, _, _, _ = W.make_inputs(w, bench.shard_seed(w, rank), B=1, H=1, n_q=4, n_k=4)
    per_rank_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    mx = bench.max_over_ranks(per_rank_ms)
    value = bench.weak_scaling_tflops(2e12, 3, mx, world)
    args = type("A", (), {"steps": 1, "warmup": 0})()
    ref = bench.run_reference(args, W.WORKLOADS["tiny_f32_b1_h1_n16_d8"]) if rank == 1 else None
    out[rank] = (q.copy(), mx, value, ref)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    (q0, mx0, v0, _), (q1, mx1, v1, ref1) = out[0], out[1]
    assert not np.array_equal(q0, q1)          # independent shards
    assert mx0 == mx1 == 15.0                  # max over ranks
    assert v0 == v1 == pytest.approx(2 * 2e12 * 3 / 0.015 / 1e12)
    assert ref1 is None                        # the reference arm runs on rank 0 only


def test_single_process_helpers():
    import bench
    from transformer_scaled_dot_mha_gb300 import workloads as W

    w = W.WORKLOADS["long_causal_b2_h16_n8192_d64"]
    assert bench.shard_seed(w, 0) == w.seed
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.weak_scaling_tflops(1e12, 10, 1000.0, 1) == pytest.approx(10.0)  # 1e13 FLOP in 1 s


def test_kernel_source_hash_ignores_comments_only():
    """The DRAM traffic the bench reports is keyed by a hash of the kernel sources; a
    comment, blank-line or indentation edit must keep the key, any code edit must change it."""
    import bench

    code = 'int f(int x) {\n  // scale\n  return 2 * x; /* twice */\n}\nconst char* s = "// kept";\n'
    assert bench._code_only(code) == bench._code_only(code.replace("// scale", "// doubled\n\n"))
    assert "// kept" in bench._code_only(code)                     # a string literal is code
    assert bench._code_only(code) != bench._code_only(code.replace("2 * x", "3 * x"))
    assert bench._code_only(code) == bench._code_only(code.replace("  return", "      return"))
    for k in bench.KERNEL_SOURCES:
        assert len(bench.kernel_source_hash(k)) == 16


def test_traffic_table_matches_current_sources():
    """Every DRAM-traffic entry the bench can report was captured on the kernel sources
    as they are now (its key is their hash) and names a defined workload: a kernel edit
    leaves its entries stale until they are captured again."""
    import bench
    from transformer_scaled_dot_mha_gb300 import workloads as W

    for (workload, kernel, src_hash), nbytes in bench.NCU_TRAFFIC.items():
        assert workload in W.WORKLOADS
        assert src_hash == bench.kernel_source_hash(kernel), (workload, kernel)
        assert nbytes > 0
