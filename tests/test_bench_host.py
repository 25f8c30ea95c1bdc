"""Host-side logic of bench.py: byte/flop accounting and the multi-rank control plane
(two gloo ranks on CPU: max-over-ranks time, sum-over-ranks units)."""
import os
import socket

import pytest

import bench


def test_algorithmic_bytes_match_the_stated_figures():
    # Llama-7B decode workload: W fp16 [11008, 4096], A [1, 4096]
    assert bench.quantize_bytes(11008, 4096, 2) == 113_778_688
    assert bench.matmul_bytes(1, 11008, 4096) == 23_631_360
    # 70B MLP layer: W fp16 [28672, 8192]
    assert bench.quantize_bytes(28672, 8192, 2) == 592_707_584
    assert bench.matmul_bytes(1, 28672, 8192) == 123_019_264
    # skinny M = 8 and prefill GEMM
    assert bench.matmul_bytes(8, 4096, 4096) == 8_912_896
    assert bench.matmul_flops(2048, 14336, 4096) == 240_518_168_576
    # tiny fp32 case
    assert bench.quantize_bytes(128, 256, 4) == 148_224


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench as b
    d = b.dist_init(world)
    t, u = b.aggregate(1.0 + rank, 10.0 * (rank + 1), d)
    b.barrier(d)
    q.put((rank, t, u))
    d.destroy_process_group()


def test_two_rank_aggregation_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u in out:
        assert t == 2.0          # max over ranks
        assert u == 30.0         # sum over ranks


def test_single_rank_aggregation_is_identity():
    assert bench.aggregate(3.5, 7.0, None) == (3.5, 7.0)


def test_reference_arm_runs_on_cpu(capsys):
    """The reference arm (CPU oracle alone) prints one JSON line with impl=reference."""
    import json
    rc = bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3",
                     "--workload", "tiny"])
    assert rc == 0
    line = capsys.readouterr().out.strip().splitlines()[-1]
    d = json.loads(line)
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("count,period", [(1, 85), (20, 85), (20, 17), (999, 5), (1000, 85),
                                          (1001, 85), (10000, 85), (10000, 7), (5000, 2000)])
def test_graph_plan_covers_exactly_count_launches(count, period):
    n, reps, rest = bench.graph_plan(count, period)
    assert n * reps + rest == count
    assert 0 < n <= max(bench.MAX_GRAPH, period)
    if count > bench.MAX_GRAPH:
        assert n % period == 0          # every full replay continues the copy rotation
    else:
        assert (n, reps, rest) == (count, 1, 0)


def test_host_cpu_reports_cores_and_model():
    cores, model = bench.host_cpu()
    assert cores >= 1 and isinstance(model, str) and model


def test_kernel_names_have_sources():
    for M, K in ((1, 4096), (8, 4096), (2048, 4096), (1, 8192)):
        name = bench.matmul_kernel_name(M, K)
        assert name in bench.KERNEL_SOURCES
        assert len(bench.source_digest(name)) == 16


def test_kernel_sources_cover_device_includes():
    """Every csrc header a kernel family's files include is part of that family's
    digest, so a profile cannot stay 'current' after a change to code the kernel runs.
    The one documented exception: the warp-MMA family takes only host-side tensor-map
    helpers from gemm_tcgen05.cuh."""
    import re
    host_only = {("gemv_mma", "gemm_tcgen05.cuh")}
    for family, files in bench.KERNEL_SOURCES.items():
        names = {os.path.basename(f) for f in files}
        for f in files:
            path = os.path.join(bench.ROOT, f)
            assert os.path.exists(path), path
            for inc in re.findall(r'#include "([^"]+)"', open(path).read()):
                if inc.endswith(".cuh") and (family, inc) not in host_only:
                    assert inc in names, (family, f, inc)


def test_all_core_oracle_rate_runs_threads_in_parallel_blocks():
    """The all-core oracle matmul baseline (the compute-bound case) reports a positive
    rate, the thread count it used and the sample it timed."""
    tf, desc, used = bench.oracle_prefill_rate(0.05, 2, workload="tiny")
    assert tf > 0 and used == 2
    assert "2 threads at once" in desc and "tiny" in desc
