"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): every rank contributes
its own step time and the job time is the maximum over ranks; units are independent per rank
(data-parallel by request), so no data-path collective exists to test."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, _ = bench.dist_env()
    t = bench.max_over_ranks(10.0 + 5.0 * r, w)
    bench.barrier(w)
    q.put((r, w, t))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 15.0), (1, 2, 15.0)]


def test_single_rank_defaults():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    os.environ.pop("RANK", None)
    assert bench.dist_env()[:2] == (0, 1)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_traffic_record_key_ignores_comments_only():
    import bench
    src = 'int a = 1;  // one\n// a comment line\n\nconst char* s = "x // y";\n'
    assert bench._code_lines(src) == ["int a = 1;", 'const char* s = "x // y";']
    assert bench._code_lines(src.replace("one", "two")) == bench._code_lines(src)
    assert bench._code_lines(src.replace("= 1", "= 2")) != bench._code_lines(src)
    assert len(bench.compress_source_sha256()) == 64


def test_traffic_record_applies_only_to_its_launch_size():
    # the committed record covers the full 16384-unit launch of the llama3_8b workload; a
    # scaled-down run (fewer requests or layers) must not report it as its own traffic
    import bench
    with open(os.path.join(bench.ROOT, "profiles", "compress_kernel_llama3_8b_traffic.json")) as f:
        rec = json.load(f)
    units = rec["units_full_launch"]
    want = rec["dram_bytes_per_launch"] if rec["source_sha256"] == bench.compress_source_sha256() else None
    assert bench._ncu_traffic("llama3_8b", units) == want
    assert bench._ncu_traffic("llama3_8b", units // 8) is None
    assert bench._ncu_traffic("no_such_workload", units) is None
