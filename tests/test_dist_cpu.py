"""The multi-rank (torchrun) path of bench.py on CPU, with gloo (no GPU).

The indexer path shards by request with no exchange step, so N ranks run N
independent replicas; the only cross-rank logic is the whole-job reduction
(slowest rank's time, summed units) and "rank 0 alone prints, the others
exit 0".  Both are checked here with world size 2 on 127.0.0.1.
"""

import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, str(ROOT))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: step times 1.5 + r and 10 - r ms, 100 * (r + 1) units
        times, units = bench.reduce_over_ranks([1.5 + rank, 10.0 - rank], 100 * (rank + 1), world,
                                               "cpu")
        Path(out_dir, f"r{rank}.json").write_text(json.dumps({"times": times, "units": units}))
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_gloo_world_2(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [json.loads((tmp_path / f"r{r}.json").read_text()) for r in range(world)]
    for g in got:          # every rank holds the same whole-job figures
        assert g["times"] == [2.5, 10.0]
        assert g["units"] == 300.0


def test_reduce_over_ranks_single_rank_is_identity():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.reduce_over_ranks([3.0, 4.0], 7, 1) == ([3.0, 4.0], 7.0)


@pytest.mark.parametrize("extra", [[], ["--sparse-mla"]])
def test_non_zero_ranks_print_nothing_and_exit_0(extra):
    """Under torchrun the reference arm runs on rank 0 only: rank 1 exits 0
    without work and without output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    res = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1", "--warmup", "0", "--scale", "0.05",
                          *extra],
                         env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip() == ""


def test_gpus_n_starts_n_ranks_and_rank_0_alone_prints():
    """`bench.py --gpus 2` without a launcher starts two ranks itself (one
    replica per GPU); rank 0 alone prints its line, with n_gpus = 2.  The
    reference arm runs on the CPU, so this needs no GPU."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    res = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--workload", "0", "--steps", "1", "--warmup", "0"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


def test_gpus_must_match_the_launchers_world_size():
    """Under a launcher, --gpus must equal WORLD_SIZE (a mismatch would report
    the wrong number of GPUs)."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0", MASTER_ADDR="127.0.0.1")
    res = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                          "--workload", "0", "--steps", "1", "--warmup", "0"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode != 0
    assert "WORLD_SIZE=2" in res.stderr
    assert res.stdout.strip() == ""


def test_committed_counters_follow_the_kernel_code():
    """The ncu traffic figure in profiles/ is used only while the kernel
    sources hash to the value recorded beside it; comments and layout do not
    count, code does."""
    sys.path.insert(0, str(ROOT))
    import bench
    a = "int f(int x) {  // a comment\n  return x + 1; /* another */\n}\n"
    b = "int f(int x) {\n    return x + 1;\n}  // reworded comment\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()
    import re
    for name in ("batched_decode", "long_context_decode"):
        text = (ROOT / "profiles" / f"score_topk_{name}.md").read_text()
        m = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
        assert m is not None, name
        # valid summary -> its figure; stale summary -> no figure (never a wrong one)
        got = bench.profiled_traffic(name)
        assert (got is not None) == (m.group(1) == h), name
        if got is not None:
            # the counters cover at least the algorithmic bytes of a launch and not
            # much more (no wasted re-reads), per the summary's own figures
            alg = (re.search(r"Algorithmic bytes of a full launch: ([0-9.]+) MB", text)
                   or re.search(r"algorithmic ([0-9.]+) MB", text))
            assert alg is not None, name
            assert 0.95 <= got / (float(alg.group(1)) * 1e6) <= 1.1, name
