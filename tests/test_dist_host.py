"""Host-side multi-rank plumbing of bench.py on CPU (gloo, world size 2).

The operator needs no collective on its data path: ranks process independent
sequences/heads.  What the N-GPU benchmark adds is host logic -- rank/world
parsing, a barrier around the timed region, and taking the slowest rank's
time -- which is what these tests exercise, without a GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, lr = bench.dist_env()
        assert (w, r, lr) == (world, rank, rank)
        bench.barrier(world)
        slowest = bench.reduce_max(1.5 + rank * 2.25, world, device="cpu")
        q.put((rank, slowest))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 3.75), (1, 3.75)]


def test_single_rank_paths_need_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.reduce_max(2.5, 1) == 2.5
    bench.barrier(1)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"steps": 1, "warmup": 0})()
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("line", [
    "kda_decode_kernel decode_256x64 {d} 123",
])
def test_profiled_traffic_lookup(tmp_path, monkeypatch, line):
    src = "linear_attention_sequence_gb300/csrc/kda_decode.cu"
    digest = bench.source_digest(src)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.txt").write_text("# comment\n" + line.format(d=digest) + "\n")
    (tmp_path / src).parent.mkdir(parents=True)
    (tmp_path / src).write_bytes(open(os.path.join(bench.ROOT, src), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("kda_decode_kernel", src, "decode_256x64") == 123.0
    assert bench.profiled_traffic("kda_decode_kernel", src, "other_workload") is None
