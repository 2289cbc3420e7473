"""Host-side logic of bench.py: byte accounting, clock parsing, and the
multi-process path (barrier + max over ranks) on CPU with gloo, world size 2."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_step_bytes_per_element():
    # amax reads 2 B; quantise reads 2 B, writes 0.5 B codes + 1/16 B scales;
    # dequantise reads 0.5625 B and writes 2 B
    assert bench.B_QUANT == pytest.approx(2.5625)
    assert bench.B_DEQ == pytest.approx(2.5625)
    assert bench.STEP_BYTES_PER_EL == pytest.approx(3 * 4.5625 + 2.5625)
    assert bench.step_bytes(8192, 4096) == pytest.approx(16.25 * 8192 * 4096)


def test_whole_job_throughput():
    assert bench.whole_job(100.0, 2.0, 1) == 50.0
    assert bench.whole_job(100.0, 2.0, 4) == 200.0   # every rank did its own 100 units


def test_parse_clock_lines():
    lines = ["0, 1965, 2032, 850.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
             "0, 1900, 2032, 1090.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "0, 1800, 2032, 1095.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
             "garbage line"]
    c = bench.parse_clock_lines(lines)
    assert c["sm_mhz"] == 1900
    assert c["sm_max_mhz"] == 2032
    assert c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clock_lines([])["error"]


def test_parse_args_contract():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.impl == "ours"
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])


def test_oracle_step_runs_on_a_tiny_sample():
    import synth
    x = synth.activation(32, 64)
    out = bench.oracle_step(synth.bf16_bits(x))
    assert set(out) == set(bench.WAYS)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        bench.barrier(torch.device("cpu"))
        t = bench.reduce_max(1.0 + rank, torch.device("cpu"))    # rank 1 is the slowest
        q.put((rank, t, bench.whole_job(10.0, t, world)))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    # both ranks see the slowest rank's time; throughput counts both ranks' units
    assert [r[1] for r in res] == [2.0, 2.0]
    assert [r[2] for r in res] == [10.0, 10.0]


def test_reduce_max_without_process_group():
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5


def test_source_digest_follows_the_translation_unit(tmp_path, monkeypatch):
    """A kernel's digest covers its .cu file and the headers it includes,
    directly or through other headers, and nothing else: an edit to a header
    another kernel includes leaves it unchanged."""
    csrc = tmp_path / "fp4_block_scaled_05_b300" / "csrc"
    inc = tmp_path / "include"
    csrc.mkdir(parents=True)
    inc.mkdir()
    (csrc / "a.cu").write_text('#include "h1.cuh"\n#include "../../include/pub.h"\nint a;\n')
    (csrc / "b.cu").write_text('#include "h2.cuh"\nint b;\n')
    (csrc / "h1.cuh").write_text('#include "h3.h"\n// h1\n')
    (csrc / "h2.cuh").write_text("// h2\n")
    (csrc / "h3.h").write_text("// h3\n")
    (inc / "pub.h").write_text("// public\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"ka": "a.cu", "kb": "b.cu"})
    da, db = bench.source_digest("ka"), bench.source_digest("kb")
    assert da and db and da != db
    (csrc / "h2.cuh").write_text("// h2 edited\n")
    assert bench.source_digest("ka") == da and bench.source_digest("kb") != db
    for path in (csrc / "h3.h", inc / "pub.h", csrc / "a.cu"):
        before = bench.source_digest("ka")
        path.write_text(path.read_text() + "// edited\n")
        assert bench.source_digest("ka") != before
    assert bench.source_digest("unknown") == ""
    (csrc / "h3.h").unlink()                      # a missing include: no digest, so no stale counters
    assert bench.source_digest("ka") == ""
