"""Host logic of bench.py's multi-rank path on CPU: two gloo ranks, max over ranks."""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    # Each rank's own time; the job's time is the slowest rank.
    got = bench.reduce_max(1.5 + rank)
    bench.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 2.5


def test_reduce_max_single_process_is_identity():
    import bench
    assert bench.reduce_max(3.25) == 3.25


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_kernel_hash_ignores_comments_only():
    """The profile summaries record a hash of the kernel sources that bench.py checks before
    reading their DRAM bytes; it is taken over the code with comments removed, so that a
    comment edit keeps the counters valid while any change of code invalidates them."""
    import bench
    a = 'int f(int x) { // add one\n  return x + 1; /* done */ }\nconst char* s = "a // b";\n'
    b = 'int f(int x) {\n  return x + 1;  }\n// a new comment\nconst char* s = "a // b";\n'
    c = 'int f(int x) {\n  return x + 2;  }\nconst char* s = "a // b";\n'
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
    assert '"a // b"' in bench.code_only(a)
    assert len(bench.kernel_hash("ffma")) == 16


def test_profile_traffic_only_for_the_current_source(tmp_path):
    """The bench takes a kernel's DRAM bytes from a committed summary only when the summary
    records the hash of the kernel's present code; a stale hash, a missing field or a missing
    file gives no traffic figure rather than an old one."""
    import bench
    current = bench.kernel_hash("ffma")
    good = tmp_path / "good.md"
    good.write_text("kernel_source_sha256_16: %s\ndram_bytes_per_launch: 342682624\n" % current)
    assert bench.profile_traffic(str(good), "ffma") == 342682624.0
    stale = tmp_path / "stale.md"
    other = "0" * 16 if current != "0" * 16 else "f" * 16
    stale.write_text("kernel_source_sha256_16: %s\ndram_bytes_per_launch: 342682624\n" % other)
    assert bench.profile_traffic(str(stale), "ffma") is None
    no_bytes = tmp_path / "no_bytes.md"
    no_bytes.write_text("kernel_source_sha256_16: %s\n" % current)
    assert bench.profile_traffic(str(no_bytes), "ffma") is None
    assert bench.profile_traffic(str(tmp_path / "missing.md"), "ffma") is None
    # A summary taken on another kernel's sources does not serve this one.
    assert bench.profile_traffic(str(good), "tf32x3") is None or \
        bench.kernel_hash("tf32x3") == current


def test_clock_sampler_summary_from_samples(tmp_path):
    """The clock record of the bench and the sweep: the median SM clock, the largest maximum,
    the sample count and every throttle reason seen active in nvidia-smi's CSV rows (index,
    clock, maximum clock, power, active mask, then the four reasons); malformed rows are
    skipped, and no rows give no record."""
    from roofline_driven_tiling_gb300.clocks import ClockSampler
    rows = ["0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage line",
            "0, [N/A], 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    clk = ClockSampler(0)
    clk.path = str(path)
    s = clk.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}
    assert not path.exists()  # the sample file is removed once read
    empty = tmp_path / "empty.csv"
    empty.write_text("")
    clk.path = str(empty)
    assert clk.summary() is None
