"""bench.py's multi-rank logic on CPU: gloo, world size 2 (no GPU)."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rate, t_max = bench.whole_job_rate(1.0 + rank, 100, world)
        q.put((rank, rate, t_max))
    finally:
        dist.destroy_process_group()


def test_whole_job_rate_takes_max_over_ranks():
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
    for rank, rate, t_max in res:
        assert t_max == pytest.approx(2.0)           # the slower rank sets the time
        assert rate == pytest.approx(2 * 100 / 2e-3)  # all ranks' units over it


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    rate, t_max = bench.whole_job_rate(4.0, 4096, 1)
    assert t_max == 4.0 and rate == pytest.approx(4096 / 4e-3)


def test_reference_arm_prints_only_on_rank_zero(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")

    class A:
        workload = "tiny_t64_d32"
        seed = 0
        steps = 3
        warmup = 3

    bench.run_reference_arm(A())
    assert capsys.readouterr().out == ""


def test_traffic_record_only_for_its_workload_and_source(tmp_path, monkeypatch):
    """The committed ncu traffic figure is reported only for the workload it was captured on and
    only while the kernel source still hashes to the recorded value."""
    import hashlib
    import json

    sys.path.insert(0, ROOT)
    import bench

    src_dir = tmp_path / "hybrid_linear_attention_prefill_gb300" / "csrc"
    src_dir.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (src_dir / "k.cu").write_bytes(b"kernel v1")
    rec = {"source": "k.cu", "source_sha256_16": hashlib.sha256(b"kernel v1").hexdigest()[:16],
           "workload": "wl_a", "dram_bytes_per_launch": 123}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"gdn_chain_kernel": rec}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("gdn_chain_kernel", "wl_a")["dram_bytes_per_launch"] == 123
    assert bench.traffic_record("gdn_chain_kernel", "wl_b") is None       # another workload
    assert bench.traffic_record("gdn_prep_kernel", "wl_a") is None        # no record
    (src_dir / "k.cu").write_bytes(b"kernel v2")
    assert bench.traffic_record("gdn_chain_kernel", "wl_a") is None       # source changed since
