"""The multi-process (N > 1) bench path on CPU: two gloo ranks check the
barrier, the max over ranks and the whole-job throughput that rank 0 reports
(one process per GPU on a GPU machine; replicas, no collective on the data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    d = bench.Dist(world, torch.device("cpu"))
    d.barrier()
    local_ms = 2.0 + rank                      # rank 1 is the slow one
    ms_max = d.max(local_ms)
    q.put((rank, ms_max, bench.whole_job_throughput(6113, ms_max, world)))
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, value in out:
        assert ms_max == 3.0                    # max over ranks, seen by every rank
        assert value == pytest.approx(2 * 6113 / 3.0e-3)


def test_traffic_record_is_ignored_when_source_changes(tmp_path, monkeypatch):
    import json
    import bench
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    import hashlib
    rec = {"chunk_chain": {"workload": "w", "source": str(src), "dram_bytes_per_launch": 123,
                           "source_sha256": hashlib.sha256(b"kernel v1").hexdigest()}}
    f = tmp_path / "t.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    monkeypatch.setattr(bench, "ROOT", "/")
    assert bench.ncu_traffic("chunk_chain", "w") == 123
    assert bench.ncu_traffic("chunk_chain", "other") is None
    src.write_text("kernel v2")
    assert bench.ncu_traffic("chunk_chain", "w") is None


def test_traffic_record_list_per_kernel(tmp_path, monkeypatch):
    import hashlib
    import json
    import bench
    src = tmp_path / "r.cu"
    src.write_text("recurrent v1")
    sha = hashlib.sha256(b"recurrent v1").hexdigest()
    rec = {"recurrent": [{"workload": "decode", "source": str(src), "dram_bytes_per_launch": 9, "source_sha256": sha},
                         {"workload": "verify", "source": str(src), "dram_bytes_per_launch": 5, "source_sha256": sha}]}
    f = tmp_path / "t.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    monkeypatch.setattr(bench, "ROOT", "/")
    assert bench.ncu_traffic("recurrent", "decode") == 9
    assert bench.ncu_traffic("recurrent", "verify") == 5
    assert bench.ncu_traffic("recurrent", "kda") is None
