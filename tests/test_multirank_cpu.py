"""Host logic of the multi-process benchmark path, run as two `gloo` ranks on
the CPU: the barrier, the max-over-ranks step time, the whole-job (weak
scaling) rate, per-rank input seeding, and the reference arm's rule that only
rank 0 works and prints."""
import contextlib
import io
import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "LOCAL_RANK": str(rank), "WORLD_SIZE": str(WORLD)})
    import bench
    from sparse_state_linear_router_gb300 import inputs as synth
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        ws, r, local = bench._dist()
        bench.rank_barrier(ws)
        # rank r "measured" 3 + 2r ms per step: the job takes the slowest rank's
        step_ms = bench.max_over_ranks_of(3.0 + 2.0 * rank, ws, torch.device("cpu"))
        value = bench.whole_job_tokens_per_s(ws, 1000, step_ms)
        # each rank draws its own batch (independent problems, no exchange)
        w = synth.WORKLOADS["tiny_f32"]
        x = synth.make_forward_inputs(w, seed=rank)
        gathered = [None] * WORLD
        dist.all_gather_object(gathered, x.q.tobytes()[:64].hex())
        # the reference arm: only rank 0 runs; other ranks return 0 at once
        buf = io.StringIO()
        rc = None
        if rank != 0:
            with contextlib.redirect_stdout(buf):
                rc = bench.main(["--impl", "reference", "--gpus", str(WORLD), "--steps", "1", "--warmup", "3"])
        bench.rank_barrier(ws)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ws": ws, "rank": r, "local": local, "step_ms": step_ms, "value": value,
                       "inputs": gathered, "ref_rc": rc, "ref_out": buf.getvalue()}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(port, str(tmp_path)), nprocs=WORLD, join=True, start_method="spawn")
    res = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(WORLD)]
    for r, x in enumerate(res):
        assert (x["ws"], x["rank"], x["local"]) == (WORLD, r, r)
        assert x["step_ms"] == 5.0                       # max over ranks, same on every rank
        assert x["value"] == pytest.approx(WORLD * 1000 / 5e-3)
    assert res[0]["inputs"] == res[1]["inputs"]          # every rank saw the same gather
    assert res[0]["inputs"][0] != res[0]["inputs"][1]    # and the two batches differ
    assert res[1]["ref_rc"] == 0 and res[1]["ref_out"] == ""


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks_of(4.5, 1, None) == 4.5
    assert bench.whole_job_tokens_per_s(1, 32768 + 256, 1.0) == pytest.approx(33024e3)
    bench.rank_barrier(1)


def test_profiled_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """roofline.traffic comes from the ncu record in profiles/dram_traffic.json
    only while the kernel source still has the hash recorded there."""
    import hashlib
    import bench
    src = tmp_path / "k.cu"
    src.write_bytes(b"kernel v1\n")
    (tmp_path / "profiles").mkdir()
    rec = {"kern": {"source": "k.cu", "source_sha256": hashlib.sha256(b"kernel v1\n").hexdigest(),
                    "dram_bytes_per_launch": 12345, "summary": "profiles/p.md"}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("kern") == (12345, "profiles/p.md")
    assert bench.profiled_traffic("other") == (None, None)
    src.write_bytes(b"kernel v2\n")
    assert bench.profiled_traffic("kern") == (None, None)
    src.unlink()
    assert bench.profiled_traffic("kern") == (None, None)


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the CPU oracle on bounded samples) prints one
    JSON line with the native arm's metric, unit and config plus its own
    cpu_baseline and a zero-copy e2e entry."""
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-seconds", "0.5"])
    assert rc == 0
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["config"]["workload"]
