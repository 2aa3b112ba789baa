"""Host logic of bench.py without a GPU: algorithmic byte counts and the replica
aggregation over ranks (gloo, world size 2)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads


def test_attention_bytes_closed_form():
    cfg = workloads.config("full")
    lens = [114689] * 4
    per_seq_tokens = sum(min(w, 114689) for w in cfg.windows[0])
    assert per_seq_tokens == 303104
    exp = 4 * per_seq_tokens * 2 * 128 * 2 + 2 * 4 * 32 * 128 * 2
    assert bench.attention_bytes(cfg, 0, lens) == exp
    # windows above the context are clipped to the context
    r = workloads.config("ragged")
    lens = np.asarray(r.prefill) + 1
    kv = sum(min(w, L) for L in lens for w in r.windows[3]) * 2 * 128 * 2
    assert bench.attention_bytes(r, 3, lens) == kv + 2 * 64 * 32 * 128 * 2


def test_materialize_and_append_bytes():
    cfg = workloads.config("long")
    assert bench.append_bytes(cfg) == 2 * 1 * 8 * 2 * 128 * 2
    w = cfg.windows[5]
    assert bench.materialize_bytes(cfg, 5) == 2 * sum(min(x, 164864) for x in w) * 512


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    ms, units = bench.aggregate(10.0 + rank * 5.0, 4.0 * (rank + 1), 2)
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_aggregate_takes_max_time_and_sum_of_units_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 15.0, 12.0), (1, 15.0, 12.0)]


def test_single_rank_aggregate_is_identity():
    assert bench.aggregate(3.5, 7.0, 1) == (3.5, 7.0)


def test_reference_arm_only_runs_on_rank_zero(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_cpu(monkeypatch, capsys):
    import json
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_times_whole_steps(monkeypatch, capsys):
    """Each timed step of the reference arm is a whole decode step (every layer), so the line's
    ms_per_step x steps is oracle time actually spent."""
    import json
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    calls = []
    real = bench.oracle_whole_step

    def spy(cfg, wl, step, steps_in, device, threads):
        calls.append((cfg.layers, step))
        return real(cfg, wl, step, steps_in, device, threads)

    monkeypatch.setattr(bench, "oracle_whole_step", spy)
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip())
    assert line["steps"] == 2 and line["warmup"] == 3
    cfg = workloads.config("tiny")
    assert calls[3:] == [(cfg.layers, 3), (cfg.layers, 4)]
    assert "2 whole decode steps" in line["cpu_baseline"]["sample"]


def test_secondary_workloads_default_only_for_the_headline_line(monkeypatch):
    seen = {}
    monkeypatch.setattr(bench, "run_hwkv", lambda args, cfg: seen.setdefault("sec", args.secondary))
    bench.main(["--steps", "1", "--warmup", "3"])
    assert seen.pop("sec") == ["ragged", "long", "long_full"]
    bench.main(["--steps", "1", "--warmup", "3", "--workload", "long"])
    assert seen.pop("sec") == []
    bench.main(["--steps", "1", "--warmup", "3", "--secondary", "none"])
    assert seen.pop("sec") == []
    with pytest.raises(KeyError):
        bench.main(["--steps", "1", "--warmup", "3", "--secondary", "nosuch"])
