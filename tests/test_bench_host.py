"""Host-side logic of bench.py without a GPU: algorithmic bytes, the
whole-job aggregation over replicas (gloo, world size 2) and the reference
arm (the oracle on the host cores)."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_alg_bytes_match_the_roofline_table():
    # R = 8, 512x8192 bf16 per rank
    N = 512 * 8192
    assert bench.alg_bytes("oneshot_fanout", 8, N) == 134_217_728
    assert bench.alg_bytes("fused_ll8", 8, N) == 369_098_752
    assert bench.alg_bytes("twophase", 8, N) == 134_217_728 + 2 * N
    assert bench.alg_bytes("oneshot_pull", 8, N) == 2 * 64 * N + 2 * 8 * N
    # R = 4 and R = 8 at 64 MiB per rank
    assert bench.alg_bytes("fused_ll8", 4, 33_554_432) == 1_342_177_280
    assert bench.alg_bytes("fused_ll8", 8, 33_554_432) == 2_952_790_016
    assert bench.alg_bytes("twophase", 1, 100) == 400
    assert bench.launches_per_call("twophase", 8) == 2
    assert bench.launches_per_call("fused_ll8", 8) == 1
    assert bench.launches_per_call("packet_3op", 8) == 3
    assert bench.alg_bytes("fused_ll8_staged", 8, N) == 4 * 8 * N + 16 * 7 * N


def test_whole_job_aggregation():
    # 2 ranks x 1000 calls in 0.05 s (slowest rank): 25 us per call overall
    assert bench.whole_job_us_per_call(0.05, 1000, 2) == pytest.approx(25.0)
    assert bench.whole_job_us_per_call(0.05, 1000, 1) == pytest.approx(50.0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    w, r = bench.dist_init("gloo")
    bench.barrier()
    t = 0.010 * (rank + 1)               # rank 1 is the slowest
    t_max = bench.max_over_ranks(t)
    tot = bench.sum_over_ranks(1000.0)
    us = bench.whole_job_us_per_call(t_max, 1000, w)
    q.put((r, w, t_max, tot, us))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_replica_timing_over_gloo_world_size_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, t_max, tot, us in res:
        assert w == 2
        assert t_max == pytest.approx(0.020)     # max over ranks
        assert tot == pytest.approx(2000.0)
        assert us == pytest.approx(10.0)         # 2000 calls in 20 ms


def test_reference_arm_prints_one_line(capsys, monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3",
                "--workload", "r8_4096"])
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    line = json.loads(out[0])
    assert line["impl"] == "reference" and line["unit"] == "us/call"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "r8_4096"


def test_reference_arm_other_ranks_stay_silent(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])


def test_spread_of_per_call_times():
    s = bench.spread([t * 1e-6 for t in (5.0, 1.0, 3.0, 2.0, 4.0)])
    assert s == {"median": 3.0, "min": 1.0, "p90": 5.0, "max": 5.0, "calls": 5}


def test_reference_arm_prints_one_contract_line():
    """bench.py --impl reference times the oracle on the host (no GPU) and
    prints one JSON line carrying the contract's keys."""
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--workload", "r8_4096"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "us/call" and d["value"] > 0
    assert d["higher_is_better"] is False and d["metric"] == bench.METRIC
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "r8_4096"


def _timings(rows):
    """{count: {variant: us}} from (count, {variant: us}) pairs."""
    return {c: dict(t) for c, t in rows}


def test_tuning_rows_merge_runs_and_split_where_the_curves_cross():
    t = _timings([
        (4096, {"oneshot_pull": 2.1, "oneshot_fanout": 2.5, "fused_ll8": 4.9}),
        (65536, {"oneshot_pull": 2.4, "oneshot_fanout": 2.7}),
        (131072, {"oneshot_pull": 3.1, "oneshot_fanout": 3.0}),
        (1048576, {"oneshot_pull": 15.0, "oneshot_fanout": 7.9, "twophase": 9.9}),
    ])
    rows = bench.tuning_rows(8, t)
    # pull up to the geometric mean of 65536 and 131072, fan-out beyond
    assert rows == [(8, 92681, "oneshot_pull"), (8, bench.MAX_TUNED_COUNT, "oneshot_fanout")]
    # every measured count lands in the row of its own winner
    for c, v in ((4096, "oneshot_pull"), (65536, "oneshot_pull"), (131072, "oneshot_fanout"),
                 (1048576, "oneshot_fanout")):
        assert next(r[2] for r in rows if c <= r[1]) == v


def test_tuning_rows_skip_the_comparison_forms_and_handle_one_size():
    t = _timings([(8, {"fused_ll8_staged": 0.1, "packet_3op": 0.1, "twophase": 3.0,
                       "oneshot_fanout_bulk": 2.0})])
    assert bench.tuning_rows(16, t) == [(16, bench.MAX_TUNED_COUNT, "oneshot_fanout_bulk")]
    # a boundary never falls below the last count the earlier variant won
    t = _timings([(7, {"oneshot_pull": 1.0, "oneshot_fanout": 2.0}),
                  (8, {"oneshot_pull": 2.0, "oneshot_fanout": 1.0})])
    assert bench.tuning_rows(2, t) == [(2, 7, "oneshot_pull"),
                                       (2, bench.MAX_TUNED_COUNT, "oneshot_fanout")]


def test_write_tuning_writes_the_library_format(tmp_path):
    path = tmp_path / "table.txt"
    bench.write_tuning(str(path), [(8, 92681, "oneshot_pull"), (8, 1 << 40, "oneshot_fanout")],
                       "test")
    lines = path.read_text().splitlines()
    assert lines[0].startswith("#")
    assert lines[1:] == ["8 92681 oneshot_pull", "8 1099511627776 oneshot_fanout"]


def test_strip_comments_keeps_code_and_literals():
    src = ('int a = 1;  // one\n'
           '/* a block\n   over lines */ const char* s = "x // y /* z */";\n'
           "char q = '\"';  /* inline */ int b;\n"
           '\n'
           '   // alone\n')
    out = bench.strip_comments(src)
    assert out == ('int a = 1;\n  const char* s = "x // y /* z */";\n'
                   "char q = '\"';    int b;")
    # a code change shows, a comment change does not
    assert bench.strip_comments(src.replace("one", "uno")) == out
    assert bench.strip_comments(src.replace("b;", "c;")) != out

