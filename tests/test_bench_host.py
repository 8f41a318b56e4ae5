"""Host logic of bench.py on CPU: the max-over-ranks timing reduction and the
whole-job value with 2 gloo ranks, the clock-sample summary and the JSON
contract helpers.  No GPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    assert bench.dist_env() == (rank, rank, world)
    bench.dist_init(world, "gloo")
    local_ms = 100.0 + 50.0 * rank  # rank 1 is the slow one
    bench.barrier(world)
    mx = bench.max_over_ranks(local_ms, world)
    val = bench.whole_job_value(1e12, 10, world, mx)
    q.put((rank, mx, val))
    dist.destroy_process_group()


def test_two_rank_gloo_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, val in res:
        assert mx == 150.0                      # max over ranks
        assert val == pytest.approx(2 * 1e12 * 10 / 0.150 / 1e12)  # both ranks' work / slowest time


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_value(2e12, 4, 1, 1000.0) == pytest.approx(8.0)


def test_clock_summary_parsing():
    c = bench.ClockSampler(0)
    c.t0, c.t1 = 10.0, 20.0
    row = lambda mhz, pc: ["0", str(mhz), "2070", "900.5", "0x0", "Not Active", "Not Active",  # noqa: E731
                           "Not Active", pc]
    c.samples = [(9.0, row(300, "Not Active")), (12.0, row(1900, "Not Active")), (15.0, row(1950, "Active")),
                 (18.0, row(1920, "Not Active")), (30.0, row(100, "Not Active"))]
    s = c.summary()
    assert s["sm_mhz"] == 1920 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 3


def test_peaks_and_traffic_lookup():
    pk = bench.measured_peaks()
    assert pk["bf16_tflops"] > 0 and pk["hbm_gbs"] > 0
    assert bench.ncu_traffic("no_such_kernel") is None


def test_oracle_sampler_counts_causal_pairs():
    s = bench.OracleSampler()
    rows = s.rows(3)
    assert list(rows) == [0, 4095, 8191]
    assert s.flops(rows) == 3.5 * 4 * 128 * (1 + 4096 + 8192)
    assert s.run((2, rows)) == 2 * s.flops(rows)
    assert "2 of 32" in s.describe((2, rows))


def test_sweep_append_file_resumes_after_a_killed_run(tmp_path):
    """Cases recorded in an --append file are skipped; a last line cut short
    by a killed run does not count, so that case runs again."""
    path = tmp_path / "sweep.jsonl"
    assert bench.sweep_done_keys(str(path)) == set()
    assert bench.sweep_done_keys(None) == set()
    path.write_text('{"T": 128, "d": 64, "causal": false, "dtype": "bf16", "fwd_ms": 0.01}\n'
                    '{"T": 8192, "d": 128, "causal": true, "dtype": "fp32", "fwd_ms": 9.0}\n'
                    '{"T": 512, "d": 128, "causal": tr')
    done = bench.sweep_done_keys(str(path))
    assert done == {bench.sweep_key(128, 64, False, "bf16"), bench.sweep_key(8192, 128, True, "fp32")}
    assert bench.sweep_key(512, 128, True, "bf16") not in done
    bench.sweep_end_partial_line(str(path))
    with open(path, "a") as f:
        f.write('{"T": 512, "d": 128, "causal": true, "dtype": "bf16", "fwd_ms": 0.02}\n')
    assert bench.sweep_key(512, 128, True, "bf16") in bench.sweep_done_keys(str(path))
    bench.sweep_end_partial_line(str(path))  # a complete file is left as it is
    assert path.read_text().count("\n") == 4
