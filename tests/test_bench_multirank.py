"""The multi-rank logic of bench.py on CPU: world size 2 over gloo.

Every rank runs an independent replica of the workload; the job time is the
slowest rank's (max over ranks) and the value aggregates the work of all
ranks over that time."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    bench.barrier(dist)
    t = bench.max_over_ranks(10.0 + 5.0 * rank, dist)
    v = bench.aggregate_throughput(2.0, 4, world, t)
    q.put((rank, t, v))
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, v in res:
        assert t == 15.0  # slowest rank's time on every rank
        assert v == pytest.approx(2 * 2.0 * 4 / 0.015)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.aggregate_throughput(1e12, 10, 1, 1000.0) == pytest.approx(1e13)


def test_rejected_clocks_are_measured_once_more():
    """A timed region whose clocks saw a thermal or hardware slowdown is run
    once more and the second result kept, with the first run's reasons noted;
    power capping alone is kept as it is."""
    import bench

    runs = []

    def timed(reasons_by_run):
        def f():
            runs.append(1)
            return {"ms": float(len(runs)), "clocks": {"reasons": list(reasons_by_run[len(runs) - 1])}}
        return f

    r = bench.timed_with_retry(timed([["hw_thermal_slowdown", "sw_power_cap"], ["sw_power_cap"]]), None)
    assert len(runs) == 2 and r["ms"] == 2.0
    assert r["clocks"]["remeasured_after"] == ["hw_thermal_slowdown", "sw_power_cap"]
    runs.clear()
    r = bench.timed_with_retry(timed([["sw_power_cap"]]), None)
    assert len(runs) == 1 and "remeasured_after" not in r["clocks"]


def _worker_one_leaves(rank, world, port, q):
    import time

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    _, _, _, pg = bench.dist_setup(world, backend="gloo", timeout_s=5)
    bench.barrier(pg)  # both ranks are up
    if rank == 1:
        q.put((rank, "left"))
        q.close()
        q.join_thread()  # the item must reach the pipe before the process vanishes
        os._exit(3)  # a rank dies between steps, without a word to the others
    t0 = time.time()
    try:
        bench.barrier(pg)
        q.put((rank, "no error", time.time() - t0))
    except Exception as e:  # noqa: BLE001 -- the failure is the point
        q.put((rank, type(e).__name__, time.time() - t0))
    q.close()
    q.join_thread()
    os._exit(0)  # no teardown of a group with a dead member


def test_a_rank_that_leaves_is_detected_by_the_others():
    """A rank that exits between steps makes the survivors' next collective
    fail within the process group's timeout rather than hang."""
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker_one_leaves, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode is not None, "a rank hung"
    res = {}
    for _ in range(world):
        item = q.get(timeout=10)
        res[item[0]] = item[1:]
    assert res[1] == ("left",)
    outcome, waited = res[0]
    assert outcome != "no error" and waited < 60.0, res


def test_causal_rank_imbalance_closed_forms():
    """The per-virtual-rank causal work the bench reports: contiguous shards
    give rank r about (r + 1/2) * Ls keys per query, so max/mean tends to
    (2 cp - 1) / cp; striped shards split every prefix evenly, ratio -> 1;
    one shard is balanced by definition."""
    sys.path.insert(0, ROOT)
    import bench

    for cp in (2, 4, 8):
        assert bench.causal_rank_imbalance(1 << 16, cp, "contiguous") == pytest.approx((2 * cp - 1) / cp, abs=1e-3)
        assert bench.causal_rank_imbalance(1 << 16, cp, "striped") == pytest.approx(1.0, abs=1e-3)
    assert bench.causal_rank_imbalance(1024, 1, "contiguous") == 1.0


def test_input_digest_covers_the_first_mib_of_raw_bytes():
    """The bench records, beside each workload's seed, the SHA-256 of the
    first MiB of every input: checked against hashlib over the bytes built
    independently (bf16 bits are the top half of the fp32 bits of values that
    bf16 holds exactly), only the first MiB counts, and a seed redraws the
    same inputs."""
    import hashlib

    import numpy as np
    import torch

    import bench
    from context_attention_gb300 import synth

    vals = np.arange(-256, 256, dtype=np.float32)  # at most 8 significant bits: exact in bf16
    t = torch.from_numpy(vals).to(torch.bfloat16)
    bits = (vals.view(np.uint32) >> 16).astype("<u2").tobytes()
    d = bench.input_digest(7, x=t)
    assert d == {"seed": 7, "x_sha256_first_MiB": hashlib.sha256(bits).hexdigest()}

    big = torch.zeros(3 << 19, dtype=torch.bfloat16)  # 3 MiB
    ref = bench.input_digest(1, big=big)["big_sha256_first_MiB"]
    assert ref == hashlib.sha256(bytes(1 << 20)).hexdigest()
    big[(1 << 19) + 5] = 1.0  # past the first MiB: no change
    assert bench.input_digest(1, big=big)["big_sha256_first_MiB"] == ref
    big[5] = 1.0
    assert bench.input_digest(1, big=big)["big_sha256_first_MiB"] != ref

    a = synth.dit_qk(1, 2, 256, 128, seed=2, device="cpu")
    b = synth.dit_qk(1, 2, 256, 128, seed=2, device="cpu")
    da = bench.input_digest(2, q=a[0], k=a[1], v=a[2])
    assert da == bench.input_digest(2, q=b[0], k=b[1], v=b[2])
    assert da != bench.input_digest(2, q=a[1], k=a[0], v=a[2])


def test_clock_summary_from_sampled_lines(tmp_path):
    """The clock record of a timed region, from nvidia-smi's CSV lines (no
    header, no units, a timestamp first): median and maximum SM clock, the
    throttle reasons seen active, unparsable lines skipped, a clock far below
    its maximum with no reason flagged as a leftover lock (which the bench
    re-measures), and only the samples taken inside the region kept when
    there are any."""
    import datetime

    import bench

    t0 = 1.8e9  # host time the region starts

    def stamp(dt):
        return datetime.datetime.fromtimestamp(t0 + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]

    def summary(lines, window=(0.0, 10.0)):
        c = bench.ClockSampler(0)
        c.path = str(tmp_path / "clk.csv")
        c.t_in, c.t_out = t0 + window[0], t0 + window[1]
        with open(c.path, "w") as f:
            f.write("".join(line + "\n" for line in lines))
        out = c.summary()
        assert not os.path.exists(c.path)  # the sample file is removed
        return out

    na, act = "Not Active", "Active"

    def row(sm, *r, dt=1.0):
        return ", ".join([stamp(dt), "0", str(sm), "2070", "850.00", "0x0"] + list(r))

    s = summary([row(1935, na, na, na, act), row(1950, na, na, na, act), row(1700, na, na, na, na),
                 stamp(1.0) + ", 0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
                 "garbage"])
    assert s == {"sm_mhz": 1935.0, "sm_max_mhz": 2070.0, "sm_mhz_min": 1700.0, "samples": 3,
                 "samples_from": "inside the timed region", "reasons": ["sw_power_cap"]}
    s = summary([row(2070, na, act, na, na), row(2070, na, na, na, na)])
    assert s["reasons"] == ["hw_thermal_slowdown"] and s["sm_mhz"] == 2070.0
    # power-capped low clocks are kept; low clocks with no reason are a lock
    assert summary([row(1732, na, na, na, act)] * 3)["reasons"] == ["sw_power_cap"]
    s = summary([row(1200, na, na, na, na)] * 3)
    assert s["reasons"] == ["sm_clock_low_no_reason"]
    assert "sm_clock_low_no_reason" in bench.REJECTED_REASONS
    assert summary([row(1800, na, na, na, na)] * 3)["reasons"] == []  # 0.87 of max: not "well below"
    assert summary([])["reasons"] == ["unsampled"]
    # idle samples before and after the region do not enter its record ...
    lines = [row(2070, na, na, na, na, dt=-0.2), row(1700, na, na, na, act, dt=0.02),
             row(1720, na, na, na, act, dt=0.07), row(2070, na, na, na, na, dt=0.15)]
    s = summary(lines, window=(0.0, 0.1))
    assert (s["sm_mhz"], s["samples"], s["reasons"]) == (1710.0, 2, ["sw_power_cap"])
    # ... unless the region is too short to hold a sample: then all of them do
    s = summary(lines, window=(0.03, 0.06))
    assert s["samples"] == 4 and s["samples_from"].startswith("around")


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """`bench.py --impl reference` times the oracle (the method's only
    reference) on the host and prints one JSON line with the contract's keys;
    a rank other than 0 prints nothing.  The row sample is cut to 64 rows so
    the test stays short."""
    import json
    import types

    import bench

    monkeypatch.setattr(bench.OracleSampler, "rows_for", lambda self, seconds: 64)
    args = types.SimpleNamespace(steps=2, warmup=1, gpus=1)
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(args)
    assert capsys.readouterr().out == ""
    monkeypatch.setenv("RANK", "0")
    bench.run_reference(args)
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["vs_baseline"] is None
    assert d["config"]["workload"] == "DiT const-max ring self-attention prefill"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and "64 query rows" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
