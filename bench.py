#!/usr/bin/env python
"""Benchmark of the context-parallel attention hot path on GB300.

One JSON line on rank 0.  A step is one pass of the hot path over one batch of
synthetic input:

* value  -- const-max ring attention prefill on the DiT workload (B=1, H=40,
  D=128, S=16384, cp=8 contiguous virtual shards, cross-head RMS-normalised
  q/k, bf16): the key pass (max |k|^2 per head) plus the fused ring kernel,
  which forms each row's bound from the q tile it loads, inputs resident in
  HBM.  Unit TFLOP/s of algorithmic work 4*B*H*S^2*D.
* decode -- DCP decode (64 sequences x 1 token, Hq=32, Hkv=8, D=128, context
  131072 over dcp=4 shards interleaved in 16-token blocks): split-KV partials
  plus the LSE merge.  Unit GB/s of K+V bytes read.
* e2e    -- the prefill step through the public API with pinned host buffers:
  q, k, v copied host->device and o copied back inside the timed region, the
  copies of one step overlapping the attention of the previous one.

* other_workloads (single-GPU runs; reported, not the value) -- online max,
  sink keys, causal GQA in both layouts, the QKV prologue, DCP prefill, paged
  decode and Ring Pass-Q decode, each timed the same way.

SM clocks and throttle reasons are sampled during the timed regions; a region
that saw a thermal or hardware slowdown, or SM clocks well below their maximum
with no reason given (a leftover clock lock), is measured once more.  Both headline
workloads' inputs (0.5 GB and 34 GB) are larger than the 129 MB L2, so no
flush runs between timed iterations.  ``--impl reference`` times the fp64
CPU oracle (the only reference this method has) on a bounded sample of the
same workload.  Under torchrun every rank runs an independent replica (the
method is not sharded across GPUs on this path) and rank 0 reports the
aggregate over ranks with the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ring-attn prefill TFLOP/s (% bf16 peak); DCP decode KV GB/s (% HBM BW)"
PREFILL = dict(B=1, H=40, S=16384, D=128, cp=8, seed=2)
DECODE = dict(N=64, Hq=32, Hkv=8, D=128, W=4, I=16, Lloc=32768, seed=5)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def prefill_flops(c=PREFILL):
    return 4.0 * c["B"] * c["H"] * c["S"] ** 2 * c["D"]


# datasheet figures of one GB300 (dense bf16 tensor rate, HBM3e bandwidth),
# reported beside the measured peaks the roofline fractions use
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0


def decode_bytes(c=DECODE):
    return 2.0 * c["W"] * c["N"] * c["Hkv"] * c["Lloc"] * c["D"] * 2


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def read_traffic(name):
    """Per-launch DRAM bytes recorded from an ncu capture (profiles/*.txt)."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            if line.startswith("traffic_bytes_per_launch:"):
                v = line.split(":", 1)[1].strip()
                return None if v in ("", "null") else float(v)
    return None


# a median SM clock below this fraction of the maximum with none of the
# sampled throttle reasons active is taken for a clock lock left by someone
LOW_CLOCK_FRACTION = 0.85


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms from before
    the timed region to after it; the summary keeps the samples taken inside
    the region (by host time), or all of them when the region is shorter than
    the sampling interval."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None
        self.t_in = self.t_out = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        self.t_in = time.time()
        return self

    def __exit__(self, *exc):
        self.t_out = time.time()
        time.sleep(0.06)  # one more sample after the region
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []  # (host time or None, sm MHz, max MHz, active reasons)
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm, top = float(parts[2]), float(parts[3])
                except ValueError:
                    continue
                try:
                    t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    t = None
                rows.append((t, sm, top, {n for n, v in zip(names, parts[6:10]) if v.lower() == "active"}))
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        inside = [r for r in rows if r[0] is not None and self.t_in is not None and self.t_out is not None
                  and self.t_in <= r[0] <= self.t_out]
        window = "inside the timed region" if inside else "around the timed region (shorter than 50 ms)"
        use = inside or rows
        sms = [r[1] for r in use]
        med, top = statistics.median(sms), max(r[2] for r in use)
        reasons = set().union(*[r[3] for r in use])
        if med < LOW_CLOCK_FRACTION * top and not reasons:
            reasons.add("sm_clock_low_no_reason")  # what a clock lock left behind looks like
        return {"sm_mhz": med, "sm_max_mhz": top, "sm_mhz_min": min(sms), "samples": len(sms),
                "samples_from": window, "reasons": sorted(reasons)}


# a rank that dies leaves the others at their next collective; they give up
# after this long (the longest gap between collectives is rank 0's CPU
# baseline, ~16 s) instead of holding every GPU for the backend's default
PG_TIMEOUT_S = 300


def dist_setup(n_gpus, backend="nccl", timeout_s=PG_TIMEOUT_S):
    import datetime

    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus and world > 1:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    pg = None
    if world > 1:
        import torch.distributed as dist

        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend, timeout=datetime.timedelta(seconds=timeout_s))
        pg = dist
    return rank, world, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


# a timed region whose clocks saw one of these is not a valid measurement:
# it is taken once more (sw_power_cap is normal under load and is kept)
REJECTED_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sm_clock_low_no_reason")


def timed_with_retry(timed, pg):
    """Run the timed region; if any rank's clocks saw a rejected slowdown,
    run it once more (all ranks together) and keep the second result, noting
    the first run's reasons in its clock summary."""
    res = timed()
    bad = any(r in REJECTED_REASONS for r in res["clocks"].get("reasons", []))
    if max_over_ranks(float(bad), pg) > 0:
        first = res["clocks"].get("reasons", [])
        res = timed()
        res["clocks"]["remeasured_after"] = first
    return res


def input_digest(seed, **tensors):
    """The seed and, per input tensor, the SHA-256 of its first MiB of raw
    bytes (the whole tensor if smaller), so that two runs can show they drew
    the same inputs."""
    import hashlib

    import torch

    out = {"seed": seed}
    for name, t in tensors.items():
        flat = t.detach().reshape(-1)
        n = min(flat.numel(), (1 << 20) // t.element_size())
        raw = flat[:n].cpu().contiguous().view(torch.uint8).numpy().tobytes()
        out[f"{name}_sha256_first_MiB"] = hashlib.sha256(raw).hexdigest()
    return out


def max_over_ranks(x, pg):
    """Max of a float over all ranks (the job's time is its slowest rank's)."""
    if pg is None:
        return x
    import torch

    dev = "cuda" if pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(work_per_step, steps, world, max_total_ms):
    """Whole-job throughput: the work of every rank's replica over the time
    of the slowest rank (work units per second)."""
    return world * work_per_step * steps / (max_total_ms / 1e3)


# --------------------------------------------------------------------------- ours


def bench_prefill(ca, torch, steps, warmup, pg, dev_index):
    from context_attention_gb300 import synth

    c = PREFILL
    q, k, v = synth.dit_qk(c["B"], c["H"], c["S"], c["D"], seed=c["seed"], device="cuda")
    digest = input_digest(c["seed"], q=q, k=k, v=v)
    o = torch.empty_like(q)
    lse = torch.empty(c["B"], c["H"], c["S"], device="cuda", dtype=torch.float32)
    kmax2 = torch.empty(c["B"], c["H"], device="cuda", dtype=torch.float32)
    lib = ca._load()
    stream = torch.cuda.current_stream()

    # the same two launches ca_ring_attn_fwd(const max) makes, through the
    # split entry points so that the ring kernel can be timed on its own
    def step():
        st = lib.ca_key_max2(k.data_ptr(), 1, c["B"], c["H"], c["S"], c["D"], kmax2.data_ptr(), stream.cuda_stream)
        assert st == 0, st
        ev_mid = torch.cuda.Event(enable_timing=True)
        ev_mid.record(stream)
        st = lib.ca_ring_attn_fwd_kmax(q.data_ptr(), k.data_ptr(), v.data_ptr(), kmax2.data_ptr(),
                                       o.data_ptr(), lse.data_ptr(), 1, c["B"], c["H"], c["H"], c["S"], c["D"],
                                       c["cp"], 0, 0, 0.0, stream.cuda_stream)
        assert st == 0, st
        return ev_mid

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    def timed():
        evs = []
        with ClockSampler(dev_index) as clk:
            t_start = torch.cuda.Event(enable_timing=True)
            t_start.record(stream)
            prev = t_start
            for _ in range(steps):
                mid = step()
                end = torch.cuda.Event(enable_timing=True)
                end.record(stream)
                evs.append((prev, mid, end))
                prev = end
            torch.cuda.synchronize()
        barrier(pg)
        torch.cuda.synchronize()
        return dict(total_ms=t_start.elapsed_time(prev),
                    ring_ms=statistics.mean([m.elapsed_time(e) for _, m, e in evs]),
                    bound_ms=statistics.mean([s.elapsed_time(m) for s, m, _ in evs]), clocks=clk.summary())

    res = timed_with_retry(timed, pg)
    res["inputs"] = digest
    assert ca.device_status() == 0
    # e2e: through the public API from pinned host memory.  Every step copies
    # its q, k, v host->device and its o device->host inside the timed region;
    # the copies of one step overlap the attention of the previous one (two
    # device buffer sets, one stream per copy direction), as a serving loop
    # would run it.
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    ohs = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    bufs = [dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v), o=torch.empty_like(o),
                 lse=torch.empty_like(lse)) for _ in range(2)]
    del q, k, v, o
    ws = torch.empty(ca.ring_attn_fwd_workspace_size(c["B"], c["H"], c["H"], c["S"], c["D"], c["cp"], "const_max"),
                     dtype=torch.uint8, device="cuda")
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def run_e2e(nsteps):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        h2d_s.wait_event(start)
        d2h_s.wait_event(start)

        def h2d(step):
            b = bufs[step % 2]
            with torch.cuda.stream(h2d_s):
                if step >= 2:
                    h2d_s.wait_event(comp_done[step % 2])  # buffer set free again
                b["q"].copy_(qh, non_blocking=True)
                b["k"].copy_(kh, non_blocking=True)
                b["v"].copy_(vh, non_blocking=True)
                h2d_done[step % 2].record(h2d_s)

        h2d(0)
        for step in range(nsteps):
            b = bufs[step % 2]
            stream.wait_event(h2d_done[step % 2])
            if step >= 2:
                stream.wait_event(d2h_done[step % 2])  # o of this buffer set already read back
            ca.ring_attn_fwd(b["q"], b["k"], b["v"], c["cp"], mode="const_max", out=b["o"], lse=b["lse"],
                             workspace=ws)
            comp_done[step % 2].record(stream)
            if step + 1 < nsteps:
                h2d(step + 1)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(comp_done[step % 2])
                ohs[step % 2].copy_(b["o"], non_blocking=True)
                d2h_done[step % 2].record(d2h_s)
        stream.wait_stream(d2h_s)
        stream.wait_stream(h2d_s)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    run_e2e(3)
    # the host link drops to about a third of its copy bandwidth after a
    # second or two without copies (the device-only timed loop before this)
    # and takes a few hundred milliseconds of traffic to come back: keep the
    # copies going for half a second before the timed steps
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < 0.5:
        run_e2e(10)
    e2e_steps = max(4, min(steps, 40))
    res["e2e_ms"] = run_e2e(e2e_steps) / e2e_steps
    res["h2d_bytes"] = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    res["d2h_bytes"] = ohs[0].numel() * ohs[0].element_size()

    # one call on its own: q, k, v in from pinned host memory, the attention,
    # o back out, all on one stream with nothing before or after it in flight
    # (the latency a caller sees for one request); the host link is still
    # warm from the pipelined loop above
    def single_call():
        b = bufs[0]
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        b["q"].copy_(qh, non_blocking=True)
        b["k"].copy_(kh, non_blocking=True)
        b["v"].copy_(vh, non_blocking=True)
        ca.ring_attn_fwd(b["q"], b["k"], b["v"], c["cp"], mode="const_max", out=b["o"], lse=b["lse"], workspace=ws)
        ohs[0].copy_(b["o"], non_blocking=True)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    single_call()
    res["single_call_ms"] = statistics.median([single_call() for _ in range(max(5, min(steps, 20)))])
    del bufs, qh, kh, vh, ohs
    torch.cuda.empty_cache()
    return res


def bench_decode(ca, torch, steps, warmup, pg, dev_index, cpu_seconds=None):
    from context_attention_gb300 import synth

    c = DECODE
    q, k, v = synth.decode_inputs(c["N"], c["Hq"], c["Hkv"], c["D"], c["W"], c["Lloc"], c["seed"], device="cuda")
    digest = input_digest(c["seed"], q=q, k=k, v=v)
    o = torch.empty_like(q)
    lse = torch.empty(c["N"], c["Hq"], device="cuda", dtype=torch.float32)
    ws = torch.empty(ca.dcp_decode_workspace_size(c["N"], c["Hq"], c["Hkv"], c["Lloc"], c["D"], c["W"], c["I"]),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        ca.dcp_decode(q, k, v, c["I"], out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    barrier(pg)
    torch.cuda.synchronize()
    def timed():
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with ClockSampler(dev_index) as clk:
            a.record(stream)
            for _ in range(steps):
                ca.dcp_decode(q, k, v, c["I"], out=o, lse=lse, workspace=ws)
            b.record(stream)
            torch.cuda.synchronize()
        barrier(pg)
        return dict(ms=a.elapsed_time(b) / steps, clocks=clk.summary())

    res = timed_with_retry(timed, pg)
    res["inputs"] = digest
    assert ca.device_status() == 0
    if cpu_seconds:
        res["cpu_baseline"] = oracle_dcp_decode_baseline(q, k, v, c["I"], cpu_seconds)
    del q, k, v
    torch.cuda.empty_cache()
    return res


class OracleSampler:
    """The fp64 oracle as it stands, on bounded samples of DiT-workload rows
    (inputs drawn once on the host with the same recipe and seed)."""

    def __init__(self, heads=8):
        import numpy as np

        import oracle
        from context_attention_gb300 import synth

        c = PREFILL
        self.oracle, self.np, self.heads = oracle, np, heads
        q, k, v = synth.dit_qk(1, c["H"], c["S"], c["D"], seed=c["seed"], device="cpu")
        self.q, self.k, self.v = (t[:, :heads].float().numpy() for t in (q, k, v))
        self.bound, _ = oracle.const_max_bound(self.q, self.k)
        self.rng = np.random.default_rng(0)

    def run(self, n):
        c = PREFILL
        rows = self.np.sort(self.rng.choice(self.heads * c["S"], size=n, replace=False))
        t0 = time.perf_counter()
        self.oracle.ring(self.q, self.k, self.v, c["cp"], mode=self.oracle.MODE_CONST_MAX, rows=rows, c=self.bound)
        return time.perf_counter() - t0

    def rows_for(self, seconds):
        t = self.run(128)
        return int(min(self.heads * PREFILL["S"], max(64, 128 * seconds / max(t, 1e-6))))

    def measure(self, n):
        t = self.run(n)
        flops = 4.0 * PREFILL["S"] * PREFILL["D"] * n
        threads = self.oracle.num_threads()
        return dict(value=flops / t / 1e12, unit="TFLOP/s", cores=threads, kind="oracle",
                    sample=f"{n} query rows of heads 0-{self.heads - 1} of the DiT workload (const max), "
                    f"{t:.1f} s on {threads} threads", seconds=t)


# ------------------------------------------------- oracle baselines of every workload
# The fp64 oracle as it stands, timed on the host cores on a bounded, seeded
# sample of each workload (inputs copied from the device tensors the GPU
# timing used), reported beside that workload's GPU figure.  Rows (or
# sequences) are independent, so a sample's rate carries over to the whole
# workload by its work count; the sample string says which.


def _oracle_threads():
    import oracle

    return oracle.num_threads()


def _visible_keys(S, cp, layout, causal, rows):
    """Keys each stored query row sees, summed over `rows` (causal: the row's
    global position + 1; otherwise all S)."""
    import numpy as np

    rows = np.asarray(rows, dtype=np.int64)
    if not causal:
        return float(S) * len(rows)
    Ls = S // cp
    g = rows if layout == "contiguous" else (rows % Ls) * cp + rows // Ls
    return float(np.sum(g + 1))


def oracle_ring_baseline(q, k, v, cp, mode, causal, layout, seconds, seed, heads=4):
    """Oracle ring attention on seeded query rows of a few (batch, head)
    pairs; TFLOP/s of visible (query, key) pairs, 4*D FLOP each."""
    import numpy as np

    import oracle

    B, Hq, S, D = q.shape
    G = Hq // k.shape[1]
    rng = np.random.default_rng(seed)
    pairs = [(int(rng.integers(0, B)), int(rng.integers(0, Hq))) for _ in range(heads)]
    omode = oracle.MODE_CONST_MAX if mode == "const_max" else oracle.MODE_ONLINE_MAX
    olay = oracle.LAYOUT_STRIPED if layout == "striped" else oracle.LAYOUT_CONTIGUOUS
    flops = spent = 0.0
    nrows, n = 0, 64
    for i, (b, h) in enumerate(pairs):
        qq = q[b:b + 1, h:h + 1].float().cpu().numpy()
        kk = k[b:b + 1, h // G:h // G + 1].float().cpu().numpy()
        vv = v[b:b + 1, h // G:h // G + 1].float().cpu().numpy()
        cc = oracle.const_max_bound(qq, kk)[0] if omode == oracle.MODE_CONST_MAX else None
        rows = np.sort(rng.choice(S, size=min(n, S), replace=False))
        t0 = time.perf_counter()
        oracle.ring(qq, kk, vv, cp, mode=omode, causal=causal, layout=olay, rows=rows, c=cc)
        dt = time.perf_counter() - t0
        flops += 4.0 * D * _visible_keys(S, cp, layout, causal, rows)
        spent += dt
        nrows += len(rows)
        left = seconds - spent
        if left <= 0 or i + 1 == len(pairs):
            break
        # spread what is left of the budget over the remaining heads
        n = int(max(16, min(S, left / (len(pairs) - i - 1) / (dt / len(rows)))))
    return {"value": round(flops / spent / 1e12, 5), "unit": "TFLOP/s", "cores": _oracle_threads(),
            "kind": "oracle", "seconds": round(spent, 2),
            "sample": f"{nrows} seeded query rows of {i + 1} (batch, head) pairs ({mode}"
                      f"{', causal ' + layout if causal else ''}), {spent:.1f} s; extrapolated to the whole "
                      f"workload by visible keys per row (rows are independent)"}


def oracle_sequence_baseline(nseq, bytes_per_seq, seconds, seed, run_one, what):
    """Oracle decode over sequences in a seeded order until the time budget
    or all of them; GB/s of the K+V bytes the sequences hold.  run_one(n)
    returns the oracle seconds of sequence n (host copies not counted)."""
    import numpy as np

    order = np.random.default_rng(seed).permutation(nseq)
    spent, done = 0.0, 0
    for n in order:
        spent += run_one(int(n))
        done += 1
        if spent >= seconds:
            break
    how = "all of them" if done == nseq else "a seeded subset, extrapolated per sequence"
    return {"value": round(done * bytes_per_seq / spent / 1e9, 3), "unit": "GB/s", "cores": _oracle_threads(),
            "kind": "oracle", "seconds": round(spent, 2),
            "sample": f"{done} of {nseq} sequences ({how}) of the {what}, {spent:.1f} s"}


def oracle_dcp_decode_baseline(q, k, v, interleave, seconds, seed=0):
    import oracle

    W, N, Hkv, Lloc, D = k.shape

    def one(n):
        qq = q[n:n + 1].float().cpu().numpy()
        kk, vv = (t[:, n:n + 1].float().cpu().numpy() for t in (k, v))
        t0 = time.perf_counter()
        oracle.dcp_decode(qq, kk, vv, interleave)
        return time.perf_counter() - t0

    return oracle_sequence_baseline(N, 2.0 * W * Hkv * Lloc * D * 2, seconds, seed, one,
                                    "DCP decode (\"Decode Compute Pattern\")")


def oracle_paged_decode_baseline(q, kc, vc, bt, bs, interleave, seq_len, seconds, seed=0):
    import numpy as np

    import oracle

    W, nblk, Hkv, _, D = kc.shape
    N, mb = bt.shape[1], bt.shape[2]

    def one(n):
        # the sequence's blocks gathered into a small cache of their own, in
        # block-table order, with the matching table
        blocks = bt[:, n].long()
        kk = torch_gather_blocks(kc, blocks).float().cpu().numpy()
        vv = torch_gather_blocks(vc, blocks).float().cpu().numpy()
        tab = np.tile(np.arange(mb, dtype=np.int32), (W, 1)).reshape(W, 1, mb)
        qq = q[n:n + 1].float().cpu().numpy()
        t0 = time.perf_counter()
        oracle.dcp_decode_paged(qq, kk, vv, tab, interleave, [seq_len])
        return time.perf_counter() - t0

    return oracle_sequence_baseline(N, 2.0 * W * Hkv * mb * bs * D * 2, seconds, seed, one,
                                    "paged DCP decode")


def torch_gather_blocks(cache, blocks):
    """cache [W, nblk, ...], blocks [W, m] -> [W, m, ...]: each rank's listed blocks."""
    import torch

    return torch.stack([cache[r].index_select(0, blocks[r]) for r in range(cache.shape[0])])


def oracle_ring_decode_baseline(q, k, v, cp, layout, seconds, seed=0):
    import oracle

    B, Hkv, S, D = k.shape
    olay = oracle.LAYOUT_STRIPED if layout == "striped" else oracle.LAYOUT_CONTIGUOUS

    def one(n):
        qq = q[n:n + 1].float().cpu().numpy()
        kk, vv = (t[n:n + 1].float().cpu().numpy() for t in (k, v))
        t0 = time.perf_counter()
        oracle.ring_decode(qq, kk, vv, cp, olay)
        return time.perf_counter() - t0

    return oracle_sequence_baseline(B, 2.0 * Hkv * S * D * 2, seconds, seed, one, f"Ring Pass-Q decode ({layout})")


def oracle_dcp_prefill_baseline(q, kp, vp, kc, vc, interleave, prior, seconds, seed=0):
    """Oracle DCP prefill on seeded chunk rows; TFLOP/s of visible pairs (a
    chunk row i sees every prior token and chunk tokens 0..i)."""
    import numpy as np

    import oracle

    Hq, Sc, D = q.shape
    host = [t.float().cpu().numpy() for t in (q, kp, vp, kc, vc)]
    rng = np.random.default_rng(seed)
    spent = flops = 0.0
    nrows, n = 0, 32
    while spent < seconds:
        rows = np.sort(rng.choice(Hq * Sc, size=n, replace=False))
        t0 = time.perf_counter()
        oracle.dcp_prefill(*host, interleave, prior, rows=rows)
        dt = time.perf_counter() - t0
        spent += dt
        flops += 4.0 * D * float(np.sum(prior + rows % Sc + 1))
        nrows += n
        n = int(max(16, min(Hq * Sc, (seconds - spent) / (dt / n))))
    return {"value": round(flops / spent / 1e12, 5), "unit": "TFLOP/s", "cores": _oracle_threads(),
            "kind": "oracle", "seconds": round(spent, 2),
            "sample": f"{nrows} seeded chunk rows (with repeats across draws), {spent:.1f} s; extrapolated to "
                      f"the whole chunk by visible keys per row"}


def oracle_prologue_baseline(x_q, x_k, x_v, g_q, g_k, cos, sin, Hq, Hkv, cp, seconds):
    """Oracle QKV prologue on blocks of consecutive tokens (a multiple of cp
    each, rotary tables of their own positions); GB/s of activations read plus
    attention inputs written (bf16), as for the kernel."""
    import oracle

    B, S, _ = x_q.shape
    D = cos.shape[1] * 2
    spent = moved = 0.0
    t0_tok, n = 0, 64
    while spent < seconds and t0_tok + n <= S:
        sl = slice(t0_tok, t0_tok + n)
        xs = [t[:, sl].float().cpu().numpy() for t in (x_q, x_k, x_v)]
        cs, sn = cos[sl].cpu().numpy(), sin[sl].cpu().numpy()
        gq, gk = g_q.cpu().numpy(), g_k.cpu().numpy()
        t0 = time.perf_counter()
        oracle.qk_prologue(xs[0], Hq, g=gq, cos=cs, sin=sn, cp=cp)
        oracle.qk_prologue(xs[1], Hkv, g=gk, cos=cs, sin=sn, cp=cp)
        oracle.qk_prologue(xs[2], Hkv, norm=False, cp=cp)
        dt = time.perf_counter() - t0
        spent += dt
        moved += 2.0 * B * n * (Hq + 2 * Hkv) * D * 2
        t0_tok += n
        n = int(min(S - t0_tok, max(cp, (seconds - spent) / (dt / n)))) // cp * cp
        if n <= 0:
            break
    return {"value": round(moved / spent / 1e9, 3), "unit": "GB/s", "cores": _oracle_threads(), "kind": "oracle",
            "seconds": round(spent, 2),
            "sample": (f"all {S} tokens in blocks, {spent:.1f} s" if t0_tok >= S else
                       f"the first {t0_tok} of {S} tokens in blocks, {spent:.1f} s; extrapolated per token")}


def causal_rank_imbalance(S, cp, layout):
    """Max over mean of the causal work per virtual rank if each rank ran its
    own queries (a multi-GPU ring): rank r's queries sit at the global
    positions of its shard, and query p sees the p + 1 keys 0..p."""
    import numpy as np

    Ls = S // cp
    a = np.arange(Ls, dtype=np.float64)
    work = [float(np.sum((r * Ls + a if layout == "contiguous" else a * cp + r) + 1)) for r in range(cp)]
    return round(max(work) / (sum(work) / cp), 4)


def median_launch_ms(torch, stream, launch, reps):
    """Median of `reps` individually timed launches: CUDA events on the
    launching stream around each, the launches back to back."""
    evs = []
    for i in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        launch(i)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def bench_other_workloads(ca, torch, reps=10, cpu_seconds=None):
    """Device time of the other workloads (online max, sink keys, causal GQA
    in both layouts, the QKV prologue, DCP prefill, paged and Ring Pass-Q
    decode, DCP decode of one and two sequences): the median of `reps`
    individually timed launches (CUDA events), after 3 warm-ups; the one- and
    two-sequence decodes are 10 * reps launches back to back under one pair
    of events.  Each is reported with its algorithmic rate (causal counts
    visible pairs).  With cpu_seconds, each also gets the oracle timed on a
    sample of about that many seconds."""
    from context_attention_gb300 import synth

    res = {}
    stream = torch.cuda.current_stream()

    def run(name, q, k, v, cp, mode, causal, layout, flops):
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], device="cuda", dtype=torch.float32)
        ws = torch.empty(max(16, ca.ring_attn_fwd_workspace_size(q.shape[0], q.shape[1], k.shape[1], q.shape[2],
                                                                 q.shape[3], cp, mode)), dtype=torch.uint8,
                         device="cuda")
        for _ in range(3):
            ca.ring_attn_fwd(q, k, v, cp, mode=mode, causal=causal, layout=layout, out=out, lse=lse, workspace=ws)
        ms = median_launch_ms(torch, stream, lambda i: ca.ring_attn_fwd(q, k, v, cp, mode=mode, causal=causal,
                                                                      layout=layout, out=out, lse=lse,
                                                                      workspace=ws), reps)
        res[name] = {"ms": round(ms, 3), "tflops": round(flops / (ms / 1e3) / 1e12, 1)}
        if cpu_seconds:
            res[name]["cpu_baseline"] = oracle_ring_baseline(q, k, v, cp, mode, causal, layout, cpu_seconds,
                                                             seed=len(res))

    q, k, v = synth.normal_qkv(2, 32, 32, 32768, 128, 3, dtype=torch.bfloat16, device="cuda")
    f = 4.0 * 2 * 32 * 32768 ** 2 * 128
    run("online_max B2 H32 S32768 cp8", q, k, v, 8, "online_max", False, "contiguous", f)
    run("const_max B2 H32 S32768 cp8", q, k, v, 8, "const_max", False, "contiguous", f)
    k = synth.apply_sinks(k, synth.sink_rows(2, 32768, seed=33, device="cuda"))
    run("online_max sinks B2 H32 S32768 cp8", q, k, v, 8, "online_max", False, "contiguous", f)
    del q, k, v
    q, k, v = synth.normal_qkv(1, 32, 8, 65536, 128, 4, dtype=torch.bfloat16, device="cuda")
    f = 4.0 * 32 * 128 * 65536 * 65537 / 2
    for layout in ("contiguous", "striped"):
        name = f"causal GQA {layout} Hq32 Hkv8 S65536 cp8"
        run(name, q, k, v, 8, "online_max", True, layout, f)
        res[name]["virtual_rank_imbalance"] = causal_rank_imbalance(65536, 8, layout)
    del q, k, v
    torch.cuda.empty_cache()
    # QKV prologue of the DiT workload (B1, S16384, 40 heads of 128, cp8):
    # whole-hidden RMS norm + gains + rotary turn for q and k, head split for
    # v, kmax2 of k; HBM bytes = activations read + outputs written + tables
    B, S, H, D = 1, 16384, 40, 128
    x_q, x_k, x_v, g_q, g_k, cos, sin = [t.cuda() for t in synth.qkv_activations(B, S, H, H, D, 27)]
    for _ in range(3):
        ca.qkv_prologue(x_q, x_k, H, H, x_v=x_v, g_q=g_q, g_k=g_k, rope_cos=cos, rope_sin=sin, cp_size=8)
    torch.cuda.synchronize()
    outs = [ca.qkv_prologue(x_q, x_k, H, H, x_v=x_v, g_q=g_q, g_k=g_k, rope_cos=cos, rope_sin=sin, cp_size=8)
            for _ in range(2)]  # two output sets (> L2 together) so no rep reads the previous one's lines
    def prologue_launch(i):
        o = outs[i % 2]
        st = ca._load().ca_qkv_prologue(x_q.data_ptr(), x_k.data_ptr(), x_v.data_ptr(), g_q.data_ptr(),
                                        g_k.data_ptr(), 1e-6, cos.data_ptr(), sin.data_ptr(), 1, B, S, H, H, D, 8, 0,
                                        o[0].data_ptr(), o[1].data_ptr(), o[2].data_ptr(), o[3].data_ptr(),
                                        stream.cuda_stream)
        assert st == 0, st

    ms = median_launch_ms(torch, stream, prologue_launch, 2 * reps)
    nbytes = 6 * B * S * H * D * 2 + 2 * S * (D // 2) * 4
    res["qkv_prologue DiT B1 S16384 H40"] = {"ms": round(ms, 4), "gbs": round(nbytes / (ms / 1e3) / 1e9, 1)}
    if cpu_seconds:
        res["qkv_prologue DiT B1 S16384 H40"]["cpu_baseline"] = oracle_prologue_baseline(
            x_q, x_k, x_v, g_q, g_k, cos, sin, H, H, 8, cpu_seconds)
    del x_q, x_k, x_v, outs
    torch.cuda.empty_cache()
    # DCP prefill: an 8192-token chunk after 122880 cached tokens, dcp=4, I=16
    Hq, Hkv, W, I, Sc, P = 32, 8, 4, 16, 8192, 122880
    q, kp, vp, kc, vc = synth.dcp_prefill_inputs(Hq, Hkv, 128, W, Sc, P // W, Sc // W, 6, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(Hq, Sc, device="cuda", dtype=torch.float32)
    for _ in range(3):
        ca.dcp_prefill(q, kp, vp, kc, vc, I, P, out=out, lse=lse)
    ms = median_launch_ms(torch, stream, lambda i: ca.dcp_prefill(q, kp, vp, kc, vc, I, P, out=out, lse=lse), reps)
    f = 4.0 * 128 * Hq * (Sc * P + Sc * (Sc + 1) / 2)
    res["dcp_prefill Hq32 Hkv8 chunk8192 prior122880 dcp4"] = {"ms": round(ms, 3),
                                                               "tflops": round(f / (ms / 1e3) / 1e12, 1)}
    if cpu_seconds:
        res["dcp_prefill Hq32 Hkv8 chunk8192 prior122880 dcp4"]["cpu_baseline"] = oracle_dcp_prefill_baseline(
            q, kp, vp, kc, vc, I, P, cpu_seconds)
    del q, kp, vp, kc, vc
    torch.cuda.empty_cache()
    # paged DCP decode: the decode workload's 34 GB of K/V in 16-slot blocks
    # scattered over each rank's cache by a random block table
    d = DECODE
    bs = 16
    mb = d["Lloc"] // bs
    nblk = d["N"] * mb
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    q = torch.randn(d["N"], d["Hq"], d["D"], generator=g, device="cuda").to(torch.bfloat16)
    kc = torch.empty(d["W"], nblk, d["Hkv"], bs, d["D"], device="cuda", dtype=torch.bfloat16)
    vc = torch.empty_like(kc)
    for t in (kc, vc):
        for r in range(d["W"]):
            t[r].copy_(torch.randn(nblk, d["Hkv"], bs, d["D"], generator=g, device="cuda").to(torch.bfloat16))
    bt = torch.stack([torch.randperm(nblk, generator=g, device="cuda").view(d["N"], mb)
                      for _ in range(d["W"])]).to(torch.int32).contiguous()
    sl = torch.full((d["N"],), d["W"] * d["Lloc"], dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(d["N"], d["Hq"], device="cuda", dtype=torch.float32)
    ws = torch.empty(ca.dcp_decode_workspace_size(d["N"], d["Hq"], d["Hkv"], d["Lloc"], d["D"], d["W"], d["I"]),
                     dtype=torch.uint8, device="cuda")
    for _ in range(3):
        ca.dcp_decode_paged(q, kc, vc, bt, d["I"], sl, out=out, lse=lse, workspace=ws)
    ms = median_launch_ms(torch, stream, lambda i: ca.dcp_decode_paged(q, kc, vc, bt, d["I"], sl, out=out, lse=lse,
                                                                     workspace=ws), reps)
    res["dcp_decode_paged bs16 64seqs L131072 dcp4"] = {"ms": round(ms, 3),
                                                        "gbs": round(decode_bytes() / (ms / 1e3) / 1e9, 1)}
    if cpu_seconds:
        res["dcp_decode_paged bs16 64seqs L131072 dcp4"]["cpu_baseline"] = oracle_paged_decode_baseline(
            q, kc, vc, bt, bs, d["I"], d["W"] * d["Lloc"], cpu_seconds)
    del q, kc, vc, bt
    torch.cuda.empty_cache()
    # Ring Pass-Q decode: the decode workload's sequences and 34 GB of K/V,
    # held in the ring prefill's layout ([B, Hkv, S, D], striped over 8 shards)
    S = d["W"] * d["Lloc"]
    q = torch.randn(d["N"], d["Hq"], d["D"], generator=g, device="cuda").to(torch.bfloat16)
    kr = torch.empty(d["N"], d["Hkv"], S, d["D"], device="cuda", dtype=torch.bfloat16)
    vr = torch.empty_like(kr)
    for t in (kr, vr):
        for n in range(d["N"]):
            t[n].copy_(torch.randn(d["Hkv"], S, d["D"], generator=g, device="cuda").to(torch.bfloat16))
    ws = torch.empty(ca.ring_decode_workspace_size(d["N"], d["Hq"], d["Hkv"], S, d["D"], 8), dtype=torch.uint8,
                     device="cuda")
    for _ in range(3):
        ca.ring_decode(q, kr, vr, 8, layout="striped", out=out, lse=lse, workspace=ws)
    ms = median_launch_ms(torch, stream, lambda i: ca.ring_decode(q, kr, vr, 8, layout="striped", out=out, lse=lse,
                                                                workspace=ws), reps)
    res["ring_decode striped cp8 64seqs L131072"] = {"ms": round(ms, 3),
                                                     "gbs": round(decode_bytes() / (ms / 1e3) / 1e9, 1)}
    if cpu_seconds:
        res["ring_decode striped cp8 64seqs L131072"]["cpu_baseline"] = oracle_ring_decode_baseline(
            q, kr, vr, 8, "striped", cpu_seconds)
    del q, kr, vr
    torch.cuda.empty_cache()
    # small-batch DCP decode: one and two of the decode workload's sequences
    # (537 MB and 1.07 GB of K/V, more than L2; launches back to back)
    for nseq in (1, 2):
        q, kd, vd = synth.decode_inputs(nseq, d["Hq"], d["Hkv"], d["D"], d["W"], d["Lloc"], 8 + nseq,
                                        device="cuda")
        out = torch.empty_like(q)
        lse = torch.empty(nseq, d["Hq"], device="cuda", dtype=torch.float32)
        ws = torch.empty(ca.dcp_decode_workspace_size(nseq, d["Hq"], d["Hkv"], d["Lloc"], d["D"], d["W"], d["I"]),
                         dtype=torch.uint8, device="cuda")
        for _ in range(3):
            ca.dcp_decode(q, kd, vd, d["I"], out=out, lse=lse, workspace=ws)
        # one pair of events around all launches: an event between two of
        # them would cut the programmatic dependency that lets each decode
        # set up while the previous one's merge runs
        n_launch = 10 * reps
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n_launch):
            ca.dcp_decode(q, kd, vd, d["I"], out=out, lse=lse, workspace=ws)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / n_launch
        nbytes = 2.0 * d["W"] * nseq * d["Hkv"] * d["Lloc"] * d["D"] * 2
        name = f"dcp_decode {nseq}seq L131072 dcp4"
        res[name] = {"ms": round(ms, 4), "gbs": round(nbytes / (ms / 1e3) / 1e9, 1)}
        if cpu_seconds:
            res[name]["cpu_baseline"] = oracle_dcp_decode_baseline(q, kd, vd, d["I"], cpu_seconds)
        del q, kd, vd
        torch.cuda.empty_cache()
    return res


def cpu_baseline_prefill(seconds=15.0):
    smp = OracleSampler()
    return smp.measure(smp.rows_for(seconds))


def run_profile_case(args):
    """One small launch of one kernel, for ncu captures (inputs > L2, a few GB)."""
    import torch

    import context_attention_gb300 as ca
    from context_attention_gb300 import synth

    torch.cuda.set_device(0)
    if args.profile in ("ring", "ring_dit"):
        # DiT recipe with 16 heads: q,k,v 201 MB (> L2), one launch ~1.2 ms;
        # ring_dit: the bench workload itself (40 heads, q,k,v 503 MB), ~3.2 ms
        heads = PREFILL["H"] if args.profile == "ring_dit" else 16
        q, k, v = synth.dit_qk(1, heads, PREFILL["S"], PREFILL["D"], seed=PREFILL["seed"], device="cuda")
        km = ca.key_max2(k)
        for _ in range(args.warmup + 1):
            ca.ring_attn_fwd_kmax(q, k, v, km, PREFILL["cp"])
    elif args.profile in ("causal_contiguous", "causal_striped"):
        # the causal GQA workload itself (B1 Hq32 Hkv8 S65536 D128, cp8, online
        # max): q,k,v 805 MB (> L2), one launch ~22 ms
        q, k, v = synth.normal_qkv(1, 32, 8, 65536, 128, 4, dtype=torch.bfloat16, device="cuda")
        layout = args.profile.split("_")[1]
        for _ in range(args.warmup + 1):
            ca.ring_attn_fwd(q, k, v, 8, mode="online_max", causal=True, layout=layout)
    elif args.profile == "prologue":
        # the DiT prologue (B1 S16384 40 heads): 1 GB moved per launch (> L2), ~0.2 ms
        B, S, H, D = 1, PREFILL["S"], PREFILL["H"], PREFILL["D"]
        x_q, x_k, x_v, g_q, g_k, cos, sin = [t.cuda() for t in synth.qkv_activations(B, S, H, H, D, 27)]
        for _ in range(args.warmup + 1):
            ca.qkv_prologue(x_q, x_k, H, H, x_v=x_v, g_q=g_q, g_k=g_k, rope_cos=cos, rope_sin=sin,
                            cp_size=PREFILL["cp"])
    elif args.profile == "key_pass":
        # the DiT workload's key pass: k is 167.8 MB (> L2), one launch ~35 us
        _, k, _ = synth.dit_qk(1, PREFILL["H"], PREFILL["S"], PREFILL["D"], seed=PREFILL["seed"], device="cuda")
        for _ in range(args.warmup + 1):
            ca.key_max2(k)
    elif args.profile == "merge":
        # a standalone LSE merge too large for L2: 8 partials of 131072 rows x 128
        # (537 MB of fp32 partials), bf16 output
        n, R, D = 8, 131072, 128
        g = torch.Generator(device="cuda")
        g.manual_seed(8)
        o_parts = torch.randn(n, R, D, generator=g, device="cuda")
        lse_parts = torch.randn(n, R, generator=g, device="cuda") * 4
        for _ in range(args.warmup + 1):
            ca.lse_merge(o_parts, lse_parts, out_dtype=torch.bfloat16)
    elif args.profile == "paged":
        # paged decode with 8 sequences (256 shard x sequence x KV-head pairs,
        # dealt in splits as the 64-sequence workload is) in 16-slot blocks
        # under a random block table: K+V 4.3 GB (> L2), one launch ~0.6 ms
        d = DECODE
        ns = 8
        q, kd, vd = synth.decode_inputs(ns, d["Hq"], d["Hkv"], d["D"], d["W"], d["Lloc"], d["seed"], device="cuda")
        bs, mb = 16, d["Lloc"] // 16
        g = torch.Generator(device="cuda")
        g.manual_seed(7)
        perm = torch.stack([torch.randperm(ns * mb, generator=g, device="cuda") for _ in range(d["W"])])
        kc = torch.empty(d["W"], ns * mb, d["Hkv"], bs, d["D"], device="cuda", dtype=torch.bfloat16)
        vc = torch.empty_like(kc)
        for src, dst in ((kd, kc), (vd, vc)):
            blocks = src.view(d["W"], ns, d["Hkv"], mb, bs, d["D"]).permute(0, 1, 3, 2, 4, 5).reshape(
                d["W"], ns * mb, d["Hkv"], bs, d["D"])
            for r in range(d["W"]):
                dst[r].index_copy_(0, perm[r], blocks[r])
        bt = perm.view(d["W"], ns, mb).to(torch.int32).contiguous()
        del kd, vd, blocks
        torch.cuda.empty_cache()
        sl = torch.full((ns,), d["W"] * d["Lloc"], dtype=torch.int32, device="cuda")
        for _ in range(args.warmup + 1):
            ca.dcp_decode_paged(q, kc, vc, bt, d["I"], sl)
    elif args.profile == "ring_decode":
        # Ring Pass-Q decode of 4 sequences of 131072 tokens, striped over 8
        # shards: K+V 2.1 GB (> L2), one launch ~0.3 ms
        d = DECODE
        g = torch.Generator(device="cuda")
        g.manual_seed(9)
        S = d["W"] * d["Lloc"]
        q = torch.randn(4, d["Hq"], d["D"], generator=g, device="cuda").to(torch.bfloat16)
        kr = torch.randn(4, d["Hkv"], S, d["D"], generator=g, device="cuda").to(torch.bfloat16)
        vr = torch.randn(4, d["Hkv"], S, d["D"], generator=g, device="cuda").to(torch.bfloat16)
        for _ in range(args.warmup + 1):
            ca.ring_decode(q, kr, vr, 8, layout="striped")
    else:
        # decode recipe with 8 sequences (256 pairs, dealt in splits as the
        # 64-sequence workload is): K+V 4.3 GB (> L2), one launch ~0.6 ms;
        # decode_small: one sequence (contiguous ranges), 537 MB, ~90 us
        d = DECODE
        ns = 1 if args.profile == "decode_small" else 8
        q, kd, vd = synth.decode_inputs(ns, d["Hq"], d["Hkv"], d["D"], d["W"], d["Lloc"], d["seed"], device="cuda")
        for _ in range(args.warmup + 1):
            ca.dcp_decode(q, kd, vd, d["I"])
    torch.cuda.synchronize()
    assert ca.device_status() == 0
    print(f"profile case {args.profile} done")


def run_ours(args):
    import torch

    rank, world, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    import context_attention_gb300 as ca

    ca._load()
    peaks, peak_src = load_peaks()
    pre = bench_prefill(ca, torch, args.steps, args.warmup, pg, local)
    cpu_each = None if (rank != 0 or args.no_cpu_baseline) else args.cpu_seconds_each
    dec = None if args.skip_decode else bench_decode(ca, torch, args.steps, args.warmup, pg, local, cpu_each)

    total_ms = max_over_ranks(pre["total_ms"], pg)
    ms_per_step = total_ms / args.steps
    flops = prefill_flops()
    value = aggregate_throughput(flops, args.steps, world, total_ms) / 1e12
    long_run = total_ms > 2000.0
    peak = peaks["bf16_tflops_sustained"] if long_run else peaks["bf16_tflops"]
    ring_tflops = flops / (pre["ring_ms"] / 1e3) / 1e12
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; cross-head RMS-normalised q/k, N(0,1) v)",
        "config": {"workload": "DiT const-max ring self-attention prefill", "B": PREFILL["B"], "H": PREFILL["H"],
                   "S": PREFILL["S"], "D": PREFILL["D"], "cp_size": PREFILL["cp"], "mode": "const_max",
                   "layout": "contiguous", "causal": False, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (no flush)", "inputs": pre["inputs"]},
        "pct_of_bf16_peak": round(100.0 * value / world / peak, 2),
        "roofline": {"kernel": "ring_tc_kernel", "bound": "tensor", "achieved": round(ring_tflops, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(ring_tflops / peak, 4),
                     "traffic": read_traffic("ring_tc_kernel_dit40h.txt"),
                     "peak_source": f"{peak_src} {'sustained' if long_run else 'burst'} bf16 "
                                    f"(timed region {total_ms / 1e3:.2f} s)",
                     "frac_of_burst": round(ring_tflops / peaks["bf16_tflops"], 4),
                     "frac_of_sustained": round(ring_tflops / peaks["bf16_tflops_sustained"], 4),
                     "frac_of_nominal": round(ring_tflops / NOMINAL_BF16_TFLOPS, 4),
                     "key_pass_ms": round(pre["bound_ms"], 4), "ring_ms": round(pre["ring_ms"], 4)},
        "clocks": pre["clocks"],
        "e2e": {"value": round(flops / (pre["e2e_ms"] / 1e3) / 1e12 * world, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": pre["h2d_bytes"], "d2h_bytes_per_step": pre["d2h_bytes"],
                "ms_per_step": round(pre["e2e_ms"], 3),
                "how": "pipelined: each step's copies overlap the previous step's attention",
                "single_call": {"value": round(flops / (pre["single_call_ms"] / 1e3) / 1e12, 2),
                                "unit": "TFLOP/s", "ms": round(pre["single_call_ms"], 3),
                                "h2d_bytes": pre["h2d_bytes"], "d2h_bytes": pre["d2h_bytes"],
                                "how": "one call alone: copy in, attention, copy out on one stream "
                                       "(median of repeated calls)"}},
        "gpu_launches": 2 * args.steps + (2 * args.steps if dec else 0),
    }
    if dec:
        dms = max_over_ranks(dec["ms"], pg)
        gbs = decode_bytes() / (dms / 1e3) / 1e9
        out["decode"] = {"workload": "DCP decode: 64 seqs x 1 token, Hq=32, Hkv=8, D=128, L=131072, dcp=4, I=16",
                         "value": round(gbs * world, 1), "unit": "GB/s", "ms_per_step": round(dms, 4),
                         "pct_of_hbm": round(100.0 * gbs / peaks["hbm_gbs"], 2),
                         "pct_of_nominal_hbm": round(100.0 * gbs / NOMINAL_HBM_GBS, 2),
                         "roofline": {"kernel": "dcp_decode_kernel + lse_merge_kernel", "bound": "hbm",
                                      "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                      "frac": round(gbs / peaks["hbm_gbs"], 4),
                                      "traffic": read_traffic("dcp_decode_kernel_131k.txt"),
                                      "peak_source": f"{peak_src} copy bandwidth",
                                      "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                                      "note": "the measured peak is a copy (half its bytes written); "
                                              "a read-only stream can pass it, so frac above 1 is "
                                              "possible: frac_of_nominal is against the 8 TB/s "
                                              "datasheet rate"},
                         "clocks": dec["clocks"], "inputs": dec["inputs"]}
        if "cpu_baseline" in dec:
            out["decode"]["cpu_baseline"] = dec["cpu_baseline"]
    # the other workloads ride along on single-GPU runs (about 20 s more); a
    # failure there is reported in the line rather than losing the line
    if args.other_workloads or (world == 1 and not args.no_other_workloads):
        try:
            ow = bench_other_workloads(ca, torch, cpu_seconds=cpu_each)
            # each workload's rate against the same measured peaks as the headline
            for w in ow.values():
                if "tflops" in w:
                    w["frac_of_burst_bf16"] = round(w["tflops"] / peaks["bf16_tflops"], 4)
                if "gbs" in w:
                    w["frac_of_copy_bw"] = round(w["gbs"] / peaks["hbm_gbs"], 4)
            out["other_workloads"] = ow
        except Exception as e:  # noqa: BLE001 -- report, keep the headline
            out["other_workloads"] = {"error": f"{type(e).__name__}: {e}"}
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_prefill(seconds=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if pg is not None:
        pg.destroy_process_group()


# --------------------------------------------------------------------------- reference arm


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    smp = OracleSampler()
    # each step: a bounded sample sized so the whole run stays within ~2 minutes
    per_step = max(0.1, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    n = smp.rows_for(per_step)
    for _ in range(args.warmup):
        smp.run(n)
    vals, secs, last = [], [], None
    for _ in range(args.steps):
        last = smp.measure(n)
        vals.append(last["value"])
        secs.append(last["seconds"])
    value = statistics.mean(vals)
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(secs),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; cross-head RMS-normalised q/k, N(0,1) v)",
        "config": {"workload": "DiT const-max ring self-attention prefill", "B": PREFILL["B"], "H": PREFILL["H"],
                   "S": PREFILL["S"], "D": PREFILL["D"], "cp_size": PREFILL["cp"], "mode": "const_max",
                   "layout": "contiguous", "causal": False, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                         "sample": f"each step: {last['sample']}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--other-workloads", action="store_true",
                    help="time the other workloads (online max, sinks, causal GQA, prologue, DCP prefill, paged "
                         "and ring decode; reported, not the value) also when running on several GPUs")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the other workloads on a single-GPU run (they run by default there)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="oracle seconds of the headline workload's CPU baseline")
    ap.add_argument("--cpu-seconds-each", type=float, default=3.0,
                    help="oracle seconds of each other workload's CPU baseline (decode and other_workloads)")
    ap.add_argument("--profile", choices=["ring", "ring_dit", "causal_contiguous", "causal_striped", "decode",
                                          "decode_small", "prologue", "key_pass", "merge", "paged", "ring_decode"],
                    default=None,
                    help="run one small launch of one kernel (for ncu captures) and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.profile:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
