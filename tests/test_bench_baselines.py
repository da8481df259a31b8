"""The bench's oracle baselines (one per workload in the JSON line) on small
host tensors: each returns a complete cpu_baseline object -- a positive rate
in the workload's own unit, the oracle's thread count, and a sample string
that says what was timed and how it is extrapolated."""
import pytest
import torch

import bench
from context_attention_gb300 import synth


def check(cb, unit):
    assert cb["kind"] == "oracle" and cb["unit"] == unit
    assert cb["value"] > 0 and cb["cores"] >= 1 and cb["seconds"] >= 0
    assert isinstance(cb["sample"], str) and cb["sample"]


@pytest.mark.parametrize("mode,causal,layout", [("online_max", False, "contiguous"), ("const_max", False, "contiguous"),
                                                ("online_max", True, "contiguous"), ("online_max", True, "striped")])
def test_ring_baseline(mode, causal, layout):
    q, k, v = synth.normal_qkv(1, 4, 2, 512, 128, 1, dtype=torch.bfloat16)
    cb = bench.oracle_ring_baseline(q, k, v, 4, mode, causal, layout, 0.2, seed=1)
    check(cb, "TFLOP/s")
    assert "extrapolated" in cb["sample"]


def test_visible_keys_counts_causal_pairs():
    import numpy as np

    S, cp = 64, 4
    rows = np.arange(S)
    assert bench._visible_keys(S, cp, "contiguous", False, rows) == S * S
    # every layout's rows cover the positions 0..S-1 once: S(S+1)/2 pairs
    for layout in ("contiguous", "striped"):
        assert bench._visible_keys(S, cp, layout, True, rows) == S * (S + 1) / 2
    # stored row 1 of a striped layout is shard 0's second token, global position cp
    assert bench._visible_keys(S, cp, "striped", True, [1]) == cp + 1


def test_decode_baselines():
    q, k, v = synth.decode_inputs(3, 8, 2, 128, 4, 256, 5)
    cb = bench.oracle_dcp_decode_baseline(q, k, v, 16, 0.05)
    check(cb, "GB/s")
    kr = torch.randn(3, 2, 1024, 128).to(torch.bfloat16)
    check(bench.oracle_ring_decode_baseline(q, kr, kr, 8, "striped", 0.05), "GB/s")
    bs, mb = 16, 16
    kc = torch.randn(4, 3 * mb, 2, bs, 128).to(torch.bfloat16)
    bt = torch.stack([torch.randperm(3 * mb).view(3, mb) for _ in range(4)]).to(torch.int32)
    check(bench.oracle_paged_decode_baseline(q, kc, kc, bt, bs, 16, 4 * 256, 0.05), "GB/s")


def test_paged_baseline_gathers_each_sequences_blocks():
    """The paged baseline hands the oracle a per-sequence cache gathered in
    block-table order: it must decode to what the oracle gives on the whole
    paged cache."""
    import numpy as np

    import oracle

    q, _, _ = synth.decode_inputs(2, 4, 2, 128, 2, 64, 9)
    bs, mb = 16, 4
    kc = torch.randn(2, 2 * mb, 2, bs, 128).to(torch.bfloat16)
    vc = torch.randn(2, 2 * mb, 2, bs, 128).to(torch.bfloat16)
    bt = torch.stack([torch.randperm(2 * mb).view(2, mb) for _ in range(2)]).to(torch.int32)
    full, _ = oracle.dcp_decode_paged(q.float().numpy(), kc.float().numpy(), vc.float().numpy(), bt.numpy(), 16,
                                      [128, 128])
    blocks = bt[:, 1].long()
    kk = bench.torch_gather_blocks(kc, blocks).float().numpy()
    vv = bench.torch_gather_blocks(vc, blocks).float().numpy()
    tab = np.tile(np.arange(mb, dtype=np.int32), (2, 1)).reshape(2, 1, mb)
    one, _ = oracle.dcp_decode_paged(q[1:2].float().numpy(), kk, vv, tab, 16, [128])
    assert np.array_equal(one[0], full[1])


def test_prefill_and_prologue_baselines():
    q, kp, vp, kc, vc = synth.dcp_prefill_inputs(8, 2, 128, 4, 256, 256, 64, 6)
    check(bench.oracle_dcp_prefill_baseline(q, kp, vp, kc, vc, 16, 1024, 0.1), "TFLOP/s")
    x_q, x_k, x_v, g_q, g_k, cos, sin = synth.qkv_activations(1, 256, 4, 4, 128, 27)
    check(bench.oracle_prologue_baseline(x_q, x_k, x_v, g_q, g_k, cos, sin, 4, 4, 8, 0.1), "GB/s")


def test_roofline_traffic_comes_from_committed_profiles():
    """The bench reports each roofline's DRAM traffic from an ncu summary
    under profiles/: every file it names exists and carries a per-launch
    figure, and the figure is within a few per cent of the kernel's
    algorithmic bytes (the ring kernel's q, k, v read and o, lse written at
    the DiT size; the decode's valid K+V), so a renamed or stale summary
    fails here rather than turning the field null."""
    import inspect
    import re

    src = inspect.getsource(bench)
    names = re.findall(r'read_traffic\("([^"]+)"\)', src)
    assert names, "bench.py reads no traffic figure"
    algorithmic = {
        "ring_tc_kernel_dit40h.txt": (3 * 40 * 16384 * 128 * 2) + (40 * 16384 * 128 * 2 + 40 * 16384 * 4),
        "dcp_decode_kernel_131k.txt": 2 * 4 * 64 * 8 * 32768 * 128 * 2,
    }
    for name in names:
        v = bench.read_traffic(name)
        assert v is not None, f"profiles/{name} has no traffic_bytes_per_launch"
        if name in algorithmic:
            assert abs(v / algorithmic[name] - 1.0) < 0.05, (name, v, algorithmic[name])
