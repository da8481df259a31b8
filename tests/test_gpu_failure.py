"""Failure detection on the GPU without a fault: a bounded wait that runs out
(on a barrier nothing completes) raises the device error word, the host reads
CA_ERR_TIMEOUT through ca_device_status, and the context stays usable."""
import pytest
import torch

import oracle
from helpers import assert_close, np32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ca(cuda_device):
    import context_attention_gb300 as m

    m.build()
    yield m
    assert m.device_status() == 0, "a bounded device wait gave up"


def test_a_wait_that_runs_out_is_reported_and_the_context_survives(ca):
    timeout = {v: k for k, v in ca.STATUS.items()}["CA_ERR_TIMEOUT"]
    assert ca.device_status() == 0
    ca.selftest_wait_timeout(2_000_000)  # ~1 ms of SM cycles
    torch.cuda.synchronize()
    assert ca.device_status(reset=False) == timeout
    assert ca.device_status() == timeout  # read and clear
    assert ca.device_status() == 0
    # the same context keeps working
    from context_attention_gb300 import synth

    q, k, v = synth.normal_qkv(1, 2, 2, 512, 128, 81, dtype=torch.bfloat16, device="cuda")
    o, lse = ca.ring_attn_fwd(q, k, v, 2, mode="online_max", causal=True)
    ro, rl, _ = oracle.ring(np32(q), np32(k), np32(v), 2, causal=True)
    assert_close(np32(o), ro, np32(lse), rl, what="ring after a reported timeout")
    assert ca.device_status() == 0
