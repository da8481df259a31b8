"""The allocation-free DCP decode entry point (ca_dcp_decode_noalloc).

It serves callers that cannot allocate device memory when they call us: the
partials live in a scratch array built into the library instead of a
caller-provided workspace.  Its results must match the regular entry point,
call after call, even though every call reuses the same scratch.  This file
is collected last so that a failure here never hides the other tests."""
import numpy as np
import pytest
import torch

from helpers import assert_close, np32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ca(cuda_device):
    import context_attention_gb300 as m

    m.build()
    yield m
    assert m.device_status() == 0, "a bounded device wait gave up"


def test_noalloc_matches_regular_decode_twice_in_a_row(ca):
    from context_attention_gb300 import synth

    cases = [
        # (N, Hq, Hkv, dcp, interleave, Lloc, seq_lens, seed)
        (4, 8, 2, 4, 16, 2048, [8192, 17, 5000, 1], 21),
        (3, 32, 8, 2, 16, 9000 - 9000 % 16, [17984, 12345, 640], 22),
        # 31 shards x 32 sequences x 32 heads: the partials fill 97.6 % of the
        # 16 MiB scratch, so the last partial slots and the log-sum-exps at
        # the top of the array are written and read
        (32, 32, 4, 31, 16, 128, None, 24),
    ]
    lib = ca._load()
    for N, Hq, Hkv, W, I, Lloc, lens, seed in cases:
        q, k, v = synth.decode_inputs(N, Hq, Hkv, 128, W, Lloc, seed, device="cuda")
        if lens is None:
            lens = [int(x) for x in np.random.default_rng(seed).integers(0, W * Lloc + 1, size=N)]
        need = ca.dcp_decode_workspace_size(N, Hq, Hkv, Lloc, 128, W, I)
        assert need <= (16 << 20)
        sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
        ref_o, ref_l = ca.dcp_decode(q, k, v, I, seq_lens=sl)
        out = torch.empty_like(q)
        lse = torch.empty(N, Hq, device="cuda", dtype=torch.float32)
        stream = torch.cuda.current_stream().cuda_stream
        for _ in range(2):  # the second call runs on the first call's leftover scratch
            out.fill_(float("nan"))
            lse.fill_(float("nan"))
            st = lib.ca_dcp_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), 1, N, Hq, Hkv, Lloc, 128,
                                           W, I, sl.data_ptr(), 0.0, out.data_ptr(), lse.data_ptr(), stream)
            assert ca.STATUS[st] == "CA_OK"
            torch.cuda.synchronize()
            assert_close(np32(out), np32(ref_o).astype(np.float64), np32(lse), np32(ref_l).astype(np.float64),
                         what=f"noalloc vs regular decode, {need} bytes of partials")
        # without the optional lse output
        out.fill_(float("nan"))
        st = lib.ca_dcp_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), 1, N, Hq, Hkv, Lloc, 128,
                                       W, I, sl.data_ptr(), 0.0, out.data_ptr(), None, stream)
        assert ca.STATUS[st] == "CA_OK"
        torch.cuda.synchronize()
        assert_close(np32(out), np32(ref_o).astype(np.float64), what="noalloc without lse")


def test_noalloc_rejects_problems_beyond_its_scratch(ca):
    from context_attention_gb300 import synth

    N, Hq, Hkv, W, Lloc = 64, 32, 8, 4, 32768  # partials need ~34 MB > 16 MiB
    assert ca.dcp_decode_workspace_size(N, Hq, Hkv, Lloc, 128, W, 16) > (16 << 20)
    q, _, _ = synth.decode_inputs(N, Hq, Hkv, 128, 1, 128, 23, device="cuda")
    # tiny real buffers stand in for the caches and the output: the size
    # check rejects the call before anything is enqueued, so they are never
    # read or written
    k = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    o = torch.zeros_like(k)
    lib = ca._load()
    st = lib.ca_dcp_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), 1, N, Hq, Hkv, Lloc, 128, W, 16, None,
                                   0.0, o.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert ca.STATUS[st] == "CA_ERR_WORKSPACE"
    assert int(o.abs().sum().item()) == 0
