"""GPU parity of DCP prefill (segmented attention over each rank's prior +
current local KV, causal by global position, LSE-merged) against the fp64
oracle, through the C ABI."""
import numpy as np
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


def make(ca, Hq, Hkv, W, I, Sc, P, seed, pad=24, poison=True):
    from context_attention_gb300 import synth

    Lcap = ca.dcp_local_filled(P, W, I, I, 0) + pad
    Lc = ca.dcp_local_filled(Sc, W, I, I, 0) + pad
    q, kp, vp, kc, vc = synth.dcp_prefill_inputs(Hq, Hkv, 128, W, Sc, Lcap, Lc, seed, device="cuda")
    if poison:
        # slots a rank does not hold: never read (NaN would poison the result)
        for R in range(W):
            lp = ca.dcp_local_filled(P, W, I, I, R)
            lc = ca.dcp_local_filled(Sc, W, I, I, R)
            kp[R, :, lp:] = float("nan")
            vp[R, :, lp:] = float("nan")
            kc[R, :, lc:] = float("nan")
            vc[R, :, lc:] = float("nan")
    return q, kp, vp, kc, vc


def clean(t):
    return np32(torch.nan_to_num(t))


@pytest.mark.parametrize("Sc,P", [(512, 0), (512, 64), (320, 1000), (200, 1072), (1024, 4096)])
def test_dcp_prefill_matches_oracle(ca, Sc, P):
    Hq, Hkv, W, I = 4, 2, 4, 16
    q, kp, vp, kc, vc = make(ca, Hq, Hkv, W, I, Sc, P, seed=Sc + P)
    o, lse = ca.dcp_prefill(q, kp, vp, kc, vc, I, P)
    ro, rl = oracle.dcp_prefill(np32(q), clean(kp), clean(vp), clean(kc), clean(vc), I, P)
    assert_close(np32(o), ro, np32(lse), rl, what=f"dcp prefill Sc={Sc} P={P}")


@pytest.mark.parametrize("W,I", [(2, 16), (8, 16), (4, 32), (1, 16)])
def test_dcp_prefill_degrees(ca, W, I):
    q, kp, vp, kc, vc = make(ca, 8, 2, W, I, 384, 700, seed=W * 100 + I)
    o, lse = ca.dcp_prefill(q, kp, vp, kc, vc, I, 700)
    ro, rl = oracle.dcp_prefill(np32(q), clean(kp), clean(vp), clean(kc), clean(vc), I, 700)
    assert_close(np32(o), ro, np32(lse), rl, what=f"dcp prefill W={W} I={I}")


def test_dcp_prefill_partials_and_explicit_merge(ca):
    """Each rank's partial matches the oracle's partial; merging the partials
    with ca_lse_merge (weights exp(lse_R - lse)) gives the fused result."""
    Hq, Hkv, W, I, Sc, P = 4, 2, 4, 16, 384, 500
    q, kp, vp, kc, vc = make(ca, Hq, Hkv, W, I, Sc, P, seed=7)
    parts_o, parts_l = [], []
    for R in range(W):
        op, lp = ca.dcp_prefill_partial(q, kp, vp, kc, vc, I, P, R)
        ro, rl = oracle.dcp_prefill(np32(q), clean(kp), clean(vp), clean(kc), clean(vc), I, P, part_rank=R)
        assert_close(np32(op), ro, np32(lp), rl, what=f"partial rank {R}")
        parts_o.append(op)
        parts_l.append(lp)
    mo, ml = ca.lse_merge(torch.stack(parts_o), torch.stack(parts_l), out_dtype=torch.float32)
    fo, fl = ca.dcp_prefill(q, kp, vp, kc, vc, I, P)
    ro, rl = oracle.dcp_prefill(np32(q), clean(kp), clean(vp), clean(kc), clean(vc), I, P)
    assert_close(np32(mo), ro, np32(ml), rl, what="merged partials")
    assert_close(np32(fo), np32(mo).astype(np.float64), np32(fl), np32(ml).astype(np.float64), what="fused vs merged")


def test_dcp_prefill_long_context_sampled(ca):
    """A 8192-token chunk after 122880 cached tokens (131072 in all), Hq=32,
    Hkv=8, dcp=4, I=16: sampled query rows of three heads against the oracle."""
    from context_attention_gb300 import synth

    Hq, Hkv, W, I, Sc, P = 32, 8, 4, 16, 8192, 122880
    Lcap, Lc = P // W, Sc // W
    q, kp, vp, kc, vc = synth.dcp_prefill_inputs(Hq, Hkv, 128, W, Sc, Lcap, Lc, 8, device="cuda")
    o, lse = ca.dcp_prefill(q, kp, vp, kc, vc, I, P)
    torch.cuda.synchronize()
    rng = np.random.default_rng(9)
    for h in (0, 13, 31):
        hk = h // (Hq // Hkv)
        rows = np.unique(np.concatenate([[0, Sc - 1, 1023, 1024], rng.integers(0, Sc, 12)]))
        ro, rl = oracle.dcp_prefill(np32(q[h:h + 1]), np32(kp[:, hk:hk + 1]), np32(vp[:, hk:hk + 1]),
                                    np32(kc[:, hk:hk + 1]), np32(vc[:, hk:hk + 1]), I, P, rows=rows)
        idx = torch.as_tensor(rows, device="cuda")
        assert_close(np32(o[h].index_select(0, idx)), ro, np32(lse[h].index_select(0, idx)), rl,
                     what=f"long dcp prefill head {h}")
