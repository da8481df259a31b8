"""GPU parity of the QKV prologue of const-max attention (whole-hidden RMS
norm, gains, rotary turn, head split into the shard layout, per-head key
maximum) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from helpers import np32

pytestmark = pytest.mark.gpu

LAYOUTS = {"contiguous": oracle.LAYOUT_CONTIGUOUS, "striped": oracle.LAYOUT_STRIPED}
REL = 2.0 ** -8  # bf16 rounding (2^-9 relative) with room for fp32 arithmetic


@pytest.fixture(scope="module")
def ca(cuda_device):
    import context_attention_gb300 as m

    m.build()
    yield m
    assert m.device_status() == 0, "a bounded device wait gave up"


def inputs(B, S, Hq, Hkv, D, seed):
    from context_attention_gb300 import synth

    return [t.cuda() for t in synth.qkv_activations(B, S, Hq, Hkv, D, seed)]


def check_tensor(gpu, ref, what):
    g = np32(gpu).astype(np.float64)
    assert np.isfinite(g).all(), what
    err = np.abs(g - ref)
    bound = REL * np.abs(ref) + 1e-6
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} values off, worst {err[bad].max():.3e}"


def run_case(ca, B, S, Hq, Hkv, D, cp, layout, seed, rope=True, gains=True, with_v=True, eps=1e-6):
    """gains: True (both), False (neither), "q" or "k" (that tensor's only)."""
    x_q, x_k, x_v, g_q, g_k, cos, sin = inputs(B, S, Hq, Hkv, D, seed)
    if not rope:
        cos = sin = None
    if gains is False or gains == "k":
        g_q = None
    if gains is False or gains == "q":
        g_k = None
    q, k, v, km = ca.qkv_prologue(x_q, x_k, Hq, Hkv, x_v=x_v if with_v else None, g_q=g_q, g_k=g_k, eps=eps,
                                  rope_cos=cos, rope_sin=sin, cp_size=cp, layout=layout)
    lay = LAYOUTS[layout]
    c = None if cos is None else np32(cos)
    s = None if sin is None else np32(sin)
    rq = oracle.qk_prologue(np32(x_q), Hq, g=None if g_q is None else np32(g_q), eps=eps, cos=c, sin=s, cp=cp,
                            layout=lay)
    rk = oracle.qk_prologue(np32(x_k), Hkv, g=None if g_k is None else np32(g_k), eps=eps, cos=c, sin=s, cp=cp,
                            layout=lay)
    check_tensor(q, rq, "q")
    check_tensor(k, rk, "k")
    if with_v:
        rv = oracle.qk_prologue(np32(x_v), Hkv, norm=False, cp=cp, layout=lay)
        assert np.array_equal(np32(v).astype(np.float64), rv), "v must be a bit-exact head split"
    else:
        assert v is None
    # kmax2 bounds the stored (rounded) keys: the oracle's key maximum of the
    # very k the kernel wrote
    _, rkm = oracle.const_max_bound(np32(k), np32(k))
    np.testing.assert_allclose(np32(km), rkm, rtol=2e-6)
    return q, k, v, km


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_prologue_dit_heads(ca, layout):
    """The DiT's 40 heads of 128 (5120-wide hidden, 20 chunks per lane),
    self-attention (Hq = Hkv), cp = 8."""
    run_case(ca, 1, 256, 40, 40, 128, 8, layout, seed=21)


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_prologue_gqa(ca, layout):
    """GQA 32:8 with different q and k widths in one launch, B = 2, cp = 4."""
    run_case(ca, 2, 128, 32, 8, 128, 4, layout, seed=22)


def test_prologue_d64_ragged_lanes_no_rope_no_gain_no_v(ca):
    """D = 64, 6 and 3 heads (rows of 48 and 24 chunks: partly filled lanes),
    no rotary tables, no gains, no value tensor, eps = 0."""
    run_case(ca, 2, 96, 6, 3, 64, 3, "striped", seed=23, rope=False, gains=False, with_v=False, eps=0.0)


@pytest.mark.parametrize("which", ["q", "k"])
def test_prologue_one_tensor_with_gains(ca, which):
    """Only q's or only k's gains given: the block stages just those, and the
    other tensor is normalised with gain 1 (GQA widths, so the two gain
    vectors differ in length)."""
    run_case(ca, 1, 64, 16, 4, 128, 2, "contiguous", seed=25, gains=which)


def test_prologue_widest_hidden(ca):
    """H*D = 8192 (64 heads of 128: 32 chunks per lane), one token per shard."""
    run_case(ca, 1, 16, 64, 16, 128, 16, "contiguous", seed=24)


def test_prologue_feeds_the_ring(ca):
    """kmax2 from the prologue drives the const-max ring exactly like the
    key pass over the same k, and the ring matches the oracle on the
    prologue's outputs."""
    from helpers import assert_close

    q, k, v, km = run_case(ca, 1, 1024, 8, 2, 128, 4, "contiguous", seed=25)
    np.testing.assert_allclose(np32(km), np32(ca.key_max2(k)), rtol=1e-6)
    o1, l1 = ca.ring_attn_fwd_kmax(q, k, v, km, 4)
    ro, rl, _ = oracle.ring(np32(q), np32(k), np32(v), 4, mode=oracle.MODE_CONST_MAX)
    assert_close(np32(o1), ro, np32(l1), rl, what="prologue -> ring")
