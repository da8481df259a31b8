"""Seeded random shapes against the fp64 oracle: every draw is a small problem
-- ring attention (ragged shard lengths, GQA ratios, shard counts 1-8, both
layouts, both modes, causal or not, fp32 head dimensions 1-128), DCP and ring
decode (random shard counts, interleaves and sequence lengths, empty ones
included), DCP prefill and paged decode, the QKV prologue (random head
counts, widths and options) -- so
shape combinations no hand-written case names are still compared element by
element."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, bf16_bound, np32

pytestmark = pytest.mark.gpu

MODES = {"online_max": oracle.MODE_ONLINE_MAX, "const_max": oracle.MODE_CONST_MAX}
LAYOUTS = {"contiguous": oracle.LAYOUT_CONTIGUOUS, "striped": oracle.LAYOUT_STRIPED}


@pytest.fixture(scope="module")
def ca(cuda_device):
    import context_attention_gb300 as m

    m.build()
    yield m
    assert m.device_status() == 0, "a bounded device wait gave up"


def ring_draws(n, seed):
    rng = np.random.default_rng(seed)
    for i in range(n):
        bf16 = bool(rng.integers(0, 2))
        yield dict(i=i, dtype=torch.bfloat16 if bf16 else torch.float32,
                   D=128 if bf16 else int(rng.integers(1, 129)),
                   B=int(rng.integers(1, 3)), Hkv=int(rng.integers(1, 4)), G=int(rng.integers(1, 5)),
                   cp=int(rng.integers(1, 9)), Ls=int(rng.integers(1, 300)),
                   causal=bool(rng.integers(0, 2)), layout=["contiguous", "striped"][int(rng.integers(0, 2))],
                   mode=["online_max", "const_max"][int(rng.integers(0, 2))],
                   scale=float(rng.choice([0.0, 0.05, 0.2])), seed=int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("c", list(ring_draws(64, 2026)), ids=lambda c: f"draw{c['i']}")
def test_ring_random_shapes(ca, c):
    from context_attention_gb300 import synth

    Hq, S = c["Hkv"] * c["G"], c["cp"] * c["Ls"]
    q, k, v = synth.normal_qkv(c["B"], Hq, c["Hkv"], S, c["D"], c["seed"], dtype=c["dtype"], device="cuda")
    scale = c["scale"] or None
    o, lse = ca.ring_attn_fwd(q, k, v, c["cp"], mode=c["mode"], causal=c["causal"], layout=c["layout"],
                              softmax_scale=scale)
    ro, rl, _ = oracle.ring(np32(q), np32(k), np32(v), c["cp"], mode=MODES[c["mode"]], causal=c["causal"],
                            layout=LAYOUTS[c["layout"]], scale=scale)
    if c["dtype"] == torch.float32:
        assert_close(np32(o), ro, np32(lse), rl, dtype=c["dtype"], what=str(c))
        return
    bf16_bound(np32(o), ro, what=str(c))
    # lse and the mean error keep the fixed bounds
    g, r = np32(lse).astype(np.float64).reshape(-1), np.asarray(rl).reshape(-1)
    assert np.abs(g - r).max() <= 1e-3, str(c)
    assert np.abs(np32(o).astype(np.float64).reshape(ro.shape) - ro).mean() <= 2e-3, str(c)


def decode_draws(n, seed):
    rng = np.random.default_rng(seed)
    for i in range(n):
        Hkv, G = int(rng.integers(1, 4)), int(rng.integers(1, 9))
        yield dict(i=i, N=int(rng.integers(1, 4)), Hkv=Hkv, G=G, W=int(rng.integers(1, 5)),
                   I=int(rng.choice([16, 32, 64])), m=int(rng.integers(1, 40)), cp=int(rng.integers(1, 9)),
                   Ls=int(rng.integers(1, 500)), layout=["contiguous", "striped"][int(rng.integers(0, 2))],
                   seed=int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("c", list(decode_draws(32, 2027)), ids=lambda c: f"draw{c['i']}")
def test_dcp_decode_random_shapes(ca, c):
    from context_attention_gb300 import synth

    Lloc = c["I"] * c["m"]
    q, k, v = synth.decode_inputs(c["N"], c["Hkv"] * c["G"], c["Hkv"], 128, c["W"], Lloc, c["seed"], device="cuda")
    rng = np.random.default_rng(c["seed"])
    lens = [int(x) for x in rng.integers(0, c["W"] * Lloc + 1, size=c["N"])]
    o, lse = ca.dcp_decode(q, k, v, c["I"], seq_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    ro, rl = oracle.dcp_decode(np32(q), np32(k), np32(v), c["I"], seq_lens=lens)
    assert_close(np32(o), ro, np32(lse), rl, what=f"{c} lens={lens}")


@pytest.mark.parametrize("c", list(decode_draws(32, 2028)), ids=lambda c: f"draw{c['i']}")
def test_ring_decode_random_shapes(ca, c):
    g = torch.Generator(device="cuda")
    g.manual_seed(c["seed"])
    B, Hkv, S = c["N"], c["Hkv"], c["cp"] * c["Ls"]
    q = torch.randn(B, Hkv * c["G"], 128, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, 128, generator=g, device="cuda").to(torch.bfloat16)
    rng = np.random.default_rng(c["seed"])
    lens = [int(x) for x in rng.integers(0, S + 1, size=B)]
    o, lse = ca.ring_decode(q, k, v, c["cp"], layout=c["layout"],
                            seq_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    ro, rl = oracle.ring_decode(np32(q), np32(k), np32(v), c["cp"], LAYOUTS[c["layout"]], seq_lens=lens)
    assert_close(np32(o), ro, np32(lse), rl, what=f"{c} lens={lens}")


def prologue_draws(n, seed):
    rng = np.random.default_rng(seed)
    for i in range(n):
        D = int(rng.choice([64, 128]))
        Hkv = int(rng.integers(1, 9))
        G = int(rng.integers(1, 5))
        while Hkv * G * D > 8192:
            G -= 1
        cp = int(rng.integers(1, 9))
        yield dict(i=i, B=int(rng.integers(1, 3)), S=cp * int(rng.integers(1, 40)), Hq=Hkv * G, Hkv=Hkv, D=D, cp=cp,
                   layout=["contiguous", "striped"][int(rng.integers(0, 2))], rope=bool(rng.integers(0, 2)),
                   gains=bool(rng.integers(0, 2)), with_v=bool(rng.integers(0, 2)), seed=int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("c", list(prologue_draws(24, 2029)), ids=lambda c: f"draw{c['i']}")
def test_qkv_prologue_random_shapes(ca, c):
    from context_attention_gb300 import synth

    x_q, x_k, x_v, g_q, g_k, cos, sin = [t.cuda() for t in synth.qkv_activations(c["B"], c["S"], c["Hq"], c["Hkv"],
                                                                                 c["D"], c["seed"])]
    if not c["rope"]:
        cos = sin = None
    if not c["gains"]:
        g_q = g_k = None
    q, k, v, km = ca.qkv_prologue(x_q, x_k, c["Hq"], c["Hkv"], x_v=x_v if c["with_v"] else None, g_q=g_q, g_k=g_k,
                                  rope_cos=cos, rope_sin=sin, cp_size=c["cp"], layout=c["layout"])
    lay = LAYOUTS[c["layout"]]
    cs = None if cos is None else np32(cos)
    sn = None if sin is None else np32(sin)
    for got, x, H, g in ((q, x_q, c["Hq"], g_q), (k, x_k, c["Hkv"], g_k)):
        ref = oracle.qk_prologue(np32(x), H, g=None if g is None else np32(g), cos=cs, sin=sn, cp=c["cp"], layout=lay)
        err = np.abs(np32(got).astype(np.float64) - ref)
        # one bf16 rounding of the exact value (plus fp32 arithmetic)
        assert (err <= 2.0 ** -8 * np.abs(ref) + 1e-6).all(), f"{c}: worst {err.max():.3e}"
    if c["with_v"]:
        assert np.array_equal(np32(v).astype(np.float64), oracle.qk_prologue(np32(x_v), c["Hkv"], norm=False,
                                                                             cp=c["cp"], layout=lay)), str(c)
    _, rkm = oracle.const_max_bound(np32(k), np32(k))
    np.testing.assert_allclose(np32(km), rkm, rtol=2e-6, err_msg=str(c))


def prefill_draws(n, seed):
    rng = np.random.default_rng(seed)
    for i in range(n):
        yield dict(i=i, Hkv=int(rng.integers(1, 4)), G=int(rng.integers(1, 5)), W=int(rng.choice([1, 2, 4, 8])),
                   I=int(rng.choice([16, 32])), Sc=int(rng.integers(1, 700)), P=int(rng.integers(0, 3000)),
                   seed=int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("c", list(prefill_draws(16, 2030)), ids=lambda c: f"draw{c['i']}")
def test_dcp_prefill_random_shapes(ca, c):
    from test_gpu_dcp_prefill import clean, make

    q, kp, vp, kc, vc = make(ca, c["Hkv"] * c["G"], c["Hkv"], c["W"], c["I"], c["Sc"], c["P"], seed=c["seed"])
    o, lse = ca.dcp_prefill(q, kp, vp, kc, vc, c["I"], c["P"])
    ro, rl = oracle.dcp_prefill(np32(q), clean(kp), clean(vp), clean(kc), clean(vc), c["I"], c["P"])
    assert_close(np32(o), ro, np32(lse), rl, what=str(c))


def paged_draws(n, seed):
    rng = np.random.default_rng(seed)
    for i in range(n):
        bs = int(rng.choice([8, 16, 32, 64, 128]))
        yield dict(i=i, N=int(rng.integers(1, 4)), Hkv=int(rng.integers(1, 3)), G=int(rng.integers(1, 9)),
                   W=int(rng.integers(1, 5)), bs=bs, mb=int(rng.integers(1, 12)), seed=int(rng.integers(0, 1 << 30)))


@pytest.mark.parametrize("c", list(paged_draws(16, 2031)), ids=lambda c: f"draw{c['i']}")
def test_paged_decode_random_shapes(ca, c):
    from context_attention_gb300 import synth
    from test_gpu_paged_decode import page

    Lloc = c["bs"] * c["mb"]
    q, ks, vs = synth.decode_inputs(c["N"], c["Hkv"] * c["G"], c["Hkv"], 128, c["W"], Lloc, c["seed"], device="cuda")
    rng = np.random.default_rng(c["seed"])
    lens = [int(x) for x in rng.integers(0, c["W"] * Lloc + 1, size=c["N"])]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kc, vc, bt = page(ks, vs, c["bs"], seed=c["seed"] % 1000)
    o, lse = ca.dcp_decode_paged(q, kc, vc, bt, c["bs"], sl)
    o_c, l_c = ca.dcp_decode(q, ks, vs, c["bs"], seq_lens=sl)
    assert torch.equal(o, o_c) and torch.equal(lse, l_c), str(c)
    ro, rl = oracle.dcp_decode(np32(q), np32(ks), np32(vs), c["bs"], seq_lens=lens)
    assert_close(np32(o), ro, np32(lse), rl, what=f"{c} lens={lens}")
