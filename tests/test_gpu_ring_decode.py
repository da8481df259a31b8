"""GPU parity of Ring Pass-Q decode (one query token per sequence over the ring
layout's KV cache) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, np32

pytestmark = pytest.mark.gpu

LAYOUTS = {"contiguous": oracle.LAYOUT_CONTIGUOUS, "striped": oracle.LAYOUT_STRIPED}


@pytest.fixture(scope="module")
def ca(cuda_device):
    import context_attention_gb300 as m

    m.build()
    yield m
    assert m.device_status() == 0, "a bounded device wait gave up"


def inputs(B, Hq, Hkv, S, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q = torch.randn(B, Hq, 128, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, 128, generator=g, device="cuda").to(torch.bfloat16)
    return q, k, v


def run_case(ca, B, Hq, Hkv, S, cp, layout, seq_lens, seed, scale=None):
    q, k, v = inputs(B, Hq, Hkv, S, seed)
    sl = None if seq_lens is None else torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    o, lse = ca.ring_decode(q, k, v, cp, layout=layout, seq_lens=sl, softmax_scale=scale)
    ro, rl = oracle.ring_decode(np32(q), np32(k), np32(v), cp, LAYOUTS[layout], seq_lens=seq_lens, scale=scale)
    assert_close(np32(o), ro, np32(lse), rl, what=f"ring decode B={B} Hq={Hq} Hkv={Hkv} S={S} cp={cp} {layout}")


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_ring_decode_full_cache(ca, layout):
    run_case(ca, B=3, Hq=8, Hkv=2, S=2048, cp=4, layout=layout, seq_lens=None, seed=1)


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_ring_decode_variable_lengths(ca, layout):
    """Lengths that leave shards empty, partly filled, or end mid-stage: 1
    (only shard 0 holds a token), cp - 1, a shard boundary and one past it,
    ragged, full."""
    S, cp = 4096, 8
    lens = [1, cp - 1, S // cp, S // cp + 1, 1000, 3333, S]
    run_case(ca, B=len(lens), Hq=4, Hkv=1, S=S, cp=cp, layout=layout, seq_lens=lens, seed=2)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (4, 1), (32, 8), (16, 2)])
def test_ring_decode_gqa_groups(ca, Hq, Hkv):
    run_case(ca, B=2, Hq=Hq, Hkv=Hkv, S=1280, cp=2, layout="striped", seq_lens=[1280, 701], seed=3, scale=0.07)


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_ring_decode_multi_split_and_garbage_tail(ca, layout):
    """Shards span several 4096-slot splits, with a ragged shard length
    (S/cp not a multiple of the 128-slot stage); slots at global positions
    >= seq_len hold NaN and must not leak into the result."""
    B, Hq, Hkv, cp = 2, 8, 2, 3
    S = cp * 9000
    q, k, v = inputs(B, Hq, Hkv, S, 4)
    lens = [S - 100, 20001]
    Ls = S // cp
    rho = torch.arange(S, device="cuda")
    gpos = rho if layout == "contiguous" else (rho % Ls) * cp + rho // Ls
    for b in range(B):
        dead = gpos >= lens[b]
        k[b, :, dead] = float("nan")
        v[b, :, dead] = float("nan")
    o, lse = ca.ring_decode(q, k, v, cp, layout=layout, seq_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    ro, rl = oracle.ring_decode(np32(q), np32(torch.nan_to_num(k)), np32(torch.nan_to_num(v)), cp, LAYOUTS[layout],
                                seq_lens=lens)
    assert_close(np32(o), ro, np32(lse), rl, what=f"ring decode nan tail {layout}")


def test_ring_decode_zero_length_sequence(ca):
    """seq_len = 0: every shard's partial is empty: o = 0, lse = -inf."""
    q, k, v = inputs(2, 4, 1, 512, 5)
    sl = torch.tensor([0, 300], dtype=torch.int32, device="cuda")
    o, lse = ca.ring_decode(q, k, v, 4, layout="striped", seq_lens=sl)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ro, rl = oracle.ring_decode(np32(q[1:]), np32(k[1:]), np32(v[1:]), 4, oracle.LAYOUT_STRIPED, seq_lens=[300])
    assert_close(np32(o[1:]), ro, np32(lse[1:]), rl, what="ring decode second seq")


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_ring_decode_of_a_sharded_global_cache(ca, layout):
    """Store a global-order cache in the ring layout with the library's own
    permutation kernel, decode, and compare with plain attention of the query
    over the global prefix (the oracle's full attention)."""
    B, Hq, Hkv, S, cp = 2, 4, 2, 2048, 8
    q, kg, vg = inputs(B, Hq, Hkv, S, 6)
    k, v = ca.layout_to_shards(kg, cp, layout), ca.layout_to_shards(vg, cp, layout)
    lens = [S, 777]
    o, lse = ca.ring_decode(q, k, v, cp, layout=layout, seq_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    for b in range(B):
        Lb = lens[b]
        qf = np.zeros((1, Hq, Lb, 128), np.float32)
        qf[0, :, 0] = np32(q[b])
        ro, rl = oracle.attention(qf, np32(kg[b:b + 1, :, :Lb]), np32(vg[b:b + 1, :, :Lb]),
                                  rows=[h * Lb for h in range(Hq)])
        assert_close(np32(o[b]), ro, np32(lse[b]), rl, what=f"ring decode vs global b={b} {layout}")


def test_ring_decode_matches_last_row_of_causal_prefill(ca):
    """The decode of the last prefill token's query against the cache it
    completes equals that token's row of the causal ring prefill (two GPU
    paths, both against the oracle)."""
    B, H, S, cp = 1, 4, 2048, 4
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    q = torch.randn(B, H, S, 128, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, H, S, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, H, S, 128, generator=g, device="cuda").to(torch.bfloat16)
    # striped: global token S-1 is local token S/cp - 1 of shard cp - 1, the last stored row
    o_pre, lse_pre = ca.ring_attn_fwd(q, k, v, cp, causal=True, layout="striped")
    o_dec, lse_dec = ca.ring_decode(q[:, :, -1].contiguous(), k, v, cp, layout="striped")
    ro, rl = oracle.ring_decode(np32(q[:, :, -1]), np32(k), np32(v), cp, oracle.LAYOUT_STRIPED)
    assert_close(np32(o_dec), ro, np32(lse_dec), rl, what="decode of the last token")
    assert_close(np32(o_pre[:, :, -1]), ro, np32(lse_pre[:, :, -1]), rl, what="prefill's last row")


def test_ring_decode_long_context_sampled(ca):
    """Eight sequences over a 131072-token striped cache (4.3 GB of K+V),
    ragged lengths; two sequences checked against the oracle in full."""
    B, Hq, Hkv, S, cp = 8, 32, 8, 131072, 8
    q, k, v = inputs(B, Hq, Hkv, S, 8)
    rng = np.random.default_rng(8)
    lens = [int(x) for x in rng.integers(1, S + 1, size=B)]
    lens[0] = S
    o, lse = ca.ring_decode(q, k, v, cp, layout="striped",
                            seq_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    for b in (0, 5):
        ro, rl = oracle.ring_decode(np32(q[b:b + 1]), np32(k[b:b + 1]), np32(v[b:b + 1]), cp,
                                    oracle.LAYOUT_STRIPED, seq_lens=[lens[b]])
        assert_close(np32(o[b:b + 1]), ro, np32(lse[b:b + 1]), rl, what=f"long ring decode b={b} len={lens[b]}")
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
