"""GPU parity of DCP decode against the fp64 oracle, through the C ABI."""
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


def run_case(ca, N, Hq, Hkv, W, I, Lloc, seq_lens, seed, scale=None):
    from context_attention_gb300 import synth

    q, k, v = synth.decode_inputs(N, Hq, Hkv, 128, W, Lloc, seed, device="cuda")
    sl = None if seq_lens is None else torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    o, lse = ca.dcp_decode(q, k, v, I, seq_lens=sl, softmax_scale=scale)
    ro, rl = oracle.dcp_decode(np32(q), np32(k), np32(v), I, seq_lens=seq_lens, scale=scale)
    assert_close(np32(o), ro, np32(lse), rl, what=f"decode N={N} Hq={Hq} Hkv={Hkv} W={W} Lloc={Lloc}")


def test_decode_full_lengths(ca):
    run_case(ca, N=3, Hq=8, Hkv=2, W=4, I=16, Lloc=512, seq_lens=None, seed=1)


def test_decode_variable_lengths(ca):
    """Lengths on and off block and virtual-block boundaries: 1 token (only
    rank 0 holds anything), 17, 63, 64, 65, 1000, a full cache; the active
    token is counted exactly once (owner only)."""
    W, I, Lloc = 4, 16, 1024
    lens = [1, 17, 63, 64, 65, 1000, W * Lloc, 2049]
    run_case(ca, N=len(lens), Hq=4, Hkv=1, W=W, I=I, Lloc=Lloc, seq_lens=lens, seed=2)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (4, 1), (32, 8), (16, 2)])
def test_decode_gqa_groups(ca, Hq, Hkv):
    run_case(ca, N=2, Hq=Hq, Hkv=Hkv, W=2, I=16, Lloc=640, seq_lens=[1280, 700], seed=3)


def test_decode_multi_split_and_garbage_tail(ca):
    """Lloc spans several 4096-token splits; slots past each rank's valid
    count hold NaN and must not leak into the result."""
    from context_attention_gb300 import synth

    N, Hq, Hkv, W, I, Lloc = 2, 8, 2, 4, 16, 9000 - 9000 % 16
    q, k, v = synth.decode_inputs(N, Hq, Hkv, 128, W, Lloc, 4, device="cuda")
    lens = [W * Lloc - 100, 20000]
    for r in range(W):
        for n in range(N):
            lf = ca.dcp_local_filled(lens[n], W, I, I, r)
            k[r, n, :, lf:] = float("nan")
            v[r, n, :, lf:] = float("nan")
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = ca.dcp_decode(q, k, v, I, seq_lens=sl)
    kk, vv = torch.nan_to_num(k), torch.nan_to_num(v)
    ro, rl = oracle.dcp_decode(np32(q), np32(kk), np32(vv), I, seq_lens=lens)
    assert_close(np32(o), ro, np32(lse), rl, what="decode nan tail")


@pytest.mark.parametrize("N", [7, 8])
def test_decode_contiguous_ranges_and_dealt_splits(ca, N):
    """224 (shard, sequence, KV head) pairs are cut into one contiguous range
    of stages per CTA, 256 are dealt as 4096-token splits: both must give the
    oracle's decode, with lengths that leave shards empty, end mid-stage and
    fill the cache, and NaN in every slot past a shard's valid count."""
    from context_attention_gb300 import synth

    Hq, Hkv, W, I, Lloc = 16, 8, 4, 16, 2560 + 1280
    q, k, v = synth.decode_inputs(N, Hq, Hkv, 128, W, Lloc, 60 + N, device="cuda")
    lens = [0, 1, 129, 5000, W * Lloc, 12345, 7, 9999][:N]
    for r in range(W):
        for n in range(N):
            lf = ca.dcp_local_filled(lens[n], W, I, I, r)
            k[r, n, :, lf:] = float("nan")
            v[r, n, :, lf:] = float("nan")
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o, lse = ca.dcp_decode(q, k, v, I, seq_lens=sl)
    ro, rl = oracle.dcp_decode(np32(q), np32(torch.nan_to_num(k)), np32(torch.nan_to_num(v)), I, seq_lens=lens)
    assert_close(np32(o), ro, np32(lse), rl, what=f"decode, {W * N * Hkv} pairs")


def test_decode_one_sequence_131k(ca):
    """One sequence over four 32768-slot shards (the small-batch decode): the
    32 pairs' 1024 stages split into one range per CTA, so a pair's stages
    meet several CTAs and its partial slots fill from several of them; a
    second length ends mid-stage with NaN past it."""
    from context_attention_gb300 import synth

    N, Hq, Hkv, W, I, Lloc = 1, 32, 8, 4, 16, 32768
    q, k, v = synth.decode_inputs(N, Hq, Hkv, 128, W, Lloc, 70, device="cuda")
    o, lse = ca.dcp_decode(q, k, v, I)
    ro, rl = oracle.dcp_decode(np32(q), np32(k), np32(v), I)
    assert_close(np32(o), ro, np32(lse), rl, what="decode, one sequence of 131072 tokens")
    L = 100001
    for r in range(W):
        lf = ca.dcp_local_filled(L, W, I, I, r)
        k[r, 0, :, lf:] = float("nan")
        v[r, 0, :, lf:] = float("nan")
    sl = torch.tensor([L], dtype=torch.int32, device="cuda")
    o, lse = ca.dcp_decode(q, k, v, I, seq_lens=sl)
    ro, rl = oracle.dcp_decode(np32(q), np32(torch.nan_to_num(k)), np32(torch.nan_to_num(v)), I, seq_lens=[L])
    assert_close(np32(o), ro, np32(lse), rl, what="decode, one sequence of 100001 tokens")


@pytest.mark.parametrize("N", [1, 8])
def test_back_to_back_decodes_share_a_workspace(ca, N):
    """Decodes queued back to back on one stream with one workspace: each is
    launched as a programmatic dependent and sets up while the previous
    call's merge still reads that workspace, so it must touch no global
    memory before its grid dependency resolves.  Every output must equal the
    same call made alone (one sequence: contiguous CTA ranges and the
    one-block-per-row merge; eight: dealt splits)."""
    from context_attention_gb300 import synth

    Hq, Hkv, W, I, Lloc = 32, 8, 4, 16, 4096
    q, k, v = synth.decode_inputs(N, Hq, Hkv, 128, W, Lloc, 80 + N, device="cuda")
    qs = [q] + [torch.randn_like(q.float()).to(q.dtype) for _ in range(3)]
    ws = torch.empty(ca.dcp_decode_workspace_size(N, Hq, Hkv, Lloc, 128, W, I), dtype=torch.uint8, device="cuda")
    alone = []
    for qq in qs:
        o, lse = ca.dcp_decode(qq, k, v, I, workspace=ws)
        torch.cuda.synchronize()
        alone.append((o.clone(), lse.clone()))
    outs = [(torch.empty_like(q), torch.empty(N, Hq, device="cuda")) for _ in qs]
    for _ in range(3):
        for qq, (o, lse) in zip(qs, outs):
            ca.dcp_decode(qq, k, v, I, out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    for (o, lse), (oa, la) in zip(outs, alone):
        assert torch.equal(o, oa) and torch.equal(lse, la)


def test_decode_single_pair_many_partials(ca):
    """One shard, one sequence, one KV head (eight query heads): the single
    pair's 1024 stages are cut over every CTA, so each row merges one partial
    per CTA (about 150, beyond the merge's groups of 32); lengths full and
    ending mid-stage, NaN past the valid slots."""
    from context_attention_gb300 import synth

    N, Hq, Hkv, W, I, Lloc = 1, 8, 1, 1, 16, 131072
    q, k, v = synth.decode_inputs(N, Hq, Hkv, 128, W, Lloc, 90, device="cuda")
    for L in (Lloc, 100001):
        kk, vv = k.clone(), v.clone()
        kk[0, 0, :, L:] = float("nan")
        vv[0, 0, :, L:] = float("nan")
        sl = torch.tensor([L], dtype=torch.int32, device="cuda")
        o, lse = ca.dcp_decode(q, kk, vv, I, seq_lens=sl)
        ro, rl = oracle.dcp_decode(np32(q), np32(torch.nan_to_num(kk)), np32(torch.nan_to_num(vv)), I,
                                   seq_lens=[L])
        assert_close(np32(o), ro, np32(lse), rl, what=f"decode, one pair, L={L}")


def test_decode_zero_length_sequence(ca):
    """seq_len = 0: every partial is empty: o = 0, lse = -inf."""
    from context_attention_gb300 import synth

    q, k, v = synth.decode_inputs(2, 4, 1, 128, 2, 256, 5, device="cuda")
    sl = torch.tensor([0, 300], dtype=torch.int32, device="cuda")
    o, lse = ca.dcp_decode(q, k, v, 16, seq_lens=sl)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ro, rl = oracle.dcp_decode(np32(q[1:]), np32(k[:, 1:]), np32(v[:, 1:]), 16, seq_lens=[300])
    assert_close(np32(o[1:]), ro, np32(lse[1:]), rl, what="decode second seq")


def test_decode_matches_global_attention(ca):
    """Shard a global KV cache with the library's interleave kernel, decode,
    and compare with plain attention of the query over the global prefix
    (the oracle's full attention)."""
    from context_attention_gb300 import synth

    N, Hq, Hkv, W, I, L = 2, 4, 2, 4, 16, 1024
    g = torch.Generator(device="cuda")
    g.manual_seed(6)
    q = torch.randn(N, Hq, 128, generator=g, device="cuda").to(torch.bfloat16)
    kg = torch.randn(N, Hkv, L, 128, generator=g, device="cuda").to(torch.bfloat16)
    vg = torch.randn(N, Hkv, L, 128, generator=g, device="cuda").to(torch.bfloat16)
    ks, vs = ca.dcp_shard_kv(kg, W, I), ca.dcp_shard_kv(vg, W, I)
    lens = [L, 555]
    o, lse = ca.dcp_decode(q, ks, vs, I, seq_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    for n in range(N):
        Ln = lens[n]
        qf = np.zeros((1, Hq, Ln, 128), np.float32)
        qf[0, :, 0] = np32(q[n])
        ro, rl = oracle.attention(qf, np32(kg[n:n + 1, :, :Ln]), np32(vg[n:n + 1, :, :Ln]),
                                  rows=[h * Ln for h in range(Hq)])
        assert_close(np32(o[n]), ro, np32(lse[n]), rl, what=f"decode vs global n={n}")
    del synth


@pytest.mark.parametrize("scale", [None, 0.5])
def test_decode_constant_v_gives_v_exactly(ca, scale):
    """When every cached token of a KV head holds the same value row, each
    query head's output is that row.  Every split divides its O by the sum
    of the bf16 weights its MMA used, and the LSE merge's weights sum to one
    up to fp32 rounding, so the bf16 output rounds back to V exactly; scale
    0.5 lets a few keys dominate each head, and one sequence holds a single
    token.  Values up to 16 in size."""
    from context_attention_gb300 import synth

    N, Hq, Hkv, W, I, Lloc = 3, 16, 2, 4, 16, 1024
    q, k, _ = synth.decode_inputs(N, Hq, Hkv, 128, W, Lloc, 41, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(42)
    row = ((torch.rand(N, Hkv, 128, generator=g, device="cuda") * 2 - 1) * 16).to(torch.bfloat16)
    v = row[None, :, :, None, :].expand(W, N, Hkv, Lloc, 128).contiguous()
    sl = torch.tensor([W * Lloc, 1, 777], dtype=torch.int32, device="cuda")
    o, lse = ca.dcp_decode(q, k, v, I, seq_lens=sl, softmax_scale=scale)
    want = row.repeat_interleave(Hq // Hkv, dim=1)
    bad = (o != want).sum().item()
    assert bad == 0, f"{bad} elements differ from V; worst {(o.float() - want.float()).abs().max().item():.3e}"
