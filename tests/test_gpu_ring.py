"""GPU parity of ring attention (fused ring, one ring step, LSE merge, bound)
against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import time

from helpers import assert_close, np32, parity_report

pytestmark = pytest.mark.gpu

MODES = {"online_max": oracle.MODE_ONLINE_MAX, "const_max": oracle.MODE_CONST_MAX}
LAYOUTS = {"contiguous": oracle.LAYOUT_CONTIGUOUS, "striped": oracle.LAYOUT_STRIPED}


@pytest.fixture(scope="module")
def ca(cuda_device):
    import context_attention_gb300 as m

    m.build()
    yield m
    assert m.device_status() == 0, "a bounded device wait gave up"


def gen(B, Hq, Hkv, S, D, seed, dtype):
    from context_attention_gb300 import synth

    return synth.normal_qkv(B, Hq, Hkv, S, D, seed, dtype=dtype, device="cuda")


def oracle_ring(q, k, v, cp, mode, causal, layout, scale=None):
    o, lse, _ = oracle.ring(np32(q), np32(k), np32(v), cp, mode=MODES[mode], causal=causal,
                            layout=LAYOUTS[layout], scale=scale)
    return o, lse


# --------------------------------------------------------------- fp32 (SIMT)


@pytest.mark.parametrize("mode", ["online_max", "const_max"])
def test_fp32_tiny_config(ca, mode):
    """fp32, B=1, H=2, S=256, D=64, cp=2: within 1e-4 of the oracle."""
    q, k, v = gen(1, 2, 2, 256, 64, 1, torch.float32)
    o, lse = ca.ring_attn_fwd(q, k, v, 2, mode=mode)
    t0 = time.perf_counter()
    ro, rl = oracle_ring(q, k, v, 2, mode, False, "contiguous")
    t = time.perf_counter() - t0
    assert_close(np32(o), ro, np32(lse), rl, dtype=torch.float32, what=f"fp32 {mode}")
    parity_report(f"tiny fp32 B1 H2 S256 D64 cp2 {mode} (every row)", np32(o), ro, np32(lse), rl, t)


@pytest.mark.parametrize("mode", ["online_max", "const_max"])
@pytest.mark.parametrize("causal,layout", [(False, "contiguous"), (True, "contiguous"), (True, "striped")])
def test_fp32_gqa_ragged_causal(ca, mode, causal, layout):
    # Ls = 70 (not a multiple of the 16-row block or the 32-key tile), GQA 4:2, D = 40
    q, k, v = gen(2, 4, 2, 210, 40, 2, torch.float32)
    o, lse = ca.ring_attn_fwd(q, k, v, 3, mode=mode, causal=causal, layout=layout, softmax_scale=0.3)
    ro, rl = oracle_ring(q, k, v, 3, mode, causal, layout, scale=0.3)
    assert_close(np32(o), ro, np32(lse), rl, dtype=torch.float32, what=f"fp32 {mode} {layout}")


@pytest.mark.parametrize("mode", ["online_max", "const_max"])
@pytest.mark.parametrize("D", [1, 17, 100])
def test_fp32_odd_head_dims(ca, mode, D):
    """fp32 with head dimensions whose rows are not whole 16-byte chunks (the
    key pass's scalar path), causal striped, GQA 4:2."""
    q, k, v = gen(1, 4, 2, 192, D, 3 + D, torch.float32)
    o, lse = ca.ring_attn_fwd(q, k, v, 2, mode=mode, causal=True, layout="striped")
    ro, rl = oracle_ring(q, k, v, 2, mode, True, "striped")
    assert_close(np32(o), ro, np32(lse), rl, dtype=torch.float32, what=f"fp32 D={D} {mode}")


# --------------------------------------------------------------- bf16 (tcgen05)


@pytest.mark.parametrize("mode", ["online_max", "const_max"])
@pytest.mark.parametrize("causal,layout", [(False, "contiguous"), (True, "contiguous"), (True, "striped")])
@pytest.mark.parametrize("wide", [False, True])
def test_bf16_constant_v_gives_v_exactly(ca, mode, causal, layout, wide):
    """Invariant (d) on the GPU: when every key of a head carries the same
    value row, the output is that row, whatever the weights.  The weights
    the PV product uses are bf16; on a tile that needs a mask (a causal
    diagonal, a shard's ragged end) O is divided by the sum of those same
    rounded weights, so o = V up to fp32 accumulation, which the bf16 output
    rounds back to V itself.  With 96-key shards every tile is ragged, so
    every row is normalised that way.  Causal rows near a shard's start see
    a handful of keys, and a wide score spread (scale 0.5; 0.25 in const
    max, whose bound must stay within ~85 nats of a row's lone key) lets one
    key dominate: the cases in which dividing by the unrounded weights' sum
    would be off by up to 2^-8 |V|.  Values up to 16 in size."""
    B, Hq, Hkv, S, D, cp = 1, 4, 2, 384, 128, 4
    scale = {"online_max": 0.5, "const_max": 0.25}[mode] if wide else None
    q, k, _ = gen(B, Hq, Hkv, S, D, 32, torch.bfloat16)
    g = torch.Generator(device="cuda")
    g.manual_seed(33)
    row = ((torch.rand(B, Hkv, 1, D, generator=g, device="cuda") * 2 - 1) * 16).to(torch.bfloat16)
    v = row.expand(B, Hkv, S, D).contiguous()
    o, lse = ca.ring_attn_fwd(q, k, v, cp, mode=mode, causal=causal, layout=layout, softmax_scale=scale)
    want = row.repeat_interleave(Hq // Hkv, dim=1).expand(B, Hq, S, D)
    bad = (o != want).sum().item()
    assert bad == 0, f"{bad} elements differ from V; worst {(o.float() - want.float()).abs().max().item():.3e}"
    ro, rl = oracle_ring(q, k, v, cp, mode, causal, layout, scale=scale)
    assert np.abs(np32(lse).astype(np.float64).reshape(-1) - np.asarray(rl).reshape(-1)).max() <= 1e-3


@pytest.mark.parametrize("mode", ["online_max", "const_max"])
@pytest.mark.parametrize("causal,layout", [(False, "contiguous"), (True, "contiguous"), (True, "striped")])
def test_bf16_small(ca, mode, causal, layout):
    """bf16, D=128, B=1, H=2, S=1024, cp=4 (Ls=256: two query tiles per unit)."""
    q, k, v = gen(1, 2, 2, 1024, 128, 3, torch.bfloat16)
    o, lse = ca.ring_attn_fwd(q, k, v, 4, mode=mode, causal=causal, layout=layout)
    ro, rl = oracle_ring(q, k, v, 4, mode, causal, layout)
    assert_close(np32(o), ro, np32(lse), rl, what=f"bf16 {mode} causal={causal} {layout}")


@pytest.mark.parametrize("mode", ["online_max", "const_max"])
@pytest.mark.parametrize("causal,layout", [(False, "contiguous"), (True, "contiguous"), (True, "striped")])
@pytest.mark.parametrize("G", [2, 3, 4])
def test_bf16_gqa_ragged(ca, mode, causal, layout, G):
    """GQA 2G:2 (kv head h//G), Ls = 300 (ragged: 3 key tiles, last one
    partial), cp = 3, B = 2.  An even G pairs the same 128 rows of heads h
    and h+1 in one unit (3 units per shard, the last mostly empty); G = 3
    keeps two consecutive row blocks of one head (the second query tile of
    the last unit mostly empty)."""
    q, k, v = gen(2, 2 * G, 2, 900, 128, 4, torch.bfloat16)
    o, lse = ca.ring_attn_fwd(q, k, v, 3, mode=mode, causal=causal, layout=layout)
    ro, rl = oracle_ring(q, k, v, 3, mode, causal, layout)
    assert_close(np32(o), ro, np32(lse), rl, what=f"bf16 gqa G={G} {mode} causal={causal} {layout}")


@pytest.mark.parametrize("S,cp", [(128, 1), (8, 8), (136, 8), (1, 1)])
def test_bf16_degenerate_shapes(ca, S, cp):
    """cp = 1 (plain attention), Ls = 1 (one token per shard), Ls = 17, S = 1."""
    q, k, v = gen(1, 2, 1, S, 128, 5, torch.bfloat16)
    for mode in ("online_max", "const_max"):
        for causal, layout in ((False, "contiguous"), (True, "striped"), (True, "contiguous")):
            o, lse = ca.ring_attn_fwd(q, k, v, cp, mode=mode, causal=causal, layout=layout)
            ro, rl = oracle_ring(q, k, v, cp, mode, causal, layout)
            assert_close(np32(o), ro, np32(lse), rl, what=f"S={S} cp={cp} {mode} {layout}")


def test_bf16_dit_const_max(ca):
    """Cross-head RMS-normalised q/k (the DiT recipe), H=8, S=2048, cp=8,
    const max and online max against the oracle."""
    from context_attention_gb300 import synth

    q, k, v = synth.dit_qk(1, 8, 2048, 128, seed=6, device="cuda")
    for mode in ("const_max", "online_max"):
        o, lse = ca.ring_attn_fwd(q, k, v, 8, mode=mode)
        ro, rl = oracle_ring(q, k, v, 8, mode, False, "contiguous")
        assert_close(np32(o), ro, np32(lse), rl, what=f"dit {mode}")


def test_bf16_error_distribution_vs_oracle_rounding(ca):
    """The GPU's error against exact attention is of the same order as the
    error of exact attention computed from bf16-rounded outputs (the const-max
    page's validation advice: compare error distributions)."""
    q, k, v = gen(1, 2, 2, 1024, 128, 7, torch.bfloat16)
    o, _ = ca.ring_attn_fwd(q, k, v, 4, mode="const_max")
    ro, _ = oracle_ring(q, k, v, 4, "const_max", False, "contiguous")
    gpu_err = np.abs(np32(o).reshape(ro.shape) - ro)
    round_err = np.abs(torch.tensor(ro).to(torch.bfloat16).double().numpy() - ro)
    assert gpu_err.mean() <= 4 * round_err.mean() + 1e-5


# --------------------------------------------------------------- steps + merge


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("causal,layout", [(False, "contiguous"), (True, "contiguous"), (True, "striped")])
def test_partial_steps_merge_to_ring(ca, dtype, causal, layout):
    """Every ring step through ca_attn_partial_step, merged with ca_lse_merge
    (online: LSE weights; const max: pure addition with the bound), equals the
    oracle's ring; each step's partial equals the oracle's shard partial."""
    cp, Ls = 4, 160
    D = 128 if dtype == torch.bfloat16 else 64
    q, k, v = gen(1, 4, 2, cp * Ls, D, 8, dtype)
    tol_dtype = dtype
    for mode in ("online_max", "const_max"):
        c_full = None
        if mode == "const_max":
            c_full, _ = ca.const_max_bound(q, k)
        ro, rl = oracle_ring(q, k, v, cp, mode, causal, layout)
        ro = ro.reshape(1, 4, cp * Ls, D)
        rl = rl.reshape(1, 4, cp * Ls)
        for r in range(cp):
            qs = q[:, :, r * Ls:(r + 1) * Ls].contiguous()
            o_parts, l_parts = [], []
            for t in range(cp):
                s = ca.ring_kv_shard(r, t, cp)
                ks = k[:, :, s * Ls:(s + 1) * Ls].contiguous()
                vs = v[:, :, s * Ls:(s + 1) * Ls].contiguous()
                cs = None if c_full is None else c_full[:, :, r * Ls:(r + 1) * Ls].contiguous()
                op, lp = ca.attn_partial_step(qs, ks, vs, r, s, cp, mode=mode, causal=causal, layout=layout, c=cs)
                if mode == "online_max":
                    rows = np.array([(hh * cp * Ls + r * Ls + a) for hh in range(4) for a in range(Ls)])
                    so, sl = oracle.shard_partial(np32(q), np32(k), np32(v), s, cp, causal=causal,
                                                  layout=LAYOUTS[layout], rows=rows)
                    assert_close(np32(op), so, np32(lp), sl, dtype=tol_dtype, what=f"step r={r} s={s}")
                o_parts.append(op)
                l_parts.append(lp)
            cm = None if c_full is None else c_full[:, :, r * Ls:(r + 1) * Ls].contiguous()
            o, lse = ca.lse_merge(torch.stack(o_parts), torch.stack(l_parts), c=cm, out_dtype=torch.float32)
            assert_close(np32(o), ro[:, :, r * Ls:(r + 1) * Ls], np32(lse), rl[:, :, r * Ls:(r + 1) * Ls],
                         dtype=tol_dtype, what=f"merged {mode} r={r}")


def test_partial_step_fully_masked(ca):
    """Contiguous causal, queries of shard 0 against keys of shard 2: nothing
    is visible, so o = 0 and lse = -inf (both dtypes)."""
    for dtype, D in ((torch.bfloat16, 128), (torch.float32, 32)):
        q, k, v = gen(1, 2, 2, 128, D, 9, dtype)
        o, lse = ca.attn_partial_step(q, k, v, 0, 2, 4, causal=True, layout="contiguous")
        assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_lse_merge_kernel(ca):
    rng = np.random.default_rng(10)
    n, R, D = 5, 300, 128
    op = rng.standard_normal((n, R, D)).astype(np.float32)
    lp = (rng.standard_normal((n, R)) * 3).astype(np.float32)
    lp[1, ::7] = -np.inf
    lp[:, 5] = -np.inf  # an all-empty row
    ro, rl = oracle.lse_merge(op, lp)
    for out_dtype in (torch.float32, torch.bfloat16):
        o, lse = ca.lse_merge(torch.tensor(op, device="cuda"), torch.tensor(lp, device="cuda"), out_dtype=out_dtype)
        assert_close(np32(o), ro, np32(lse), rl, dtype=torch.float32 if out_dtype == torch.float32 else torch.bfloat16,
                     what=f"merge {out_dtype}")


@pytest.mark.parametrize("n,R,D", [(3, 44000, 128), (2, 44000, 192)])
def test_lse_merge_larger_than_l2(ca, n, R, D):
    """Partials of more than 64 MB take the merge kernel that requests the
    partial rows before the weights (the one HBM-bound callers get); it must
    give the oracle's merge, online (with empty partials and an all-empty
    row) and with a shared const-max bound: unnormalised sums o_i with
    lse_i = c + ln l_i merge to what the oracle gives for the normalised
    partials o_i / l_i."""
    assert n * R * D * 4 > (64 << 20)
    rng = np.random.default_rng(20 + D)
    op = rng.standard_normal((n, R, D)).astype(np.float32)
    lp = (rng.standard_normal((n, R)) * 3).astype(np.float32)
    lp[0, ::5] = -np.inf
    lp[:, 7] = -np.inf
    ro, rl = oracle.lse_merge(op, lp)
    for out_dtype in (torch.float32, torch.bfloat16):
        o, lse = ca.lse_merge(torch.tensor(op, device="cuda"), torch.tensor(lp, device="cuda"), out_dtype=out_dtype)
        assert_close(np32(o), ro, np32(lse), rl, dtype=torch.float32 if out_dtype == torch.float32 else torch.bfloat16,
                     what=f"large merge {out_dtype}")
    # const max: every row's bound c above its partials' lse, no empty rows
    lc = (rng.standard_normal((n, R)) * 3).astype(np.float32)
    c = (lc.max(axis=0) + 2.0).astype(np.float32)
    l_i = np.exp(lc.astype(np.float64) - c.astype(np.float64))
    unnorm = (op * l_i[:, :, None]).astype(np.float32)
    ro, rl = oracle.lse_merge(unnorm.astype(np.float64) / l_i[:, :, None], lc)
    o, lse = ca.lse_merge(torch.tensor(unnorm, device="cuda"), torch.tensor(lc, device="cuda"),
                          c=torch.tensor(c, device="cuda"), out_dtype=torch.float32)
    assert_close(np32(o), ro, np32(lse), rl, dtype=torch.float32, what="large const-max merge")


@pytest.mark.parametrize("n,R,D", [(5, 300, 128),     # one warp per row, partials in L2
                                   (24, 32, 128),     # one block per row (a decode's shape)
                                   (40, 1000, 192),   # one block per row, two lse groups, wide rows
                                   (20, 64, 512),
                                   (3, 44000, 128)])  # rows requested before the weights (> 64 MB)
def test_lse_merge_ignores_rows_of_zero_weight(ca, n, R, D):
    """A partial whose lse is -inf adds nothing, whatever its o row holds:
    rows of NaN there must give the oracle's merge of the same partials with
    those rows zero, online and with a const-max bound."""
    rng = np.random.default_rng(30 + n)
    op = rng.standard_normal((n, R, D)).astype(np.float32)
    lp = (rng.standard_normal((n, R)) * 3).astype(np.float32)
    lp[0, ::3] = -np.inf
    lp[n - 1, 1::4] = -np.inf
    lp[:, 2] = -np.inf  # an all-empty row
    dead = np.isneginf(lp)
    clean = np.where(dead[:, :, None], 0.0, op)
    dirty = np.where(dead[:, :, None], np.float32(np.nan), op).astype(np.float32)
    ro, rl = oracle.lse_merge(clean, lp)
    o, lse = ca.lse_merge(torch.tensor(dirty, device="cuda"), torch.tensor(lp, device="cuda"),
                          out_dtype=torch.float32)
    assert_close(np32(o), ro, np32(lse), rl, dtype=torch.float32, what=f"merge, NaN rows of weight 0, n={n} R={R}")
    # const max: unnormalised sums o_i l_i with lse_i = c + ln l_i; rows with
    # l_i = 0 (lse_i = -inf) hold NaN
    c = (np.where(dead, -np.inf, lp).max(axis=0) + 1.5).astype(np.float32)
    c[2] = 0.0
    l_i = np.exp(lp.astype(np.float64) - c.astype(np.float64))
    unnorm = np.where(dead[:, :, None], np.float32(np.nan), (op * l_i[:, :, None])).astype(np.float32)
    live = ~dead.all(axis=0)
    o, lse = ca.lse_merge(torch.tensor(unnorm, device="cuda"), torch.tensor(lp, device="cuda"),
                          c=torch.tensor(c, device="cuda"), out_dtype=torch.float32)
    assert_close(np32(o)[live], ro[live], np32(lse)[live], rl[live], dtype=torch.float32,
                 what=f"const-max merge, NaN rows of weight 0, n={n} R={R}")
    assert np.all(np32(o)[~live] == 0.0)  # no partial: the 1e-37 clamp leaves o = 0


def test_const_max_bound_kernel(ca):
    from context_attention_gb300 import synth

    for dtype, D in ((torch.bfloat16, 128), (torch.float32, 64), (torch.float32, 20)):
        q, k, _ = synth.normal_qkv(2, 4, 2, 700, D, 11, dtype=dtype, device="cuda")
        c, kmax2 = ca.const_max_bound(q, k, softmax_scale=0.2)
        rc, rk = oracle.const_max_bound(np32(q), np32(k), scale=0.2)
        np.testing.assert_allclose(np32(kmax2), rk, rtol=2e-6)
        np.testing.assert_allclose(np32(c), rc, rtol=2e-6)


def test_key_max2_kernel(ca):
    """kmax2 alone (vector paths with 32, 16 and 2 lanes a row, the scalar
    path for rows not a multiple of 16 bytes, one-row heads)."""
    from context_attention_gb300 import synth

    for dtype, D, S in ((torch.bfloat16, 128, 700), (torch.float32, 128, 333), (torch.bfloat16, 48, 257),
                        (torch.float32, 20, 700), (torch.bfloat16, 128, 1), (torch.float32, 17, 300),
                        (torch.float32, 1, 50)):
        _, k, _ = synth.normal_qkv(2, 2, 3, S, D, 12, dtype=dtype, device="cuda")
        km = ca.key_max2(k)
        _, rk = oracle.const_max_bound(np32(k), np32(k))
        np.testing.assert_allclose(np32(km), rk, rtol=2e-6, err_msg=f"{dtype} D={D} S={S}")


def test_key_max2_of_key_blocks_combines_by_max(ca):
    """The per-process key maxima combine by an elementwise max (the
    all-reduce of the const-max page's "Global key max"): bit-exact."""
    from context_attention_gb300 import synth

    _, k, _ = synth.normal_qkv(1, 4, 4, 4096, 128, 13, dtype=torch.bfloat16, device="cuda")
    whole = ca.key_max2(k)
    parts = [ca.key_max2(k[:, :, i * 1024:(i + 1) * 1024].contiguous()) for i in range(4)]
    assert torch.equal(torch.stack(parts).amax(0), whole)


def aligned_qk(B, Hq, Hkv, S, D, seed, alpha_max, beta, dtype):
    """Keys and queries near one direction u per kv head, so the bound is
    tight and large: s_ij ~ scale * alpha_i * beta, alpha_i log-uniform in
    [1, alpha_max].  A bound off by tens of nats overflows or underflows."""
    g = torch.Generator().manual_seed(seed)
    G = Hq // Hkv
    u = torch.randn(B, Hkv, 1, D, generator=g)
    u = u / u.norm(dim=-1, keepdim=True)
    k = beta * (u + 0.03 * torch.randn(B, Hkv, S, D, generator=g))
    alpha = torch.exp(torch.rand(B, Hq, S, 1, generator=g) * np.log(alpha_max))
    q = alpha * (u.repeat_interleave(G, dim=1) + 0.03 * torch.randn(B, Hq, S, D, generator=g))
    v = torch.randn(B, Hkv, S, D, generator=g)
    return (t.to(dtype).cuda() for t in (q, k, v))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("causal,layout", [(False, "contiguous"), (True, "contiguous"), (True, "striped")])
def test_const_max_in_kernel_bound_large_scores(ca, dtype, causal, layout):
    """Scores up to ~170 nats with a tight bound: only a correct per-row bound
    formed in the kernel from kmax2 and the q row keeps exp(s - c) finite and
    non-zero.  Fused entry (own key pass) and caller-provided kmax2 both match
    the oracle; Ls = 300 is ragged."""
    # bf16: D = 128, scores up to 0.088 * 48 * 40 = 170; fp32 (exact fp32
    # scores must stay within 1e-4): D = 64, up to 0.125 * 48 * 16.7 = 100
    D, beta = (128, 40.0) if dtype == torch.bfloat16 else (64, 16.7)
    q, k, v = aligned_qk(2, 4, 2, 900, D, 14, 48.0, beta, dtype)
    ro, rl = oracle_ring(q, k, v, 3, "const_max", causal, layout)
    assert np.isfinite(rl).all() and rl.max() > 90
    o, lse = ca.ring_attn_fwd(q, k, v, 3, mode="const_max", causal=causal, layout=layout)
    assert_close(np32(o), ro, np32(lse), rl, dtype=dtype, what=f"fused {dtype} {layout}")
    o2, lse2 = ca.ring_attn_fwd_kmax(q, k, v, ca.key_max2(k), 3, causal=causal, layout=layout)
    assert_close(np32(o2), ro, np32(lse2), rl, dtype=dtype, what=f"kmax {dtype} {layout}")


@pytest.mark.parametrize("causal,layout", [(False, "contiguous"), (True, "striped")])
def test_online_max_large_jumps(ca, causal, layout):
    """Online max where the row maximum keeps jumping from tile to tile by up
    to ~245 log2 units (keys of growing norm along the sequence, scores to
    170 nats): the kernel's reference moves by whole powers of two after a
    speculative pass, or recomputes the tile when a jump is too large to
    represent; both must agree with the oracle."""
    q, k, v = aligned_qk(1, 4, 2, 2048, 128, 16, 48.0, 40.0, torch.float32)
    ramp = torch.linspace(0.02, 1.0, 2048, device="cuda").view(1, 1, 2048, 1)
    q, k, v = q.bfloat16(), (k * ramp).bfloat16(), v.bfloat16()
    ro, rl = oracle_ring(q, k, v, 4, "online_max", causal, layout)
    o, lse = ca.ring_attn_fwd(q, k, v, 4, mode="online_max", causal=causal, layout=layout)
    assert_close(np32(o), ro, np32(lse), rl, what=f"online jumps {layout}")


def test_const_max_in_kernel_bound_equals_given_bound(ca):
    """The row bound formed in the kernel and the one ca_const_max_bound
    writes agree to fp32 rounding, so the two entry points agree."""
    q, k, v = aligned_qk(1, 8, 2, 2048, 128, 15, 30.0, 40.0, torch.bfloat16)
    c, km = ca.const_max_bound(q, k)
    o1, l1 = ca.ring_attn_fwd_bounded(q, k, v, c, 4)
    o2, l2 = ca.ring_attn_fwd_kmax(q, k, v, km, 4)
    np.testing.assert_allclose(np32(l2), np32(l1), rtol=0, atol=2e-5)
    assert (np32(o2) - np32(o1)).__abs__().max() <= 1e-2


# --------------------------------------------------------------- layouts (bit-exact)


def test_layout_permutations_bit_exact(ca):
    x = torch.randint(-2**15, 2**15, (2, 3, 96, 64), dtype=torch.int16, device="cuda").view(torch.bfloat16)
    for cp in (1, 4, 8):
        Ls = 96 // cp
        for layout in ("contiguous", "striped"):
            y = ca.layout_to_shards(x, cp, layout)
            rows = [ca.layout_global_index(layout, cp, Ls, r) for r in range(96)]
            assert torch.equal(y.view(torch.int16), x[:, :, rows].view(torch.int16))
            assert torch.equal(ca.layout_from_shards(y, cp, layout).view(torch.int16), x.view(torch.int16))


def test_dcp_shard_kv_bit_exact(ca):
    W, I, L = 4, 16, 256
    kv = torch.randint(-2**15, 2**15, (3, 2, L, 128), dtype=torch.int16, device="cuda").view(torch.bfloat16)
    sh = ca.dcp_shard_kv(kv, W, I)
    own, loc = oracle.dcp_deal(L, W, I)
    ref = np.zeros((W, 3, 2, L // W, 128), np.int16)
    kvn = kv.view(torch.int16).cpu().numpy()
    for p in range(L):
        ref[own[p], :, :, loc[p]] = kvn[:, :, p]
    assert np.array_equal(sh.view(torch.int16).cpu().numpy(), ref)


def test_striped_ring_equals_contiguous_after_unpermuting(ca):
    """Invariant (e) on the GPU path: causal ring attention over striped
    storage, un-permuted, equals the contiguous causal result of the global
    sequence (both from the CUDA kernels), and both match the oracle."""
    cp, S = 4, 1024
    qg, kg, vg = gen(1, 2, 2, S, 128, 12, torch.bfloat16)
    oc, lc = ca.ring_attn_fwd(qg, kg, vg, cp, causal=True, layout="contiguous")
    qs, ks, vs = (ca.layout_to_shards(t, cp, "striped") for t in (qg, kg, vg))
    os_, ls_ = ca.ring_attn_fwd(qs, ks, vs, cp, causal=True, layout="striped")
    back = ca.layout_from_shards(os_, cp, "striped")
    lback = ca.layout_from_shards(ls_.unsqueeze(-1).repeat(1, 1, 1, 4).contiguous(), cp, "striped")[..., 0]
    d = (back.float() - oc.float()).abs()
    assert d.max().item() <= 2e-2 and d.mean().item() <= 2e-3
    assert (lback - lc).abs().max().item() <= 1e-3


def test_concurrent_calls_from_two_threads(ca):
    """Two host threads, each with its own stream, call the library at the
    same time (the ring on one, DCP decode on the other, repeatedly); every
    result is bit-identical to the same call made alone."""
    import threading

    from context_attention_gb300 import synth

    q, k, v = gen(1, 4, 2, 1024, 128, 51, torch.bfloat16)
    qd, kd, vd = synth.decode_inputs(4, 8, 2, 128, 4, 512, 52, device="cuda")
    o_ref, l_ref = ca.ring_attn_fwd(q, k, v, 4, mode="online_max", causal=True, layout="striped")
    od_ref, ld_ref = ca.dcp_decode(qd, kd, vd, 16)
    torch.cuda.synchronize()
    results, errors = {}, []

    def worker(name, fn):
        try:
            s = torch.cuda.Stream()
            outs = []
            with torch.cuda.stream(s):
                for _ in range(8):
                    outs.append(fn())
            s.synchronize()
            results[name] = outs
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append(e)

    t1 = threading.Thread(target=worker, args=("ring", lambda: ca.ring_attn_fwd(q, k, v, 4, mode="online_max",
                                                                                 causal=True, layout="striped")))
    t2 = threading.Thread(target=worker, args=("decode", lambda: ca.dcp_decode(qd, kd, vd, 16)))
    t1.start()
    t2.start()
    t1.join()
    t2.join()
    assert not errors, errors
    for o, lse in results["ring"]:
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    for o, lse in results["decode"]:
        assert torch.equal(o, od_ref) and torch.equal(lse, ld_ref)


def test_calls_replay_inside_a_cuda_graph(ca):
    """The entry points only enqueue work on the caller's stream, so a caller
    can capture them in a CUDA graph (after one warm-up call per kernel, which
    sets the kernels' shared-memory limits): replaying the graph on new
    inputs gives the same bits as eager calls."""
    from context_attention_gb300 import synth

    q, k, v = gen(1, 4, 4, 2048, 128, 61, torch.bfloat16)
    qd, kd, vd = synth.decode_inputs(4, 8, 2, 128, 4, 512, 62, device="cuda")
    ca.ring_attn_fwd(q, k, v, 4, mode="const_max")
    ca.dcp_decode(qd, kd, vd, 16)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        o, lse = ca.ring_attn_fwd(q, k, v, 4, mode="const_max")
        od, ld = ca.dcp_decode(qd, kd, vd, 16)
    for seed in (63, 64):
        q2, k2, v2 = gen(1, 4, 4, 2048, 128, seed, torch.bfloat16)
        q.copy_(q2), k.copy_(k2), v.copy_(v2)
        qd.copy_(torch.randn_like(qd.float()).to(qd.dtype))
        g.replay()
        torch.cuda.synchronize()
        o_e, l_e = ca.ring_attn_fwd(q, k, v, 4, mode="const_max")
        od_e, ld_e = ca.dcp_decode(qd, kd, vd, 16)
        torch.cuda.synchronize()
        assert torch.equal(o, o_e) and torch.equal(lse, l_e)
        assert torch.equal(od, od_e) and torch.equal(ld, ld_e)
    assert ca.device_status() == 0
