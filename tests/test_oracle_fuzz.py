"""The oracle's own invariants on seeded random shapes (CPU, fp64).  Each check
compares two different routes through the oracle: the ring of per-shard
partials merged by log-sum-exp against plain attention (the authority), const
max against online max, striped storage against contiguous storage of the
same global sequence, and the decodes against attention of the query over the
cached prefix.  A shape-dependent slip in one route fails the comparison."""
import numpy as np
import pytest

import oracle as ora

TOL = 1e-11


def draws(n, seed):
    rng = np.random.default_rng(seed)
    for i in range(n):
        yield dict(i=i, B=int(rng.integers(1, 3)), Hkv=int(rng.integers(1, 4)), G=int(rng.integers(1, 4)),
                   cp=int(rng.integers(1, 7)), Ls=int(rng.integers(1, 40)), D=int(rng.integers(1, 17)),
                   causal=bool(rng.integers(0, 2)), scale=float(rng.choice([0.0, 0.1, 0.7])),
                   seed=int(rng.integers(0, 1 << 30)))


def to_striped(x, cp):
    """Global token order [..., S, D] -> striped shard-major storage: row
    r*Ls + a holds token a*cp + r."""
    S = x.shape[-2]
    Ls = S // cp
    rows = np.array([(rho % Ls) * cp + rho // Ls for rho in range(S)])
    return x[..., rows, :]


@pytest.mark.parametrize("c", list(draws(40, 7)), ids=lambda c: f"draw{c['i']}")
def test_ring_routes_agree(c):
    rng = np.random.default_rng(c["seed"])
    Hq, S = c["Hkv"] * c["G"], c["cp"] * c["Ls"]
    q = rng.standard_normal((c["B"], Hq, S, c["D"])).astype(np.float32)
    k = rng.standard_normal((c["B"], c["Hkv"], S, c["D"])).astype(np.float32)
    v = rng.standard_normal((c["B"], c["Hkv"], S, c["D"])).astype(np.float32)
    scale = c["scale"] or None
    o_ref, l_ref = ora.attention(q, k, v, scale=scale, causal=c["causal"])
    # contiguous storage: the ring in both modes equals plain attention
    for mode in (ora.MODE_ONLINE_MAX, ora.MODE_CONST_MAX):
        o, lse, _ = ora.ring(q, k, v, c["cp"], mode=mode, scale=scale, causal=c["causal"])
        np.testing.assert_allclose(np.asarray(o).reshape(o_ref.shape), o_ref, atol=TOL, err_msg=str(c))
        np.testing.assert_allclose(np.asarray(lse).reshape(l_ref.shape), l_ref, atol=TOL, err_msg=str(c))
    # the same global sequence stored striped: the same rows, permuted
    qs, ks, vs = to_striped(q, c["cp"]), to_striped(k, c["cp"]), to_striped(v, c["cp"])
    o, lse, _ = ora.ring(qs, ks, vs, c["cp"], scale=scale, causal=c["causal"], layout=ora.LAYOUT_STRIPED)
    o = np.asarray(o).reshape(c["B"], Hq, S, c["D"])
    np.testing.assert_allclose(o, to_striped(o_ref.reshape(c["B"], Hq, S, c["D"]), c["cp"]), atol=TOL,
                               err_msg=str(c))


@pytest.mark.parametrize("c", list(draws(20, 8)), ids=lambda c: f"draw{c['i']}")
def test_decode_routes_agree(c):
    rng = np.random.default_rng(c["seed"])
    Hq, W, I = c["Hkv"] * c["G"], min(c["cp"], 4), 4
    L = W * I * int(rng.integers(1, 6))  # whole interleave blocks on every rank
    q = rng.standard_normal((c["B"], Hq, c["D"])).astype(np.float32)
    kg = rng.standard_normal((c["B"], c["Hkv"], L, c["D"])).astype(np.float32)
    vg = rng.standard_normal((c["B"], c["Hkv"], L, c["D"])).astype(np.float32)
    lens = [int(x) for x in rng.integers(0, L + 1, size=c["B"])]
    scale = c["scale"] or None
    # DCP shards: slot s of rank R holds global (s // I) * (W * I) + R * I + s % I
    Lloc = L // W
    ks = np.zeros((W, c["B"], c["Hkv"], Lloc, c["D"]), np.float32)
    vs = np.zeros_like(ks)
    for R in range(W):
        for s in range(Lloc):
            gpos = (s // I) * (W * I) + R * I + s % I
            ks[R, :, :, s], vs[R, :, :, s] = kg[:, :, gpos], vg[:, :, gpos]
    o_d, l_d = ora.dcp_decode(q, ks, vs, I, seq_lens=lens, scale=scale)
    # the ring layout of the same cache, striped over W shards
    o_r, l_r = ora.ring_decode(q, to_striped(kg, W), to_striped(vg, W), W, ora.LAYOUT_STRIPED, seq_lens=lens,
                               scale=scale)
    for b in range(c["B"]):
        if lens[b] == 0:
            assert np.all(o_d[b] == 0) and np.all(np.isneginf(l_d[b])) and np.all(np.isneginf(l_r[b]))
            continue
        Lb = lens[b]
        qf = np.zeros((1, Hq, Lb, c["D"]), np.float32)
        qf[0, :, 0] = q[b]
        ro, rl = ora.attention(qf, kg[b:b + 1, :, :Lb], vg[b:b + 1, :, :Lb], scale=scale,
                               rows=[h * Lb for h in range(Hq)])
        for o, lse in ((o_d, l_d), (o_r, l_r)):
            np.testing.assert_allclose(o[b], ro, atol=TOL, err_msg=str(c))
            np.testing.assert_allclose(lse[b], rl, atol=TOL, err_msg=str(c))
