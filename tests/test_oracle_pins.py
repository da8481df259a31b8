"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

None of these tests re-types the oracle's formulas.  Each one checks a value
that is known independently: a closed form, an invariant the pages state, a
brute-force enumeration, or a hand-computed case.  Each is chosen so that a
plausible slip in the oracle (a dropped scale, a wrong GQA index, an
off-by-one on the causal diagonal, a transposed striped map, a wrong merge
weight) fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle as ora

RNG = np.random.default_rng(1234)


def rnd(*shape):
    return RNG.standard_normal(shape).astype(np.float32)


# ---------------------------------------------------------------- closed forms


def test_two_keys_hand_computed():
    """D=1, scale 0.5, q=1, keys 0 and 2 ln 3: weights 1:3, o=(v1+3 v2)/4, lse=ln 4."""
    q = np.ones((1, 1, 2, 1), np.float32)
    k = np.array([0.0, 2 * math.log(3.0)], np.float32).reshape(1, 1, 2, 1)
    v = np.array([2.0, 6.0], np.float32).reshape(1, 1, 2, 1)
    o, lse = ora.attention(q, k, v, scale=0.5)
    k2 = float(np.float32(2 * math.log(3.0)))  # the stored key, rounded to fp32
    w2 = math.exp(0.5 * k2)
    expect_o = (2.0 + w2 * 6.0) / (1.0 + w2)
    assert abs(o[0, 0] - expect_o) < 1e-12
    assert abs(lse[0] - math.log(1.0 + w2)) < 1e-12
    assert abs(o[0, 0] - 5.0) < 1e-6 and abs(lse[0] - math.log(4.0)) < 1e-6


def test_zero_query_gives_mean_and_log_count_noncausal_gqa():
    """q = 0: every score is 0, so o = mean of the head's values, lse = ln S.
    Hq=4, Hkv=2: heads 0,1 read kv head 0, heads 2,3 kv head 1."""
    B, Hq, Hkv, S, D = 2, 4, 2, 24, 8
    q = np.zeros((B, Hq, S, D), np.float32)
    k, v = rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    o, lse = ora.attention(q, k, v)
    o = o.reshape(B, Hq, S, D)
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_allclose(o[b, h], np.broadcast_to(v[b, h // 2].astype(np.float64).mean(0), (S, D)), atol=1e-12)
    np.testing.assert_allclose(lse, math.log(S), atol=1e-12)


def test_zero_query_causal_contiguous_prefix_means():
    """Causal, q = 0: query at global position i sees keys 0..i (diagonal
    included), so o_i = mean(v_0..v_i) and lse_i = ln(i + 1)."""
    B, H, S, D, cp = 1, 1, 32, 4, 4
    q = np.zeros((B, H, S, D), np.float32)
    k, v = rnd(B, H, S, D), rnd(B, H, S, D)
    o, lse = ora.attention(q, k, v, causal=True, layout=ora.LAYOUT_CONTIGUOUS, cp=cp)
    vd = v[0, 0].astype(np.float64)
    for i in range(S):
        np.testing.assert_allclose(o[i], vd[: i + 1].mean(0), atol=1e-12)
        assert abs(lse[i] - math.log(i + 1)) < 1e-12


def test_zero_query_causal_striped_prefix_means():
    """Striped storage: stored row r*Ls + a is global token a*cp + r.  With
    q = 0 the output of that row is the mean of the values of global tokens
    0..a*cp + r, wherever they are stored."""
    B, H, S, D, cp = 1, 1, 24, 3, 4
    Ls = S // cp
    q = np.zeros((B, H, S, D), np.float32)
    k, v = rnd(B, H, S, D), rnd(B, H, S, D)
    o, lse = ora.attention(q, k, v, causal=True, layout=ora.LAYOUT_STRIPED, cp=cp)
    # position of each stored row, built from the page's "token t on shard t mod cp"
    pos_of_row = np.empty(S, np.int64)
    for t in range(S):
        pos_of_row[(t % cp) * Ls + t // cp] = t
    vd = v[0, 0].astype(np.float64)
    for rho in range(S):
        vis = pos_of_row <= pos_of_row[rho]
        np.testing.assert_allclose(o[rho], vd[vis].mean(0), atol=1e-12)
        assert abs(lse[rho] - math.log(vis.sum())) < 1e-12


def test_single_visible_key():
    """Causal: the query at global position 0 sees only key 0: o = v_0,
    lse = scale * q_0 . k_0."""
    B, H, S, D = 1, 2, 16, 8
    q, k, v = rnd(B, H, S, D), rnd(B, H, S, D), rnd(B, H, S, D)
    rows = [0, S]  # (h=0, rho=0) and (h=1, rho=0)
    o, lse = ora.attention(q, k, v, causal=True, rows=rows, scale=0.3)
    for i, h in enumerate((0, 1)):
        np.testing.assert_allclose(o[i], v[0, h, 0], atol=1e-12)
        assert abs(lse[i] - 0.3 * float(np.dot(q[0, h, 0].astype(np.float64), k[0, h, 0]))) < 1e-12


def test_constant_values_give_the_constant():
    """Invariant (d): every v row equal to u  =>  o = u for any q, k."""
    B, Hq, Hkv, S, D = 1, 4, 2, 40, 6
    q, k = rnd(B, Hq, S, D) * 3, rnd(B, Hkv, S, D) * 3
    u = rnd(Hkv, D)
    v = np.broadcast_to(u[None, :, None, :], (B, Hkv, S, D)).copy()
    for causal in (False, True):
        o, _ = ora.attention(q, k, v, causal=causal, cp=4)
        o = o.reshape(B, Hq, S, D)
        for h in range(Hq):
            np.testing.assert_allclose(o[0, h], np.broadcast_to(u[h // 2], (S, D)), atol=1e-12)
        o2, _, _ = ora.ring(q, k, v, cp=4, mode=ora.MODE_CONST_MAX, causal=causal)
        np.testing.assert_allclose(o2.reshape(B, Hq, S, D)[0, 3], np.broadcast_to(u[1], (S, D)), atol=1e-12)


def test_against_textbook_softmax_tiny():
    """Brute force on a tiny case with scipy's softmax / logsumexp as the
    library routine: o = softmax(scale*q k^T) v per head."""
    from scipy.special import logsumexp, softmax

    B, Hq, Hkv, S, D = 1, 2, 1, 9, 5
    q, k, v = rnd(B, Hq, S, D), rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    o, lse = ora.attention(q, k, v, scale=0.7)
    o = o.reshape(Hq, S, D)
    lse = lse.reshape(Hq, S)
    for h in range(Hq):
        sc = 0.7 * q[0, h].astype(np.float64) @ k[0, 0].astype(np.float64).T
        np.testing.assert_allclose(o[h], softmax(sc, axis=1) @ v[0, 0].astype(np.float64), atol=1e-12)
        np.testing.assert_allclose(lse[h], logsumexp(sc, axis=1), atol=1e-12)


def test_noncausal_key_permutation_invariance():
    B, H, S, D = 1, 2, 20, 4
    q, k, v = rnd(B, H, S, D), rnd(B, H, S, D), rnd(B, H, S, D)
    perm = RNG.permutation(S)
    o1, l1 = ora.attention(q, k, v)
    o2, l2 = ora.attention(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


# ---------------------------------------------------------------- merge (a)


def test_merge_hand_computed():
    """Two partials with lse 0 and ln 3: weights 1/4 and 3/4; total lse ln 4."""
    o_parts = np.array([[[4.0, 0.0]], [[0.0, 8.0]]])
    lse_parts = np.array([[0.0], [math.log(3.0)]])
    o, lse = ora.lse_merge(o_parts, lse_parts)
    np.testing.assert_allclose(o[0], [1.0, 6.0], atol=1e-12)
    assert abs(lse[0] - math.log(4.0)) < 1e-12


def test_merge_empty_partials():
    o_parts = np.array([[[1.0, 2.0]], [[3.0, 4.0]]])
    o, lse = ora.lse_merge(o_parts, np.array([[-np.inf], [-np.inf]]))
    assert lse[0] == -np.inf and np.all(o == 0)
    o, lse = ora.lse_merge(o_parts, np.array([[-np.inf], [0.5]]))
    np.testing.assert_allclose(o[0], [3.0, 4.0], atol=1e-15)
    assert abs(lse[0] - 0.5) < 1e-15


@pytest.mark.parametrize("causal,layout", [(False, 0), (True, 0), (True, 1)])
def test_merged_shard_partials_equal_full_attention(causal, layout):
    """Invariant (a): LSE-merging every shard's partial gives full attention,
    in any merge order; splitting a shard in two changes nothing."""
    B, Hq, Hkv, S, D, cp = 1, 4, 2, 32, 8, 4
    q, k, v = rnd(B, Hq, S, D), rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    o_full, l_full = ora.attention(q, k, v, causal=causal, layout=layout, cp=cp)
    parts = [ora.shard_partial(q, k, v, s, cp, causal=causal, layout=layout) for s in range(cp)]
    for order in (range(cp), [2, 0, 3, 1]):
        o, l = ora.lse_merge(np.stack([parts[i][0] for i in order]), np.stack([parts[i][1] for i in order]))
        np.testing.assert_allclose(o, o_full, atol=1e-12)
        np.testing.assert_allclose(l, l_full, atol=1e-12)
    if layout == 0:
        # contiguous shards of cp=2 are pairs of cp=4 shards
        for s2 in range(2):
            o2, l2 = ora.shard_partial(q, k, v, s2, 2, causal=causal, layout=0)
            o4, l4 = ora.lse_merge(np.stack([parts[2 * s2][0], parts[2 * s2 + 1][0]]),
                                   np.stack([parts[2 * s2][1], parts[2 * s2 + 1][1]]))
            fin = np.isfinite(l2)
            np.testing.assert_allclose(o4, o2, atol=1e-12)
            np.testing.assert_allclose(l4[fin], l2[fin], atol=1e-12)
            assert np.array_equal(fin, np.isfinite(l4))


# ---------------------------------------------------------------- ring, (b), (c)


@pytest.mark.parametrize("causal,layout", [(False, 0), (True, 0), (True, 1)])
def test_ring_online_and_const_max_equal_full(causal, layout):
    """Invariant (b): shifting a row by any constant leaves softmax unchanged,
    so the const-max ring equals the online-max ring equals full attention."""
    B, Hq, Hkv, S, D, cp = 2, 4, 2, 48, 16, 4
    q, k, v = rnd(B, Hq, S, D), rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    o_full, l_full = ora.attention(q, k, v, causal=causal, layout=layout, cp=cp)
    o_on, l_on, _ = ora.ring(q, k, v, cp, mode=ora.MODE_ONLINE_MAX, causal=causal, layout=layout)
    o_cm, l_cm, ov = ora.ring(q, k, v, cp, mode=ora.MODE_CONST_MAX, causal=causal, layout=layout)
    for o, l in ((o_on, l_on), (o_cm, l_cm)):
        np.testing.assert_allclose(o, o_full, atol=1e-12)
        np.testing.assert_allclose(l, l_full, atol=1e-11)
    assert np.all(ov >= -1e-12)


def test_ring_cp1_is_plain_attention():
    B, H, S, D = 1, 2, 16, 4
    q, k, v = rnd(B, H, S, D), rnd(B, H, S, D), rnd(B, H, S, D)
    o, l = ora.attention(q, k, v)
    o1, l1, _ = ora.ring(q, k, v, 1)
    np.testing.assert_allclose(o1, o, atol=1e-13)
    np.testing.assert_allclose(l1, l, atol=1e-13)


def test_bound_dominates_every_score_and_is_tight_when_parallel():
    """Invariant (c): scale*q_i.k_j <= c_i for all j (Cauchy-Schwarz), with
    equality when q_i is parallel to the longest key of its head."""
    B, Hq, Hkv, S, D = 1, 4, 2, 30, 8
    q, k = rnd(B, Hq, S, D), rnd(B, Hkv, S, D)
    jmax = int(np.argmax((k[0, 1].astype(np.float64) ** 2).sum(1)))
    q[0, 2, 5] = 2.5 * k[0, 1, jmax]  # head 2 reads kv head 1
    c, kmax2 = ora.const_max_bound(q, k, scale=0.25)
    for h in range(Hq):
        sc = 0.25 * q[0, h].astype(np.float64) @ k[0, h // 2].astype(np.float64).T
        assert np.all(sc <= c[0, h][:, None] * (1 + 1e-15) + 1e-15)
    np.testing.assert_allclose(kmax2[0], [(k[0, j].astype(np.float64) ** 2).sum(1).max() for j in range(Hkv)], rtol=1e-15)
    s_eq = 0.25 * float(q[0, 2, 5].astype(np.float64) @ k[0, 1, jmax].astype(np.float64))
    assert abs(c[0, 2, 5] - s_eq) <= 1e-12 * abs(s_eq)


def test_const_max_overshoot_and_clamp_failure_mode():
    """A key sink lifts every row's bound (the const-max page, "Adapting this
    kernel").  A moderate sink leaves the result exact; once the overshoot
    c_i - max_j s_ij passes ln(1/1e-37) ~ 85.2 nats the row sum falls under
    the 1e-37 clamp and the row comes out (nearly) all zeros, the page's
    "Output is all zeros" symptom, while lse = c + ln(acc_l) stays right."""
    B, H, S, D, cp = 1, 1, 64, 16, 2
    q, k, v = rnd(B, H, S, D), rnd(B, H, S, D), rnd(B, H, S, D)
    _, _, ov0 = ora.ring(q, k, v, cp, mode=ora.MODE_CONST_MAX)
    of0, _ = ora.attention(q, k, v)
    # moderate sink: overshoot grows but stays far below the clamp
    k4 = k.copy()
    k4[0, 0, 7] *= 4
    o4, l4, ov4 = ora.ring(q, k4, v, cp, mode=ora.MODE_CONST_MAX)
    assert np.median(ov4) > 3 * np.median(ov0) and ov4.max() < 80
    of4, lf4 = ora.attention(q, k4, v)
    np.testing.assert_allclose(o4, of4, atol=1e-11)
    np.testing.assert_allclose(l4, lf4, atol=1e-11)
    # huge sink: rows past ~85.2 nats of overshoot hit the clamp
    k40 = k.copy()
    k40[0, 0, 7] *= 40
    o40, l40, ov40 = ora.ring(q, k40, v, cp, mode=ora.MODE_CONST_MAX)
    of40, lf40 = ora.attention(q, k40, v)
    hit = ov40 > 85.2 + 1.0
    safe = ov40 < 85.2 - 1.0
    assert hit.sum() > 0
    assert np.all(np.abs(o40[hit]).max(axis=1) < 1e-3 * np.abs(of40[hit]).max(axis=1))
    np.testing.assert_allclose(o40[safe], of40[safe], atol=1e-10)
    np.testing.assert_allclose(l40, lf40, atol=1e-9)
    del of0


# ---------------------------------------------------------------- layouts (e)


def test_striped_causal_equals_contiguous_after_unpermuting():
    """Invariant (e): store a globally ordered sequence striped (token t at row
    (t mod cp)*Ls + t div cp), run causal attention with the striped layout,
    un-permute the rows: the result equals the contiguous causal result."""
    B, Hq, Hkv, S, D, cp = 1, 2, 1, 40, 8, 4
    Ls = S // cp
    qg, kg, vg = rnd(B, Hq, S, D), rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    row_of_token = np.array([(t % cp) * Ls + t // cp for t in range(S)])
    perm = np.empty(S, np.int64)
    perm[row_of_token] = np.arange(S)  # stored row -> global token
    qs, ks, vs = qg[:, :, perm], kg[:, :, perm], vg[:, :, perm]
    o_c, l_c = ora.attention(qg, kg, vg, causal=True, layout=ora.LAYOUT_CONTIGUOUS, cp=cp)
    o_s, l_s = ora.attention(qs, ks, vs, causal=True, layout=ora.LAYOUT_STRIPED, cp=cp)
    o_c = o_c.reshape(B, Hq, S, D)
    o_s = o_s.reshape(B, Hq, S, D)
    np.testing.assert_allclose(o_s[:, :, row_of_token], o_c, atol=1e-12)
    np.testing.assert_allclose(l_s.reshape(B, Hq, S)[:, :, row_of_token], l_c.reshape(B, Hq, S), atol=1e-12)
    # the ring in both layouts agrees as well
    o_r, _, _ = ora.ring(qs, ks, vs, cp, causal=True, layout=ora.LAYOUT_STRIPED)
    np.testing.assert_allclose(o_r.reshape(B, Hq, S, D)[:, :, row_of_token], o_c, atol=1e-12)


def test_global_pos_matches_page_maps():
    # contiguous: start = cp_rank * local_S (golden: rank 7 of S=1024, cp=8 -> 896..1023)
    assert ora.global_pos(0, 8, 128, 7 * 128) == 896
    assert ora.global_pos(0, 8, 128, 7 * 128 + 127) == 1023
    # striped: token t on shard t mod cp
    for t in range(64):
        r, a = t % 8, t // 8
        assert ora.global_pos(1, 8, 8, r * 8 + a) == t


# ---------------------------------------------------------------- DCP decode


def _shard_by_page_formula(kg, W, I):
    """Shard global K [N,Hkv,L,D] with the page's slot -> global formula."""
    N, Hkv, L, D = kg.shape
    Lloc = L // W
    out = np.zeros((W, N, Hkv, Lloc, D), kg.dtype)
    for R in range(W):
        for s in range(Lloc):
            out[R, :, :, s] = kg[:, :, (s // I) * (W * I) + R * I + (s % I)]
    return out


def test_dcp_decode_equals_attention_over_the_global_sequence():
    """Decoding against interleaved shards = plain attention of the query over
    global positions [0, seq_len), for lengths on and off block boundaries."""
    N, Hq, Hkv, D, W, I = 3, 4, 2, 8, 4, 4
    L = 64
    q = rnd(N, Hq, D)
    kg, vg = rnd(N, Hkv, L, D), rnd(N, Hkv, L, D)
    ks, vs = _shard_by_page_formula(kg, W, I), _shard_by_page_formula(vg, W, I)
    seq_lens = np.array([64, 37, 1])
    o, lse = ora.dcp_decode(q, ks, vs, I, seq_lens=seq_lens)
    for n in range(N):
        Ln = seq_lens[n]
        # full attention of the single query over the visible prefix
        kk = kg[n, :, :Ln][None]
        vv = vg[n, :, :Ln][None]
        qfull = np.zeros((1, Hq, Ln, D), np.float32)
        qfull[0, :, 0] = q[n]
        rows = [h * Ln for h in range(Hq)]
        o_ref, l_ref = ora.attention(qfull, kk, vv, rows=rows)
        np.testing.assert_allclose(o[n], o_ref, atol=1e-12)
        np.testing.assert_allclose(lse[n], l_ref, atol=1e-12)


def test_dcp_decode_zero_query_closed_form():
    N, Hq, Hkv, D, W, I = 2, 2, 1, 4, 2, 16
    L = 128
    q = np.zeros((N, Hq, D), np.float32)
    kg, vg = rnd(N, Hkv, L, D), rnd(N, Hkv, L, D)
    ks, vs = _shard_by_page_formula(kg, W, I), _shard_by_page_formula(vg, W, I)
    seq_lens = np.array([100, 17])
    o, lse = ora.dcp_decode(q, ks, vs, I, seq_lens=seq_lens)
    for n in range(N):
        np.testing.assert_allclose(o[n], np.broadcast_to(vg[n, 0, : seq_lens[n]].astype(np.float64).mean(0), (Hq, D)), atol=1e-12)
        np.testing.assert_allclose(lse[n], math.log(seq_lens[n]), atol=1e-12)


# ---------------------------------------------------------------- ring Pass-Q decode


def _ring_cache(kg, cp, layout):
    """Store a global-order cache [B, Hkv, S, D] in the ring layout by dealing
    tokens as "Sharding the Input" describes: contiguous blocks of S/cp tokens
    per shard, or (striped) token t to shard t mod cp as its (t div cp)-th."""
    B, Hkv, S, D = kg.shape
    Ls = S // cp
    out = np.empty_like(kg)
    for t in range(S):
        r, a = (t // Ls, t % Ls) if layout == ora.LAYOUT_CONTIGUOUS else (t % cp, t // cp)
        out[:, :, r * Ls + a] = kg[:, :, t]
    return out


@pytest.mark.parametrize("layout", [ora.LAYOUT_CONTIGUOUS, ora.LAYOUT_STRIPED])
def test_ring_decode_equals_attention_over_the_prefix(layout):
    """Pass-Q decode over the ring layout's shards = plain attention of the
    query over global positions [0, seq_len); cache slots at or past seq_len
    hold junk that must not be read."""
    B, Hq, Hkv, D, cp, S = 3, 4, 2, 8, 4, 48
    q = rnd(B, Hq, D)
    kg, vg = rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    seq_lens = np.array([48, 29, 1])
    kj, vj = kg.copy(), vg.copy()
    for b in range(B):
        kj[b, :, seq_lens[b]:] = 1e3
        vj[b, :, seq_lens[b]:] = -1e3
    k, v = _ring_cache(kj, cp, layout), _ring_cache(vj, cp, layout)
    o, lse = ora.ring_decode(q, k, v, cp, layout, seq_lens=seq_lens)
    for b in range(B):
        Lb = seq_lens[b]
        qfull = np.zeros((1, Hq, Lb, D), np.float32)
        qfull[0, :, 0] = q[b]
        o_ref, l_ref = ora.attention(qfull, kg[b, :, :Lb][None], vg[b, :, :Lb][None], rows=[h * Lb for h in range(Hq)])
        np.testing.assert_allclose(o[b], o_ref, atol=1e-12)
        np.testing.assert_allclose(lse[b], l_ref, atol=1e-12)


def test_ring_decode_closed_forms():
    """q = 0: the mean of the visible values and lse = ln(seq_len); one
    visible token: its value and lse = scale q.k; no visible token: o = 0,
    lse = -inf."""
    B, Hq, Hkv, D, cp, S = 3, 2, 1, 4, 8, 64
    kg, vg = rnd(B, Hkv, S, D), rnd(B, Hkv, S, D)
    for layout in (ora.LAYOUT_CONTIGUOUS, ora.LAYOUT_STRIPED):
        k, v = _ring_cache(kg, cp, layout), _ring_cache(vg, cp, layout)
        seq_lens = np.array([64, 21, 3])
        o, lse = ora.ring_decode(np.zeros((B, Hq, D), np.float32), k, v, cp, layout, seq_lens=seq_lens)
        for b in range(B):
            mean = vg[b, 0, : seq_lens[b]].astype(np.float64).mean(0)
            np.testing.assert_allclose(o[b], np.broadcast_to(mean, (Hq, D)), atol=1e-12)
            np.testing.assert_allclose(lse[b], math.log(seq_lens[b]), atol=1e-12)
        q = rnd(B, Hq, D)
        o, lse = ora.ring_decode(q, k, v, cp, layout, seq_lens=np.array([1, 1, 0]), scale=0.25)
        for b in range(2):
            np.testing.assert_allclose(o[b], np.broadcast_to(vg[b, 0, 0].astype(np.float64), (Hq, D)), atol=1e-12)
            np.testing.assert_allclose(lse[b], 0.25 * q[b].astype(np.float64) @ kg[b, 0, 0].astype(np.float64), atol=1e-12)
        assert np.all(o[2] == 0.0) and np.all(np.isneginf(lse[2]))


# ---------------------------------------------------------------- DCP prefill


def _dcp_prefill_shards(kg, P, Sc, W, I, Lcap):
    """Split a global K [Hkv, P+Sc, D] into prior shards [W,Hkv,Lcap,D] (prior
    slot s of rank R = global (s//I)*(W*I) + R*I + s%I) and current shards
    [W,Hkv,Sc/W,D] (chunk token j of rank R = global P + (j//I)*(W*I) + R*I + j%I),
    both maps as the DCP page's "Segmented Attention CP" step 3 prints them."""
    Hkv, L, D = kg.shape
    prior = np.full((W, Hkv, Lcap, D), 1e3, np.float32)  # unused slots: junk that must never be read
    cur = np.zeros((W, Hkv, Sc // W, D), np.float32)
    for R in range(W):
        for s in range(Lcap):
            g = (s // I) * (W * I) + R * I + s % I
            if g < P:
                prior[R, :, s] = kg[:, g]
        for j in range(Sc // W):
            cur[R, :, j] = kg[:, P + (j // I) * (W * I) + R * I + j % I]
    return prior, cur


@pytest.mark.parametrize("P", [0, 16, 64, 77])
def test_dcp_prefill_equals_causal_attention_over_prefix(P):
    """A chunk of Sc new tokens after P cached ones, split over W ranks:
    the merged result equals plain causal attention of the chunk's queries
    (global positions P..P+Sc-1) over the whole global sequence."""
    Hq, Hkv, D, W, I, Sc = 4, 2, 8, 4, 4, 32
    L = P + Sc
    Lcap = 40
    q = rnd(Hq, Sc, D)
    kg, vg = rnd(Hkv, L, D), rnd(Hkv, L, D)
    kp, kc = _dcp_prefill_shards(kg, P, Sc, W, I, Lcap)
    vp, vc = _dcp_prefill_shards(vg, P, Sc, W, I, Lcap)
    o, lse = ora.dcp_prefill(q, kp, vp, kc, vc, I, P)
    qfull = np.zeros((1, Hq, L, D), np.float32)
    qfull[0, :, P:] = q
    rows = [h * L + P + i for h in range(Hq) for i in range(Sc)]
    ro, rl = ora.attention(qfull, kg[None], vg[None], causal=True, rows=rows)
    np.testing.assert_allclose(o.reshape(-1, D), ro, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(-1), rl, atol=1e-12)
    # per-rank partials, LSE-merged, give the same (page steps 4-7)
    parts = [ora.dcp_prefill(q, kp, vp, kc, vc, I, P, part_rank=R) for R in range(W)]
    mo, ml = ora.lse_merge(np.stack([p[0].reshape(-1, D) for p in parts]), np.stack([p[1].reshape(-1) for p in parts]))
    np.testing.assert_allclose(mo, ro, atol=1e-12)
    np.testing.assert_allclose(ml, rl, atol=1e-12)


def test_dcp_prefill_zero_query_prefix_means():
    """q = 0: the chunk query at global position P+i gets the mean of v over
    positions 0..P+i and lse = ln(P+i+1)."""
    Hq, Hkv, D, W, I, Sc, P = 2, 1, 4, 2, 4, 16, 24
    q = np.zeros((Hq, Sc, D), np.float32)
    kg, vg = rnd(Hkv, P + Sc, D), rnd(Hkv, P + Sc, D)
    kp, kc = _dcp_prefill_shards(kg, P, Sc, W, I, 16)
    vp, vc = _dcp_prefill_shards(vg, P, Sc, W, I, 16)
    o, lse = ora.dcp_prefill(q, kp, vp, kc, vc, I, P)
    for i in range(Sc):
        np.testing.assert_allclose(o[:, i], np.broadcast_to(vg[0, : P + i + 1].astype(np.float64).mean(0), (Hq, D)), atol=1e-12)
        np.testing.assert_allclose(lse[:, i], math.log(P + i + 1), atol=1e-12)


# ---------------------------------------------------------------- paged DCP decode


def test_dcp_decode_paged_equals_contiguous_shards():
    """Scattering each rank's local slots over shuffled physical blocks of a
    paged cache (block table per rank and sequence) changes nothing: the
    paged decode equals the decode over the contiguous shards."""
    N, Hq, Hkv, D, W, I, bs = 3, 4, 2, 8, 4, 16, 16
    Lloc = 64
    max_blocks = Lloc // bs
    q = rnd(N, Hq, D)
    ks, vs = rnd(W, N, Hkv, Lloc, D), rnd(W, N, Hkv, Lloc, D)
    seq_lens = np.array([W * Lloc, 100, 1])
    nblk = N * max_blocks + 5
    kc = rnd(W, nblk, Hkv, bs, D) * 100  # unused blocks: junk
    vc = rnd(W, nblk, Hkv, bs, D) * 100
    bt = np.zeros((W, N, max_blocks), np.int32)
    rng = np.random.default_rng(5)
    for r in range(W):
        perm = rng.permutation(nblk)[: N * max_blocks].reshape(N, max_blocks)
        bt[r] = perm
        for n in range(N):
            for lb in range(max_blocks):
                kc[r, perm[n, lb]] = ks[r, n, :, lb * bs:(lb + 1) * bs]
                vc[r, perm[n, lb]] = vs[r, n, :, lb * bs:(lb + 1) * bs]
    o1, l1 = ora.dcp_decode(q, ks, vs, I, seq_lens=seq_lens)
    o2, l2 = ora.dcp_decode_paged(q, kc, vc, bt, I, seq_lens)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2, l1, atol=1e-12)


# ---------------------------------------------------------------- QK prologue (RMS norm, RoPE, layout)


def _rope_tables(S, D, base=10000.0):
    """Per-position angles p * base^(-2i/D) (one per channel pair)."""
    ang = np.arange(S)[:, None] * base ** (-2.0 * np.arange(D // 2) / D)[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32), ang


def test_prologue_rms_norm_unit_mean_square_and_scale_invariance():
    """With eps = 0 and no gain every token's normalised hidden has mean
    square exactly 1, and rescaling a token's activations changes nothing."""
    B, S, H, D = 2, 6, 3, 8
    x = rnd(B, S, H * D)
    out = ora.qk_prologue(x, H, eps=0.0)
    ms = (out.transpose(0, 2, 1, 3).reshape(B, S, H * D) ** 2).mean(-1)
    np.testing.assert_allclose(ms, 1.0, atol=1e-12)
    alpha = np.array([0.25, 4.0, 1e3, 1e-3, 7.0, 0.5])[None, :, None].astype(np.float32)
    out2 = ora.qk_prologue(x * alpha, H, eps=0.0)
    np.testing.assert_allclose(out2, out, atol=1e-6)


def test_prologue_eps_and_gain_per_channel_of_the_whole_hidden():
    """A token whose activations are all c: y = c / sqrt(c^2 + eps) * g_j,
    with the gain indexed by the channel of the whole hidden (h*D + d)."""
    B, S, H, D = 1, 2, 2, 4
    x = np.full((B, S, H * D), 0.5, np.float32)
    g = (1.0 + np.arange(H * D)).astype(np.float32)
    eps = 0.75
    out = ora.qk_prologue(x, H, g=g, eps=eps)
    want = 0.5 / math.sqrt(0.25 + eps) * g.reshape(H, D)
    for s in range(S):
        np.testing.assert_allclose(out[0, :, s, :], want, atol=1e-12)


def test_prologue_rope_identity_and_quarter_turn():
    """cos = 1, sin = 0 leaves the normalised values alone; a quarter turn
    maps each channel pair (y0, y1) of every head to (-y1, y0)."""
    B, S, H, D = 1, 3, 2, 8
    x = rnd(B, S, H * D)
    plain = ora.qk_prologue(x, H)
    one, zero = np.ones((S, D // 2), np.float32), np.zeros((S, D // 2), np.float32)
    np.testing.assert_allclose(ora.qk_prologue(x, H, cos=one, sin=zero), plain, atol=1e-15)
    turned = ora.qk_prologue(x, H, cos=zero, sin=one)
    np.testing.assert_allclose(turned[..., 0::2], -plain[..., 1::2], atol=1e-15)
    np.testing.assert_allclose(turned[..., 1::2], plain[..., 0::2], atol=1e-15)


def test_prologue_rope_keeps_norms_and_depends_on_relative_position():
    """Rotation keeps every head's norm; with angles p * w_i the product of a
    rotated query at m and key at n depends on m - n only."""
    S, H, D = 12, 1, 16
    cos, sin, _ = _rope_tables(S, D)
    u, w = rnd(D), rnd(D)
    # the same q vector (before norm) at every position; likewise k
    xq = np.tile(u, (1, S, 1)).astype(np.float32)
    xk = np.tile(w, (1, S, 1)).astype(np.float32)
    q = ora.qk_prologue(xq, H, cos=cos, sin=sin, eps=0.0)[0, 0]
    k = ora.qk_prologue(xk, H, cos=cos, sin=sin, eps=0.0)[0, 0]
    q0 = ora.qk_prologue(xq, H, eps=0.0)[0, 0]
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), np.linalg.norm(q0, axis=-1), rtol=1e-6)
    for m, n, t in ((3, 1, 5), (0, 7, 4), (9, 9, 2)):
        np.testing.assert_allclose(q[m] @ k[n], q[m + t] @ k[n + t], atol=1e-5)


def test_prologue_striped_rows_hold_the_dealt_tokens():
    """Striped layout: stored row r*Ls + a of every head holds token a*cp + r
    (the contiguous output's row), for q-style and value-style tensors."""
    B, S, H, D, cp = 2, 12, 2, 4, 3
    x = rnd(B, S, H * D)
    cos, sin, _ = _rope_tables(S, D)
    Ls = S // cp
    for norm in (True, False):
        cont = ora.qk_prologue(x, H, cos=cos, sin=sin, norm=norm)
        strp = ora.qk_prologue(x, H, cos=cos, sin=sin, norm=norm, cp=cp, layout=ora.LAYOUT_STRIPED)
        for r in range(cp):
            for a in range(Ls):
                np.testing.assert_array_equal(strp[:, :, r * Ls + a], cont[:, :, a * cp + r])
    # value-style (no norm, no rope): the plain head split and transpose
    v = ora.qk_prologue(x, H, norm=False)
    np.testing.assert_array_equal(v, x.reshape(B, S, H, D).transpose(0, 2, 1, 3))
