"""Index maps: the pages' worked examples, the oracle's enumeration, and the
library's closed forms (host helpers of libctxattn.so), all bit-exact."""
import os

import numpy as np
import pytest

import oracle as ora

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    rows, params = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line:
                continue
            if line.startswith("#"):
                for tok in line[1:].split():
                    if tok.count("=") == 1:
                        k, v = tok.split("=")
                        if v.isdigit():
                            params[k] = int(v)
                continue
            rows.append([int(x) for x in line.split()])
    return rows, params


@pytest.fixture(scope="module")
def ca():
    import context_attention_gb300 as m

    m.build()
    return m


# ----------------------------------------------------------- oracle vs pages


def test_oracle_deal_matches_page_block_table():
    rows, p = read_golden("dcp_block_owner_I16_W4.txt")
    own, _ = ora.dcp_deal(100, p["dcp"], p["interleave"])
    for block, first, last, owner in rows:
        assert np.all(own[first:last + 1] == owner), block


def test_oracle_deal_matches_prefill_token_groups():
    rows, p = read_golden("dcp_prefill_token_groups_TP8_DCP4.txt")
    I = 16
    own, _ = ora.dcp_deal(12 * I, p["dcp"], I)
    for tp_rank, cp_rank, *blocks in rows:
        assert tp_rank // (p["tp"] // p["dcp"]) == cp_rank
        for b in blocks:
            assert np.all(own[b * I:(b + 1) * I] == cp_rank)


def test_oracle_deal_matches_decode_even_odd():
    rows, p = read_golden("dcp_decode_ranks_TP16_DCP2.txt")
    I = 16
    own, _ = ora.dcp_deal(20 * I, p["dcp"], I)
    for tp_rank, dcp_rank, parity in rows:
        assert tp_rank % p["dcp"] == dcp_rank
        blocks = [b for b in range(20) if own[b * I] == dcp_rank]
        assert all(b % 2 == parity for b in blocks)


def test_oracle_local_index_matches_page_global_formula():
    rows, p = read_golden("dcp_global_position_example.txt")
    W, I = p["dcp"], p["interleave"]
    own, loc = ora.dcp_deal(400, W, I)
    for rank, slot, gpos in rows:
        assert own[gpos] == rank and loc[gpos] == slot


def test_oracle_slot_view_of_owned_positions():
    """The model runner's owned-slot view view(S//(W*I), W, I)[:, R, :] picks
    exactly the positions the deal gives rank R, in local order."""
    W, I, S = 4, 16, 512
    own, loc = ora.dcp_deal(S, W, I)
    view = np.arange(S).reshape(S // (W * I), W, I)
    for R in range(W):
        owned = view[:, R, :].reshape(-1)
        assert np.array_equal(owned, np.nonzero(own == R)[0])
        assert np.array_equal(loc[owned], np.arange(len(owned)))


def test_oracle_local_filled_sums_to_n():
    for W, I in ((4, 16), (2, 16), (3, 4)):
        for N in (0, 1, 15, 16, 17, 63, 64, 65, 1000, 1237):
            assert sum(ora.dcp_local_filled(N, W, I, R) for R in range(W)) == N


# ----------------------------------------------------------- library vs oracle


def test_contiguous_golden(ca):
    rows, p = read_golden("cp_contiguous_ranks_S1024_CP8.txt")
    cp, Ls = p["cp"], p["S"] // p["cp"]
    for rank, first, last in rows:
        assert ca.layout_global_index("contiguous", cp, Ls, rank * Ls) == first
        assert ca.layout_global_index("contiguous", cp, Ls, rank * Ls + Ls - 1) == last


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_layout_maps_are_inverse_bijections(ca, layout):
    for cp, Ls in ((8, 8), (4, 5), (1, 7), (3, 1)):
        S = cp * Ls
        glob = [ca.layout_global_index(layout, cp, Ls, r) for r in range(S)]
        assert sorted(glob) == list(range(S))
        for rho, g in enumerate(glob):
            assert ca.layout_shard_row(layout, cp, Ls, g) == rho
            assert g == ora.global_pos(ora.LAYOUT_STRIPED if layout == "striped" else 0, cp, Ls, rho)
    assert ca.layout_global_index(layout, 4, 4, 16) == -1


def test_striped_is_token_mod_cp(ca):
    cp, Ls = 8, 16
    for t in range(cp * Ls):
        rho = ca.layout_shard_row("striped", cp, Ls, t)
        assert rho // Ls == t % cp


def test_ring_schedule(ca):
    # step t on rank r uses the K/V of rank r - t (mod cp); over cp steps every shard once
    for cp in (1, 2, 5, 8):
        for r in range(cp):
            seen = [ca.ring_kv_shard(r, t, cp) for t in range(cp)]
            assert seen[0] == r and sorted(seen) == list(range(cp))
            assert all(seen[t] == (r - t) % cp for t in range(cp))


@pytest.mark.parametrize("W,I", [(4, 16), (2, 16), (3, 4), (1, 8)])
def test_dcp_maps_bit_exact_against_deal(ca, W, I):
    n = W * I * 9 + 5
    own, loc = ora.dcp_deal(n, W, I)
    for p in range(n):
        assert ca.dcp_owner(p, W, I) == own[p]
        assert ca.dcp_local_index(p, W, I) == loc[p]
        assert ca.dcp_local_to_global(int(loc[p]), int(own[p]), W, I) == p


@pytest.mark.parametrize("W,I,mult", [(4, 16, 1), (2, 16, 1), (3, 4, 1), (4, 16, 2), (2, 4, 4)])
def test_local_filled_formula_equals_enumeration(ca, W, I, mult):
    """The page's formula (block_size a multiple of the interleave) equals the
    count of dealt tokens, for every N below a few thousand."""
    bs = I * mult
    for N in range(0, 3 * W * bs + 7):
        for R in range(W):
            assert ca.dcp_local_filled(N, W, I, bs, R) == ora.dcp_local_filled(N, W, I, R), (N, R)


def test_active_mask_owner_only(ca):
    W, I = 4, 16
    own, _ = ora.dcp_deal(600, W, I)
    for N in range(0, 600):
        masks = [ca.dcp_active_mask(N, W, I, I, R) for R in range(W)]
        assert sum(masks) == 1 and masks[own[N]] == 1


def test_slot_mapping(ca):
    W, I, bs = 4, 16, 16
    positions = np.arange(0, 512)
    block_table = np.array([7, 3, 9, 1, 2, 5, 6, 8], dtype=np.int32)
    own, loc = ora.dcp_deal(512, W, I)
    for R in range(W):
        slots = ca.dcp_slot_mapping(positions, block_table, bs, W, R, I)
        for p in positions:
            if own[p] != R:
                assert slots[p] == -1
            else:
                # local token loc[p] lives in the rank's local block loc // bs
                lb = loc[p] // bs
                assert slots[p] == block_table[lb] * bs + loc[p] % bs


def test_sequence_divisibility_error(ca):
    import torch

    rows, _ = read_golden("cp_seq_divisibility.txt")
    S, cp, rem, accepted = rows[0]
    assert S % cp == rem and accepted == 0
    from helpers import real_allocation

    lib = ca._load()
    keep, buf = real_allocation(1 << 16)  # real memory, never read: validation fails first
    st = lib.ca_ring_attn_fwd(buf, buf, buf, buf, None, 1, 1, 40, 40, S, 128, cp, 0, 0, 0, 0.0,
                              None, 0, None)
    assert ca.STATUS[st] == "CA_ERR_SHAPE"
    del keep
    del torch
