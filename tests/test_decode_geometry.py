"""How the decode divides its work, checked on the host.

The decode deals the 128-token stages of every (shard, sequence, KV head)
pair to its CTAs: round robin in splits of 32 stages when there are 256
pairs or more, otherwise as one contiguous range per CTA.  A CTA writes one
partial per pair its range meets, into slot (its index - the index of the
pair's first CTA); the workspace query sizes the partials for the most slots
any launch of up to 256 CTAs can use.  These tests restate the kernel's
integer arithmetic and enumerate every CTA count, so a wrong bound (a slot
past the workspace) or a gap in the dealing (a slot nobody writes, a stage
read twice) fails here without a GPU."""
import ctypes

import pytest

K_TOK = 128
MAX_CTAS = 256
DEAL_PAIRS = 256
SPLIT_STAGES = 32


def slots_for(pairs, Lloc, ctas_max):
    stages = -(-Lloc // K_TOK)
    if pairs >= DEAL_PAIRS:
        return -(-stages // SPLIT_STAGES)
    units = pairs * stages
    ctas = min(units, ctas_max)
    return min((stages - 1) // (units // ctas) + 2, stages)


def deal_contiguous(pairs, stages, ctas):
    """Every CTA's segments: (pair, first stage, end stage, slot, last)."""
    units = pairs * stages
    segs = []
    for c in range(ctas):
        u, u1 = c * units // ctas, (c + 1) * units // ctas
        while u < u1:
            p = u // stages
            pu0 = p * stages
            s1 = min(u1, pu0 + stages)
            first_cta = ((pu0 + 1) * ctas - 1) // units
            segs.append((c, p, u - pu0, s1 - pu0, c - first_cta, s1 == pu0 + stages))
            u = s1
    return segs


@pytest.fixture(scope="module")
def lib():
    import context_attention_gb300 as m

    m.build()
    L = ctypes.CDLL(m.library_path())
    L.ca_dcp_decode_workspace_size.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.ca_dcp_decode_workspace_size.restype = ctypes.c_size_t
    L.ca_ring_decode_workspace_size.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                                ctypes.c_int, ctypes.c_int]
    L.ca_ring_decode_workspace_size.restype = ctypes.c_size_t
    return L


@pytest.mark.parametrize("N,Hq,Hkv,Lloc,W", [(1, 32, 8, 32768, 4), (2, 32, 8, 32768, 4), (7, 16, 8, 3840, 4),
                                             (8, 16, 8, 3840, 4), (64, 32, 8, 32768, 4), (1, 8, 1, 131072, 1),
                                             (3, 4, 1, 100, 2), (32, 32, 4, 128, 31)])
def test_workspace_holds_the_most_slots_a_launch_can_use(lib, N, Hq, Hkv, Lloc, W):
    a256 = lambda x: -(-x // 256) * 256
    parts = W * slots_for(W * N * Hkv, Lloc, MAX_CTAS)
    want = a256(4 * parts * N * Hq * 128) + a256(4 * parts * N * Hq)
    assert lib.ca_dcp_decode_workspace_size(N, Hq, Hkv, Lloc, 128, W, 16) == want
    # the ring layout's decode: cp shards of S / cp slots, the same partials
    assert lib.ca_ring_decode_workspace_size(N, Hq, Hkv, W * Lloc, 128, W) == want


@pytest.mark.parametrize("pairs", [1, 2, 3, 8, 24, 32, 64, 100, 224, 255])
@pytest.mark.parametrize("Lloc", [1, 128, 129, 1000, 3840, 32768])
def test_contiguous_ranges_cover_every_stage_once_within_the_slot_bound(pairs, Lloc):
    stages = -(-Lloc // K_TOK)
    bound = slots_for(pairs, Lloc, MAX_CTAS)
    for ctas_max in list(range(1, 17)) + [100, 148, 152, 160, 255, 256]:
        ctas = min(pairs * stages, ctas_max)
        slots = slots_for(pairs, Lloc, ctas_max)
        assert slots <= bound
        segs = deal_contiguous(pairs, stages, ctas)
        covered = [0] * (pairs * stages)
        written = set()
        for c, p, s0, s1, slot, last in segs:
            assert 0 <= slot < slots, (pairs, Lloc, ctas, c, slot, slots)
            for s in range(s0, s1):
                covered[p * stages + s] += 1
            assert (p, slot) not in written
            written.add((p, slot))
            if last:  # the pair's last CTA marks the slots nobody reaches
                for sl in range(slot + 1, slots):
                    assert (p, sl) not in written
                    written.add((p, sl))
        assert covered == [1] * (pairs * stages)
        assert written == {(p, sl) for p in range(pairs) for sl in range(slots)}


def test_dealt_splits_cover_every_stage_once():
    for pairs, Lloc, ctas in ((256, 32768, 152), (300, 1000, 152), (2048, 4097, 148), (256, 128, 256)):
        stages = -(-Lloc // K_TOK)
        splits = slots_for(pairs, Lloc, ctas)
        covered = [0] * (pairs * stages)
        units = pairs * splits
        for c in range(min(units, ctas)):
            for u in range(c, units, min(units, ctas)):
                p, sp = divmod(u, splits)
                for s in range(sp * SPLIT_STAGES, min((sp + 1) * SPLIT_STAGES, stages)):
                    covered[p * stages + s] += 1
        assert covered == [1] * (pairs * stages)
