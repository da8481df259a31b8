"""GPU parity of DCP decode over paged KV caches and of the slot-mapping
cache write, through the C ABI."""
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


def page(ks, vs, bs, seed, spare=7):
    """Scatter contiguous shards [W,N,Hkv,Lloc,D] into per-rank paged caches
    [W,nblk,Hkv,bs,D] over shuffled physical blocks; unused blocks hold NaN."""
    W, N, Hkv, Lloc, D = ks.shape
    mb = Lloc // bs
    nblk = N * mb + spare
    kc = torch.full((W, nblk, Hkv, bs, D), float("nan"), dtype=ks.dtype, device=ks.device)
    vc = torch.full_like(kc, float("nan"))
    bt = torch.zeros(W, N, mb, dtype=torch.int32)
    g = torch.Generator().manual_seed(seed)
    for r in range(W):
        perm = torch.randperm(nblk, generator=g)[: N * mb].view(N, mb)
        bt[r] = perm
        for n in range(N):
            for lb in range(mb):
                kc[r, perm[n, lb]] = ks[r, n, :, lb * bs:(lb + 1) * bs]
                vc[r, perm[n, lb]] = vs[r, n, :, lb * bs:(lb + 1) * bs]
    return kc, vc, bt.cuda()


@pytest.mark.parametrize("bs", [8, 16, 32, 64, 128])
def test_paged_decode_matches_contiguous_and_oracle(ca, bs):
    from context_attention_gb300 import synth

    N, Hq, Hkv, W, I, Lloc = 3, 8, 2, 4, 16, 1024
    q, ks, vs = synth.decode_inputs(N, Hq, Hkv, 128, W, Lloc, 40 + bs, device="cuda")
    lens = [W * Lloc, 1000, 17]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    kc, vc, bt = page(ks, vs, bs, seed=bs)
    o, lse = ca.dcp_decode_paged(q, kc, vc, bt, I, sl)
    o2, l2 = ca.dcp_decode(q, ks, vs, I, seq_lens=sl)
    assert torch.equal(o, o2) and torch.equal(lse, l2)  # same kernels, same arithmetic order
    ro, rl = oracle.dcp_decode_paged(np32(q), np32(torch.nan_to_num(kc)), np32(torch.nan_to_num(vc)),
                                     bt.cpu().numpy(), I, lens)
    assert_close(np32(o), ro, np32(lse), rl, what=f"paged decode bs={bs}")


def test_paged_kv_write_then_decode(ca):
    """Append one decoded token per sequence: slots from the slot mapping of
    the owning rank (-1 elsewhere), written bit-exactly into the paged caches;
    decoding the grown sequences equals attention over the global prefix."""
    from context_attention_gb300 import synth

    N, Hq, Hkv, W, I, bs, Lloc, D = 3, 4, 2, 4, 16, 16, 512, 128
    q, ks, vs = synth.decode_inputs(N, Hq, Hkv, D, W, Lloc, 50, device="cuda")
    kc, vc, bt = page(ks, vs, bs, seed=3)
    old = [700, 1023, 64]  # tokens already cached; the new token sits at position old[n]
    g = torch.Generator(device="cuda").manual_seed(51)
    k_new = torch.randn(N, Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    v_new = torch.randn(N, Hkv, D, generator=g, device="cuda").to(torch.bfloat16)
    slots = np.full((W, N), -1, np.int64)
    for r in range(W):
        for n in range(N):
            slots[r, n] = ca.dcp_slot_mapping([old[n]], bt[r, n].cpu().numpy(), bs, W, r, I)[0]
    assert all((slots[:, n] >= 0).sum() == 1 for n in range(N))  # the owner only
    for n in range(N):
        owners = [r for r in range(W) if ca.dcp_active_mask(old[n], W, I, bs, r)]
        assert owners == [int(np.nonzero(slots[:, n] >= 0)[0][0])]
    before_k, before_v = kc.clone(), vc.clone()
    ca.paged_kv_write(k_new, v_new, torch.tensor(slots, device="cuda"), kc, vc)
    # bit-exact: exactly the owners' slots changed, to the new rows
    exp_k, exp_v = before_k.clone(), before_v.clone()
    for r in range(W):
        for n in range(N):
            s = int(slots[r, n])
            if s >= 0:
                exp_k[r, s // bs, :, s % bs] = k_new[n]
                exp_v[r, s // bs, :, s % bs] = v_new[n]
    same = lambda a, b: torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert same(kc, exp_k) and same(vc, exp_v)
    lens = [o + 1 for o in old]
    o, lse = ca.dcp_decode_paged(q, kc, vc, bt, I, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    ro, rl = oracle.dcp_decode_paged(np32(q), np32(torch.nan_to_num(kc)), np32(torch.nan_to_num(vc)),
                                     bt.cpu().numpy(), I, lens)
    assert_close(np32(o), ro, np32(lse), rl, what="decode after append")
