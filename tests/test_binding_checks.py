"""The Python binding's argument checks, on the CPU.

The C ABI takes plain pointers and sizes, so the binding is where a tensor of
the wrong shape or dtype is caught before a kernel would read or write past
it.  Shapes and dtypes are checked before placement, so host tensors reach
every check here: a call with the documented shapes gets as far as "must be a
CUDA tensor" (the shapes are accepted and nothing runs on the host), and each
operand changed on its own is refused by name."""
import pytest
import torch

BF, F32, I32, I64 = torch.bfloat16, torch.float32, torch.int32, torch.int64


@pytest.fixture(scope="module")
def ca():
    import context_attention_gb300 as m

    m.build()
    return m


def z(*shape, dtype=BF):
    return torch.zeros(*shape, dtype=dtype)


def accepted(fn, *args, **kw):
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        fn(*args, **kw)


def refused(fn, what, *args, **kw):
    with pytest.raises(ValueError, match=what):
        fn(*args, **kw)


def test_ring_forward_family(ca):
    B, Hq, Hkv, S, D = 2, 8, 2, 256, 128
    q, k, v = z(B, Hq, S, D), z(B, Hkv, S, D), z(B, Hkv, S, D)
    accepted(ca.ring_attn_fwd, q, k, v, 4)
    accepted(ca.ring_attn_fwd, q, k, v, 4, out=z(B, Hq, S, D), lse=z(B, Hq, S, dtype=F32),
             workspace=z(64, dtype=torch.uint8))
    accepted(ca.ring_attn_fwd, q, k, v, 4, return_lse=False, lse=z(3))  # lse unused
    refused(ca.ring_attn_fwd, "k: shape", q, z(B, Hkv, S + 1, D), v, 4)
    refused(ca.ring_attn_fwd, "v: shape", q, k, z(B, Hkv + 1, S, D), 4)
    refused(ca.ring_attn_fwd, "k: dtype", q, z(B, Hkv, S, D, dtype=F32), v, 4)
    refused(ca.ring_attn_fwd, "q: dtype", z(B, Hq, S, D, dtype=torch.float16), k, v, 4)
    refused(ca.ring_attn_fwd, "out: shape", q, k, v, 4, out=z(B, Hq, S, D // 2))
    refused(ca.ring_attn_fwd, "out: dtype", q, k, v, 4, out=z(B, Hq, S, D, dtype=F32))
    refused(ca.ring_attn_fwd, "lse: shape", q, k, v, 4, lse=z(B, Hq, S - 1, dtype=F32))
    refused(ca.ring_attn_fwd, "lse: dtype", q, k, v, 4, lse=z(B, Hq, S))
    refused(ca.ring_attn_fwd, "q must be a 4-d", z(Hq, S, D), k, v, 4)
    # caller-provided bound / key maximum (non-contiguous ones are made contiguous)
    accepted(ca.ring_attn_fwd_bounded, q, k, v, z(B, Hq, S, dtype=F32), 4)
    accepted(ca.ring_attn_fwd_bounded, q, k, v, z(B, S, Hq, dtype=F32).transpose(1, 2), 4)
    refused(ca.ring_attn_fwd_bounded, "c: shape", q, k, v, z(B, Hq, dtype=F32), 4)
    refused(ca.ring_attn_fwd_bounded, "c: dtype", q, k, v, z(B, Hq, S), 4)
    accepted(ca.ring_attn_fwd_kmax, q, k, v, z(B, Hkv, dtype=F32), 4)
    refused(ca.ring_attn_fwd_kmax, "kmax2: shape", q, k, v, z(B, Hq, dtype=F32), 4)
    refused(ca.ring_attn_fwd_kmax, "kmax2: dtype", q, k, v, z(B, Hkv, dtype=torch.float64), 4)
    # key pass and bound
    accepted(ca.key_max2, k)
    refused(ca.key_max2, "out: shape", k, out=z(B, Hkv, 1, dtype=F32))
    accepted(ca.const_max_bound, q, k)
    refused(ca.const_max_bound, "k: shape", q, z(B, Hkv, S, 64))


def test_partial_step_and_merge(ca):
    B, Hq, Hkv, Ls, D, cp = 1, 4, 2, 160, 128, 4
    qs, ks, vs = z(B, Hq, Ls, D), z(B, Hkv, Ls, D), z(B, Hkv, Ls, D)
    accepted(ca.attn_partial_step, qs, ks, vs, 0, 1, cp)
    accepted(ca.attn_partial_step, qs, ks, vs, 0, 1, cp, mode="const_max", c=z(B, Hq, Ls, dtype=F32))
    refused(ca.attn_partial_step, "k_shard: shape", qs, z(B, Hkv, Ls * 2, D), vs, 0, 1, cp)
    refused(ca.attn_partial_step, "c: shape", qs, ks, vs, 0, 1, cp, mode="const_max", c=z(B, Hq, Ls * cp, dtype=F32))
    # merge: o_parts [n, ..., D], lse_parts [n, ...], bound [...] (any shape of that size)
    op, lp = z(cp, B, Hq, Ls, D, dtype=F32), z(cp, B, Hq, Ls, dtype=F32)
    accepted(ca.lse_merge, op, lp)
    accepted(ca.lse_merge, op, lp, c=z(B, Hq, Ls, dtype=F32), out_dtype=BF)
    accepted(ca.lse_merge, z(5, 300, 128, dtype=F32), z(5, 300, dtype=F32))
    refused(ca.lse_merge, "lse_parts: shape", op, z(cp, B, Hq, Ls + 1, dtype=F32))
    refused(ca.lse_merge, "o_parts: dtype", op.to(BF), lp)
    refused(ca.lse_merge, "c: .* elements", op, lp, c=z(B, Hq, dtype=F32))
    refused(ca.lse_merge, "out_dtype", op, lp, out_dtype=torch.float16)


def test_prologue(ca):
    B, S, Hq, Hkv, D = 1, 64, 8, 2, 128
    x_q, x_k, x_v = z(B, S, Hq * D), z(B, S, Hkv * D), z(B, S, Hkv * D)
    g_q, g_k = z(Hq * D, dtype=F32), z(Hkv * D, dtype=F32)
    cos, sin = z(S, D // 2, dtype=F32), z(S, D // 2, dtype=F32)
    accepted(ca.qkv_prologue, x_q, x_k, Hq, Hkv, x_v=x_v, g_q=g_q, g_k=g_k, rope_cos=cos, rope_sin=sin, cp_size=2)
    accepted(ca.qkv_prologue, x_q, x_k, Hq, Hkv)  # no gains, no rotation, no v
    refused(ca.qkv_prologue, "x_k: shape", x_q, z(B, S, Hq * D), Hq, Hkv)
    refused(ca.qkv_prologue, "x_v: dtype", x_q, x_k, Hq, Hkv, x_v=z(B, S, Hkv * D, dtype=F32))
    refused(ca.qkv_prologue, "g_q: .* elements", x_q, x_k, Hq, Hkv, g_q=g_k)
    refused(ca.qkv_prologue, "g_k: dtype", x_q, x_k, Hq, Hkv, g_k=z(Hkv * D))
    refused(ca.qkv_prologue, "rope_cos: .* elements", x_q, x_k, Hq, Hkv, rope_cos=z(S - 1, D // 2, dtype=F32),
            rope_sin=z(S - 1, D // 2, dtype=F32))
    refused(ca.qkv_prologue, "go together", x_q, x_k, Hq, Hkv, rope_cos=cos)
    refused(ca.qkv_prologue, "not Hq=", x_q, x_k, 3, Hkv)


def test_decode_family(ca):
    N, Hq, Hkv, W, Lloc, D = 3, 8, 2, 4, 512, 128
    q, ks, vs = z(N, Hq, D), z(W, N, Hkv, Lloc, D), z(W, N, Hkv, Lloc, D)
    sl = z(N, dtype=I32)
    accepted(ca.dcp_decode, q, ks, vs, 16)
    accepted(ca.dcp_decode, q, ks, vs, 16, seq_lens=sl, out=z(N, Hq, D), lse=z(N, Hq, dtype=F32),
             workspace=z(1024, dtype=torch.uint8))
    refused(ca.dcp_decode, "k_shards: shape", q, z(W, N + 1, Hkv, Lloc, D), vs, 16)
    refused(ca.dcp_decode, "v_shards: shape", q, ks, z(W, N, Hkv, Lloc - 16, D), 16)
    refused(ca.dcp_decode, "seq_lens: shape", q, ks, vs, 16, seq_lens=z(N - 1, dtype=I32))
    refused(ca.dcp_decode, "seq_lens: dtype", q, ks, vs, 16, seq_lens=z(N, dtype=I64))
    refused(ca.dcp_decode, "lse: shape", q, ks, vs, 16, lse=z(N, Hkv, dtype=F32))
    accepted(ca.dcp_decode_noalloc, q, ks, vs, 16, seq_lens=sl)
    refused(ca.dcp_decode_noalloc, "out: dtype", q, ks, vs, 16, out=z(N, Hq, D, dtype=F32))
    # Ring Pass-Q decode over [B, Hkv, S, D]
    k, v = z(N, Hkv, 512, D), z(N, Hkv, 512, D)
    accepted(ca.ring_decode, q, k, v, 4, layout="striped", seq_lens=sl)
    refused(ca.ring_decode, "k: shape", q, z(N, Hkv, 512, 64), v, 4)
    refused(ca.ring_decode, "seq_lens: shape", q, k, v, 4, seq_lens=z(N + 1, dtype=I32))


def test_paged_cache(ca):
    N, Hq, Hkv, W, nblk, bs, mb, D = 3, 8, 2, 4, 40, 16, 8, 128
    q, kc, vc = z(N, Hq, D), z(W, nblk, Hkv, bs, D), z(W, nblk, Hkv, bs, D)
    bt, sl = z(W, N, mb, dtype=I32), z(N, dtype=I32)
    accepted(ca.dcp_decode_paged, q, kc, vc, bt, 16, sl)
    refused(ca.dcp_decode_paged, "block_tables: shape", q, kc, vc, z(W - 1, N, mb, dtype=I32), 16, sl)
    refused(ca.dcp_decode_paged, "block_tables: dtype", q, kc, vc, bt.to(I64), 16, sl)
    refused(ca.dcp_decode_paged, "v_cache: shape", q, kc, z(W, nblk, Hkv, bs * 2, D), bt, 16, sl)
    refused(ca.dcp_decode_paged, "seq_lens is required", q, kc, vc, bt, 16, None)
    T = 5
    k_new, v_new, slots = z(T, Hkv, D), z(T, Hkv, D), z(W, T, dtype=I64)
    accepted(ca.paged_kv_write, k_new, v_new, slots, kc, vc)
    refused(ca.paged_kv_write, "slots: shape", k_new, v_new, z(W, T + 1, dtype=I64), kc, vc)
    refused(ca.paged_kv_write, "slots: dtype", k_new, v_new, slots.to(I32), kc, vc)
    refused(ca.paged_kv_write, "v_new: shape", k_new, z(T, Hkv, 64), slots, kc, vc)
    refused(ca.paged_kv_write, "k_cache: dtype", k_new, v_new, slots, kc.to(F32), vc)


def test_dcp_prefill(ca):
    Hq, Hkv, W, Sc, Lcap, Lc, D = 4, 2, 4, 384, 128, 96, 128
    q = z(Hq, Sc, D)
    kp, vp, kc, vc = z(W, Hkv, Lcap, D), z(W, Hkv, Lcap, D), z(W, Hkv, Lc, D), z(W, Hkv, Lc, D)
    accepted(ca.dcp_prefill, q, kp, vp, kc, vc, 16, 500)
    accepted(ca.dcp_prefill, q, kp, vp, kc, vc, 16, 500, out=z(Hq, Sc, D), lse=z(Hq, Sc, dtype=F32))
    accepted(ca.dcp_prefill_partial, q, kp, vp, kc, vc, 16, 500, 1)
    refused(ca.dcp_prefill, "v_prior: shape", q, kp, z(W, Hkv, Lcap + 1, D), kc, vc, 16, 500)
    refused(ca.dcp_prefill, "k_cur: shape", q, kp, vp, z(W - 1, Hkv, Lc, D), vc, 16, 500)
    refused(ca.dcp_prefill, "v_cur: dtype", q, kp, vp, kc, vc.to(F32), 16, 500)
    refused(ca.dcp_prefill, "out: shape", q, kp, vp, kc, vc, 16, 500, out=z(Hq, Sc, 64))
    refused(ca.dcp_prefill_partial, "k_prior: shape", q, z(W, Hkv, Lcap, 64), vp, kc, vc, 16, 500, 1)


def test_workspace_size_counts_bytes(ca):
    """A workspace of any dtype is passed with its size in bytes."""
    assert ca._ws_bytes(z(10, dtype=F32)) == 40
    assert ca._ws_bytes(z(10, dtype=torch.uint8)) == 10
    assert ca._ws_bytes(None) == 0


def test_layout_permutations_refuse_host_tensors(ca):
    """The row permutations move raw rows of any dtype; host tensors and
    tensors with fewer than three dimensions are refused before any copy."""
    x = z(2, 4, 64, 128)
    for fn in (lambda t: ca.layout_to_shards(t, 4, "striped"), lambda t: ca.layout_from_shards(t, 4),
               lambda t: ca.dcp_shard_kv(t, 4, 16)):
        with pytest.raises(ValueError, match="contiguous CUDA tensor"):
            fn(x)
        with pytest.raises(ValueError, match="contiguous CUDA tensor"):
            fn(z(64, 128))
