"""The C ABI without a GPU: the library builds, loads and exports every entry
point declared in include/ctxattn.h, and host-side validation returns the
documented status codes before anything touches a device."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Base address of a real 1 MiB allocation that these tests pass wherever a
# call wants a tensor (set by the fixture below; FAKE + 2 and the like stay
# inside it).  Every call here fails host validation, or is the zero-token
# cache write that does nothing, so the memory is never read; it is real
# memory all the same, so that no test hands the library an address nothing
# owns.
FAKE = None


@pytest.fixture(scope="module")
def ca():
    import context_attention_gb300 as m

    m.build()
    return m


@pytest.fixture(scope="module", autouse=True)
def real_buffer():
    from helpers import real_allocation

    global FAKE
    keep, FAKE = real_allocation(1 << 20)
    yield
    FAKE = None
    del keep


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ctxattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ca_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(ca):
    import ctypes

    names = declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(ca.library_path())
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(ca):
    lib = ca._load()
    for code, name in ca.STATUS.items():
        assert lib.ca_status_string(code).decode() == name
    assert lib.ca_version() >= 100


def ring(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, dtype=1, B=1, Hq=4, Hkv=2, S=1024, D=128, cp=4,
             mode=0, causal=0, layout=0, scale=0.0, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.ca_ring_attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dtype"], a["B"], a["Hq"],
                                a["Hkv"], a["S"], a["D"], a["cp"], a["mode"], a["causal"], a["layout"],
                                a["scale"], a["ws"], a["ws_bytes"], a["stream"])


def test_ring_validation_codes(ca):
    lib = ca._load()
    S = ca.STATUS
    assert S[ring(lib, q=None)] == "CA_ERR_INVALID_ARG"
    assert S[ring(lib, mode=7)] == "CA_ERR_INVALID_ARG"
    assert S[ring(lib, layout=2)] == "CA_ERR_INVALID_ARG"
    assert S[ring(lib, cp=0)] == "CA_ERR_INVALID_ARG"
    assert S[ring(lib, dtype=5)] == "CA_ERR_INVALID_ARG"
    assert S[ring(lib, S=3645, cp=8)] == "CA_ERR_SHAPE"
    assert S[ring(lib, Hq=6, Hkv=4)] == "CA_ERR_SHAPE"
    assert S[ring(lib, D=64)] == "CA_ERR_UNSUPPORTED"           # bf16 needs D = 128
    assert S[ring(lib, dtype=0, D=160)] == "CA_ERR_UNSUPPORTED"  # fp32 needs D <= 128
    assert S[ring(lib, q=FAKE + 2)] == "CA_ERR_ALIGNMENT"
    # the kernels view q as a [B*Hq*S, D] matrix with 32-bit row indices
    assert S[ring(lib, B=1 << 12, Hq=8, Hkv=8, S=1 << 16, cp=8)] == "CA_ERR_UNSUPPORTED"
    assert S[ring(lib, B=1 << 12, Hq=8, Hkv=8, S=(1 << 16) - 8, cp=8, q=None)] == "CA_ERR_INVALID_ARG"
    assert S[ring(lib, mode=1)] == "CA_ERR_WORKSPACE"            # const max needs the bound buffer
    need = lib.ca_ring_attn_fwd_workspace_size(1, 4, 2, 1024, 128, 4, 1)
    assert need >= 4 * 2                                         # kmax2 [B, Hkv]
    assert S[ring(lib, mode=1, ws=FAKE, ws_bytes=need - 1)] == "CA_ERR_WORKSPACE"
    assert lib.ca_ring_attn_fwd_workspace_size(1, 4, 2, 1024, 128, 4, 0) == 0


def test_key_max_and_kmax_ring_validation(ca):
    lib = ca._load()
    S = ca.STATUS
    assert S[lib.ca_key_max2(None, 1, 1, 2, 1024, 128, FAKE, None)] == "CA_ERR_INVALID_ARG"
    assert S[lib.ca_key_max2(FAKE, 1, 1, 2, 0, 128, FAKE, None)] == "CA_ERR_INVALID_ARG"
    assert S[lib.ca_key_max2(FAKE, 3, 1, 2, 1024, 128, FAKE, None)] == "CA_ERR_INVALID_ARG"
    assert S[lib.ca_key_max2(FAKE + 4, 1, 1, 2, 1024, 128, FAKE, None)] == "CA_ERR_ALIGNMENT"
    assert S[lib.ca_key_max2(FAKE, 1, 1, 2, 1024, 128, FAKE + 2, None)] == "CA_ERR_ALIGNMENT"

    def kring(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, km=FAKE, o=FAKE, lse=None, dtype=1, B=1, Hq=4, Hkv=2, S=1024, D=128,
                 cp=4, causal=0, layout=0, scale=0.0)
        a.update(kw)
        return lib.ca_ring_attn_fwd_kmax(a["q"], a["k"], a["v"], a["km"], a["o"], a["lse"], a["dtype"], a["B"],
                                         a["Hq"], a["Hkv"], a["S"], a["D"], a["cp"], a["causal"], a["layout"],
                                         a["scale"], None)

    assert S[kring(km=None)] == "CA_ERR_INVALID_ARG"
    assert S[kring(S=1020, cp=8)] == "CA_ERR_SHAPE"
    assert S[kring(Hq=6, Hkv=4)] == "CA_ERR_SHAPE"
    assert S[kring(D=64)] == "CA_ERR_UNSUPPORTED"
    assert S[kring(km=FAKE + 2)] == "CA_ERR_ALIGNMENT"


def test_partial_step_validation_codes(ca):
    lib = ca._load()
    S = ca.STATUS

    def step(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=1, B=1, Hq=2, Hkv=2, Ls=256, D=128, qr=0, kr=0, cp=2, mode=0,
                 causal=0, layout=0, scale=0.0, c=None, o=FAKE, lse=FAKE, stream=None)
        a.update(kw)
        return lib.ca_attn_partial_step(a["q"], a["k"], a["v"], a["dtype"], a["B"], a["Hq"], a["Hkv"], a["Ls"],
                                        a["D"], a["qr"], a["kr"], a["cp"], a["mode"], a["causal"], a["layout"],
                                        a["scale"], a["c"], a["o"], a["lse"], a["stream"])

    assert S[step(qr=2)] == "CA_ERR_INVALID_ARG"
    assert S[step(kr=-1)] == "CA_ERR_INVALID_ARG"
    assert S[step(mode=1)] == "CA_ERR_INVALID_ARG"      # const max needs c
    assert S[step(c=FAKE)] == "CA_ERR_INVALID_ARG"      # online max takes no c
    assert S[step(lse=None)] == "CA_ERR_INVALID_ARG"
    assert S[step(o=FAKE + 8)] == "CA_ERR_ALIGNMENT"


def test_merge_bound_decode_layout_validation(ca):
    lib = ca._load()
    S = ca.STATUS
    assert S[lib.ca_lse_merge(FAKE, FAKE, 0, 16, 128, None, FAKE, 0, None, None)] == "CA_ERR_INVALID_ARG"
    assert S[lib.ca_lse_merge(FAKE, FAKE, 2, 16, 126, None, FAKE, 0, None, None)] == "CA_ERR_UNSUPPORTED"
    assert S[lib.ca_const_max_bound(FAKE, FAKE, 1, 1, 6, 4, 64, 128, 0.0, FAKE, FAKE, None)] == "CA_ERR_SHAPE"
    assert S[lib.ca_const_max_bound(FAKE, FAKE, 1, 1, 4, 4, 64, 128, 0.0, FAKE, None, None)] == "CA_ERR_INVALID_ARG"

    def dec(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=1, N=2, Hq=8, Hkv=2, Lloc=256, D=128, W=4, I=16, seq=None,
                 scale=0.0, o=FAKE, lse=FAKE, ws=FAKE, ws_bytes=1 << 30, stream=None)
        a.update(kw)
        return lib.ca_dcp_decode(a["q"], a["k"], a["v"], a["dtype"], a["N"], a["Hq"], a["Hkv"], a["Lloc"], a["D"],
                                 a["W"], a["I"], a["seq"], a["scale"], a["o"], a["lse"], a["ws"], a["ws_bytes"],
                                 a["stream"])

    assert S[dec(Lloc=250)] == "CA_ERR_SHAPE"           # Lloc % interleave
    assert S[dec(Hq=6, Hkv=4)] == "CA_ERR_SHAPE"
    assert S[dec(dtype=0)] == "CA_ERR_UNSUPPORTED"
    assert S[dec(Hq=32, Hkv=2)] == "CA_ERR_UNSUPPORTED"  # more than 8 query heads per KV head
    assert S[dec(N=1 << 14, Hkv=8, Hq=8, Lloc=1 << 16, W=2)] == "CA_ERR_UNSUPPORTED"  # 2^31 cache rows
    assert S[dec(ws=None)] == "CA_ERR_WORKSPACE"
    assert S[dec(ws_bytes=16)] == "CA_ERR_WORKSPACE"
    assert lib.ca_dcp_decode_workspace_size(64, 32, 8, 32768, 128, 4, 16) > 64 * 32 * 128 * 4 * 4

    def rdec(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=1, B=2, Hq=8, Hkv=2, S=1024, D=128, cp=4, layout=0, seq=None,
                 scale=0.0, o=FAKE, lse=FAKE, ws=FAKE, ws_bytes=1 << 30, stream=None)
        a.update(kw)
        return lib.ca_ring_decode(a["q"], a["k"], a["v"], a["dtype"], a["B"], a["Hq"], a["Hkv"], a["S"], a["D"],
                                  a["cp"], a["layout"], a["seq"], a["scale"], a["o"], a["lse"], a["ws"],
                                  a["ws_bytes"], a["stream"])

    assert S[rdec(S=1022)] == "CA_ERR_SHAPE"            # S % cp_size
    assert S[rdec(Hq=6, Hkv=4)] == "CA_ERR_SHAPE"
    assert S[rdec(layout=2)] == "CA_ERR_INVALID_ARG"
    assert S[rdec(v=None)] == "CA_ERR_INVALID_ARG"
    assert S[rdec(dtype=0)] == "CA_ERR_UNSUPPORTED"
    assert S[rdec(D=64)] == "CA_ERR_UNSUPPORTED"
    assert S[rdec(Hq=32, Hkv=2)] == "CA_ERR_UNSUPPORTED"  # more than 8 query heads per KV head
    assert S[rdec(B=1 << 12, Hkv=8, Hq=8, S=1 << 16)] == "CA_ERR_UNSUPPORTED"  # 2^31 cache rows
    assert S[rdec(k=FAKE + 8)] == "CA_ERR_ALIGNMENT"
    assert S[rdec(ws=None)] == "CA_ERR_WORKSPACE"
    assert S[rdec(ws_bytes=16)] == "CA_ERR_WORKSPACE"
    # cp partials (each shard split like a DCP rank's slots) of every (sequence, head)
    assert lib.ca_ring_decode_workspace_size(2, 8, 2, 1024, 128, 4) == lib.ca_dcp_decode_workspace_size(
        2, 8, 2, 256, 128, 4, 16)
    assert lib.ca_ring_decode_workspace_size(2, 8, 2, 1022, 128, 4) == 0

    assert S[lib.ca_layout_to_shards(FAKE, FAKE, 2, 100, 256, 8, 0, None)] == "CA_ERR_SHAPE"
    assert S[lib.ca_layout_to_shards(FAKE, FAKE, 2, 64, 100, 8, 0, None)] == "CA_ERR_UNSUPPORTED"
    assert S[lib.ca_dcp_shard_kv(FAKE, FAKE, 2, 100, 256, 4, 16, None)] == "CA_ERR_SHAPE"


def test_paged_decode_validation(ca):
    """Host checks of the paged decode, none of which reaches the GPU: the
    caches' rows and the slots the block tables address must each stay
    below 2^31 (the kernel walks its work in 32-bit integers)."""
    lib = ca._load()
    S = ca.STATUS

    def pdec(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, dtype=1, N=2, Hq=8, Hkv=2, nblk=64, bs=16, mb=32, D=128, W=4,
                 I=16, seq=FAKE, scale=0.0, o=FAKE, lse=FAKE, ws=FAKE, ws_bytes=1 << 30, stream=None)
        a.update(kw)
        return S[lib.ca_dcp_decode_paged(a["q"], a["k"], a["v"], a["bt"], a["dtype"], a["N"], a["Hq"], a["Hkv"],
                                         a["nblk"], a["bs"], a["mb"], a["D"], a["W"], a["I"], a["seq"], a["scale"],
                                         a["o"], a["lse"], a["ws"], a["ws_bytes"], a["stream"])]

    assert pdec(seq=None) == "CA_ERR_INVALID_ARG"       # lengths are required
    assert pdec(bt=None) == "CA_ERR_INVALID_ARG"
    assert pdec(Hq=6, Hkv=4) == "CA_ERR_SHAPE"
    assert pdec(bs=24) == "CA_ERR_UNSUPPORTED"
    assert pdec(D=64) == "CA_ERR_UNSUPPORTED"
    assert pdec(nblk=1 << 26) == "CA_ERR_UNSUPPORTED"   # 4 * 2^26 * 2 * 16 cache rows
    assert pdec(N=1 << 12, mb=1 << 12) == "CA_ERR_UNSUPPORTED"  # 4 * 2^12 * 2 * 2^12 * 16 addressed slots
    # 2^30 addressed slots pass the size checks; the 16-byte workspace then
    # stops the call before anything is launched
    assert pdec(N=1 << 11, mb=1 << 12, ws_bytes=16) == "CA_ERR_WORKSPACE"
    assert pdec(k=FAKE + 8) == "CA_ERR_ALIGNMENT"
    assert pdec(ws=None) == "CA_ERR_WORKSPACE"


def test_dcp_prefill_validation(ca):
    lib = ca._load()
    S = ca.STATUS

    def pre(**kw):
        a = dict(q=FAKE, kp=FAKE, vp=FAKE, kc=FAKE, vc=FAKE, dtype=1, Hq=8, Hkv=2, Sc=512, D=128, W=4, I=16,
                 P=1024, Lcap=256, Lc=128, scale=0.0, o=FAKE, lse=None, stream=None)
        a.update(kw)
        return lib.ca_dcp_prefill(a["q"], a["kp"], a["vp"], a["kc"], a["vc"], a["dtype"], a["Hq"], a["Hkv"], a["Sc"],
                                  a["D"], a["W"], a["I"], a["P"], a["Lcap"], a["Lc"], a["scale"], a["o"], a["lse"],
                                  a["stream"])

    assert S[pre(q=None)] == "CA_ERR_INVALID_ARG"
    assert S[pre(P=-1)] == "CA_ERR_INVALID_ARG"
    assert S[pre(Hq=6, Hkv=4)] == "CA_ERR_SHAPE"
    assert S[pre(Lcap=255)] == "CA_ERR_SHAPE"   # rank 0 holds 256 of 1024 prior tokens
    assert S[pre(Lc=127)] == "CA_ERR_SHAPE"     # and 128 of the 512-token chunk
    assert S[pre(W=9)] == "CA_ERR_UNSUPPORTED"
    assert S[pre(dtype=0)] == "CA_ERR_UNSUPPORTED"
    assert S[pre(kc=FAKE + 8)] == "CA_ERR_ALIGNMENT"
    assert S[lib.ca_dcp_prefill_partial(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 512, 128, 4, 16, 1024, 256, 128, 4,
                                        0.0, FAKE, FAKE, None)] == "CA_ERR_INVALID_ARG"  # rank out of range


def test_qkv_prologue_validation(ca):
    lib = ca._load()
    S = ca.STATUS

    def pro(**kw):
        a = dict(xq=FAKE, xk=FAKE, xv=None, gq=None, gk=None, eps=1e-6, cs=None, sn=None, dtype=1, B=1, S=64,
                 Hq=8, Hkv=2, D=128, cp=4, layout=0, q=FAKE, k=FAKE, v=None, km=None)
        a.update(kw)
        return lib.ca_qkv_prologue(a["xq"], a["xk"], a["xv"], a["gq"], a["gk"], a["eps"], a["cs"], a["sn"],
                                   a["dtype"], a["B"], a["S"], a["Hq"], a["Hkv"], a["D"], a["cp"], a["layout"],
                                   a["q"], a["k"], a["v"], a["km"], None)

    assert S[pro(xq=None)] == "CA_ERR_INVALID_ARG"
    assert S[pro(xv=FAKE)] == "CA_ERR_INVALID_ARG"          # x_v without v
    assert S[pro(cs=FAKE)] == "CA_ERR_INVALID_ARG"          # cos without sin
    assert S[pro(eps=-1.0)] == "CA_ERR_INVALID_ARG"
    assert S[pro(layout=5)] == "CA_ERR_INVALID_ARG"
    assert S[pro(Hq=6, Hkv=4)] == "CA_ERR_SHAPE"
    assert S[pro(S=66)] == "CA_ERR_SHAPE"                   # S % cp
    assert S[pro(dtype=0)] == "CA_ERR_UNSUPPORTED"
    assert S[pro(D=96)] == "CA_ERR_UNSUPPORTED"
    assert S[pro(Hq=128, Hkv=2)] == "CA_ERR_UNSUPPORTED"    # hidden wider than 8192
    assert S[pro(S=1 << 30, cp=1)] == "CA_ERR_UNSUPPORTED"  # rows past 32-bit indices
    assert S[pro(k=FAKE + 8)] == "CA_ERR_ALIGNMENT"
    assert S[pro(km=FAKE + 2)] == "CA_ERR_ALIGNMENT"


def test_empty_problems(ca):
    """A problem with no rows, heads or sequences is an invalid argument
    (nothing is enqueued); the one exception is the paged cache write, for
    which zero new tokens is a valid no-op that touches no device."""
    lib = ca._load()
    S = ca.STATUS
    for kw in (dict(S=0), dict(B=0), dict(Hq=0), dict(Hkv=0), dict(D=0)):
        assert S[ring(lib, **kw)] == "CA_ERR_INVALID_ARG", kw
    assert S[lib.ca_dcp_decode(FAKE, FAKE, FAKE, 1, 0, 8, 2, 256, 128, 4, 16, None, 0.0, FAKE, None, FAKE,
                               1 << 30, None)] == "CA_ERR_INVALID_ARG"
    assert S[lib.ca_ring_decode(FAKE, FAKE, FAKE, 1, 0, 8, 2, 1024, 128, 4, 0, None, 0.0, FAKE, None, FAKE,
                                1 << 30, None)] == "CA_ERR_INVALID_ARG"
    assert S[lib.ca_qkv_prologue(FAKE, FAKE, None, None, None, 1e-6, None, None, 1, 1, 0, 8, 2, 128, 4, 0,
                                 FAKE, FAKE, None, None, None)] == "CA_ERR_INVALID_ARG"
    assert S[lib.ca_key_max2(FAKE, 1, 1, 2, 0, 128, FAKE, None)] == "CA_ERR_INVALID_ARG"
    assert S[lib.ca_paged_kv_write(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 2, 128, 4, 64, 16, None)] == "CA_OK"


def test_selftest_wait_timeout_validation(ca):
    lib = ca._load()
    S = ca.STATUS
    assert S[lib.ca_selftest_wait_timeout(0, None)] == "CA_ERR_INVALID_ARG"
    assert S[lib.ca_selftest_wait_timeout(5_000_000_000, None)] == "CA_ERR_INVALID_ARG"  # above the kernels' limit


def test_no_cpu_fallback(ca):
    """Host tensors are refused before anything runs: the product path has no
    CPU implementation to fall back on."""
    import torch

    q = torch.zeros(1, 2, 256, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ca.ring_attn_fwd(q, q, q, 2)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ca.dcp_decode(torch.zeros(1, 2, 128, dtype=torch.bfloat16), torch.zeros(2, 1, 2, 64, 128, dtype=torch.bfloat16),
                      torch.zeros(2, 1, 2, 64, 128, dtype=torch.bfloat16), 16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ca.ring_decode(torch.zeros(1, 2, 128, dtype=torch.bfloat16), q, q, 2)


def test_missing_library_fails_loudly(ca, monkeypatch):
    """Without the built library the binding raises instead of computing
    anything another way."""
    monkeypatch.setattr(ca, "_lib", None)
    monkeypatch.setattr(ca, "_LIB_PATH", "/nonexistent/libctxattn.so")
    with pytest.raises(ca.CtxAttnError):
        ca._load()


def test_noalloc_decode_checks_match_the_regular_decode(ca):
    """The allocation-free decode applies ca_dcp_decode's argument checks
    first and in the same order, so a problem too large for its 16 MiB
    scratch still reports whatever else is wrong with it; only a well-formed
    problem that does not fit gets CA_ERR_WORKSPACE (where the regular call,
    given room, would go ahead)."""
    lib = ca._load()
    S = ca.STATUS

    def both(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=1, N=64, Hq=32, Hkv=8, Lloc=32768, D=128, W=4, I=16, seq=None,
                 scale=0.0, o=FAKE, lse=FAKE)
        a.update(kw)
        args = (a["q"], a["k"], a["v"], a["dtype"], a["N"], a["Hq"], a["Hkv"], a["Lloc"], a["D"], a["W"], a["I"],
                a["seq"], a["scale"], a["o"], a["lse"])
        return S[lib.ca_dcp_decode(*args, None, 0, None)], S[lib.ca_dcp_decode_noalloc(*args, None)]

    # partials of 64 sequences x 32 heads over 4 shards of 32768 slots: ~34 MB
    assert lib.ca_dcp_decode_workspace_size(64, 32, 8, 32768, 128, 4, 16) > (16 << 20)
    for kw, want in ((dict(q=None), "CA_ERR_INVALID_ARG"), (dict(N=0), "CA_ERR_INVALID_ARG"),
                     (dict(Hq=30), "CA_ERR_SHAPE"), (dict(Lloc=32760), "CA_ERR_SHAPE"),
                     (dict(dtype=0), "CA_ERR_UNSUPPORTED"), (dict(D=64), "CA_ERR_UNSUPPORTED"),
                     (dict(Hq=72, Hkv=8), "CA_ERR_UNSUPPORTED"), (dict(k=FAKE + 8), "CA_ERR_ALIGNMENT"),
                     (dict(lse=FAKE + 2), "CA_ERR_ALIGNMENT")):
        assert both(**kw) == (want, want), kw
    # well formed: the regular call wants its workspace, the other has no room
    assert both() == ("CA_ERR_WORKSPACE", "CA_ERR_WORKSPACE")
