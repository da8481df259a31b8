"""fp64 CPU oracle for context-parallel attention (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA library in ``context_attention_gb300``
and never imports it; the CUDA library never imports this package.

Every routine here is a thin marshalling layer over the C functions in
``oracle.c`` (which cite the passages they follow).  Inputs are numpy arrays
whose values are the exact stored inputs (bf16 widened to fp32 is exact);
results are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

LAYOUT_CONTIGUOUS = 0
LAYOUT_STRIPED = 1
MODE_ONLINE_MAX = 0
MODE_CONST_MAX = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            Dbl = ctypes.c_double
            lib.ora_global_pos.argtypes = [I, I, I64, I64]
            lib.ora_global_pos.restype = I64
            lib.ora_attention_rows.argtypes = [P, P, P, I, I, I, I64, I, Dbl, I, I, I, P, I64, P, P]
            lib.ora_shard_partial_rows.argtypes = [P, P, P, I, I, I, I64, I, Dbl, I, I, I, I, P, I64, P, P]
            lib.ora_lse_merge.argtypes = [P, P, I, I64, I, P, P]
            lib.ora_const_max_bound.argtypes = [P, P, I, I, I, I64, I, Dbl, P, P]
            lib.ora_ring_rows.argtypes = [P, P, P, I, I, I, I64, I, Dbl, I, I, I, I, P, P, I64, P, P, P]
            lib.ora_dcp_deal.argtypes = [I64, I, I, P, P]
            lib.ora_qk_prologue.argtypes = [P, P, Dbl, P, P, I, I64, I, I, I, I, I, P]
            lib.ora_dcp_local_filled.argtypes = [I64, I, I, I]
            lib.ora_dcp_local_filled.restype = I64
            lib.ora_dcp_decode.argtypes = [P, P, P, I, I, I, I64, I, I, I, P, Dbl, P, P]
            lib.ora_dcp_prefill.argtypes = [P, P, P, P, P, I, I, I64, I, I, I, I64, I64, I64, Dbl, I, P, I64, P, P]
            lib.ora_ring_decode.argtypes = [P, P, P, I, I, I, I64, I, I, I, P, Dbl, P, P]
            lib.ora_dcp_decode_paged.argtypes = [P, P, P, P, I, I, I, I64, I, I64, I, I, I, P, Dbl, P, P]
            lib.ora_num_threads.restype = I
            _lib = lib
    return _lib


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return _load().ora_num_threads()


def _geometry(q, k):
    B, Hq, S, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    assert (B, S, D) == (Bk, Sk, Dk) and Hq % Hkv == 0
    return B, Hq, Hkv, S, D


def _rows(rows, B, Hq, S):
    if rows is None:
        return np.arange(B * Hq * S, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


def global_pos(layout: int, cp: int, Ls: int, rho: int) -> int:
    """Global token position of stored row ``rho`` (shard-major storage)."""
    return int(_load().ora_global_pos(layout, cp, Ls, rho))


def attention(q, k, v, scale=None, causal=False, layout=LAYOUT_CONTIGUOUS, cp=1, rows=None):
    """Full softmax attention (the authority).  Returns (o [n, D], lse [n]).

    ``rows`` selects flat row ids (b*Hq + h)*S + rho; default all rows."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, Hkv, S, D = _geometry(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    r = _rows(rows, B, Hq, S)
    o = np.zeros((len(r), D))
    lse = np.zeros(len(r))
    _load().ora_attention_rows(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, S, D, scale,
                               int(causal), layout, cp, _ptr(r), len(r), _ptr(o), _ptr(lse))
    return o, lse


def shard_partial(q, k, v, kv_shard, cp, scale=None, causal=False,
                  layout=LAYOUT_CONTIGUOUS, rows=None):
    """Partial attention against one virtual K/V shard.  Returns (o, lse)."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, Hkv, S, D = _geometry(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    r = _rows(rows, B, Hq, S)
    o = np.zeros((len(r), D))
    lse = np.zeros(len(r))
    _load().ora_shard_partial_rows(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, S, D, scale,
                                   int(causal), layout, cp, int(kv_shard), _ptr(r), len(r),
                                   _ptr(o), _ptr(lse))
    return o, lse


def lse_merge(o_parts, lse_parts):
    """LSE merge of partials o_parts [n, rows, D], lse_parts [n, rows]."""
    o_parts = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    lse_parts = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    n, R, D = o_parts.shape
    o = np.zeros((R, D))
    lse = np.zeros(R)
    _load().ora_lse_merge(_ptr(o_parts), _ptr(lse_parts), n, R, D, _ptr(o), _ptr(lse))
    return o, lse


def const_max_bound(q, k, scale=None):
    """Per-row Cauchy-Schwarz bound.  Returns (c [B,Hq,S], kmax2 [B,Hkv])."""
    q, k = _f32(q), _f32(k)
    B, Hq, Hkv, S, D = _geometry(q, k)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    c = np.zeros((B, Hq, S))
    kmax2 = np.zeros((B, Hkv))
    _load().ora_const_max_bound(_ptr(q), _ptr(k), B, Hq, Hkv, S, D, scale, _ptr(c), _ptr(kmax2))
    return c, kmax2


def ring(q, k, v, cp, mode=MODE_ONLINE_MAX, scale=None, causal=False,
         layout=LAYOUT_CONTIGUOUS, rows=None, c=None):
    """Ring attention step by step.  Returns (o, lse, overshoot).

    In const-max mode the bound c defaults to ``const_max_bound(q, k)``."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, Hq, Hkv, S, D = _geometry(q, k)
    assert S % cp == 0
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    r = _rows(rows, B, Hq, S)
    if mode == MODE_CONST_MAX and c is None:
        c, _ = const_max_bound(q, k, scale)
    cc = None if c is None else np.ascontiguousarray(np.asarray(c, dtype=np.float64))
    o = np.zeros((len(r), D))
    lse = np.zeros(len(r))
    ov = np.zeros(len(r))
    _load().ora_ring_rows(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, S, D, scale, int(causal),
                          layout, cp, mode, None if cc is None else _ptr(cc), _ptr(r), len(r),
                          _ptr(o), _ptr(lse), _ptr(ov))
    return o, lse, ov


def dcp_deal(n: int, W: int, I: int):
    """Owner rank and local index of global positions 0..n-1, by dealing."""
    own = np.zeros(max(n, 1), dtype=np.int32)
    loc = np.zeros(max(n, 1), dtype=np.int64)
    _load().ora_dcp_deal(n, W, I, _ptr(own), _ptr(loc))
    return own[:n], loc[:n]


def dcp_local_filled(N: int, W: int, I: int, R: int) -> int:
    """Tokens among positions 0..N-1 held by rank R, by dealing."""
    return int(_load().ora_dcp_local_filled(N, W, I, R))


def dcp_decode(q, k_shards, v_shards, interleave, seq_lens=None, scale=None):
    """DCP decode.  q [N,Hq,D]; k/v shards [W,N,Hkv,Lloc,D].  Returns (o, lse)."""
    q = _f32(q)
    k_shards, v_shards = _f32(k_shards), _f32(v_shards)
    N, Hq, D = q.shape
    W, Nk, Hkv, Lloc, Dk = k_shards.shape
    assert Nk == N and Dk == D and Hq % Hkv == 0
    if seq_lens is None:
        seq_lens = np.full(N, W * Lloc, dtype=np.int64)
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int64))
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.zeros((N, Hq, D))
    lse = np.zeros((N, Hq))
    _load().ora_dcp_decode(_ptr(q), _ptr(k_shards), _ptr(v_shards), N, Hq, Hkv, Lloc, D, W,
                           int(interleave), _ptr(sl), scale, _ptr(o), _ptr(lse))
    return o, lse


def ring_decode(q, k, v, cp, layout=LAYOUT_CONTIGUOUS, seq_lens=None, scale=None):
    """Ring Pass-Q decode over the ring layout's cache.  q [B,Hq,D]; k/v
    [B,Hkv,S,D] shard-major; seq_lens [B] (default S).  Returns (o, lse)."""
    q = _f32(q)
    k, v = _f32(k), _f32(v)
    B, Hq, D = q.shape
    Bk, Hkv, S, Dk = k.shape
    assert Bk == B and Dk == D and Hq % Hkv == 0 and S % cp == 0
    if seq_lens is None:
        seq_lens = np.full(B, S, dtype=np.int64)
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int64))
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    _load().ora_ring_decode(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, S, D, int(cp), int(layout), _ptr(sl), scale,
                            _ptr(o), _ptr(lse))
    return o, lse


def dcp_prefill(q, k_prior, v_prior, k_cur, v_cur, interleave, prior_tokens, scale=None, part_rank=-1,
                rows=None):
    """DCP prefill of one chunk.  q [Hq,Sc,D]; prior shards [W,Hkv,Lcap,D];
    current shards [W,Hkv,Lc,D].  Returns (o [Hq,Sc,D], lse [Hq,Sc]); with
    part_rank >= 0 returns that rank's partial instead of the merge.  With
    ``rows`` (flat ids h*Sc + i) returns only those rows: (o [n,D], lse [n])."""
    q = _f32(q)
    k_prior, v_prior, k_cur, v_cur = _f32(k_prior), _f32(v_prior), _f32(k_cur), _f32(v_cur)
    Hq, Sc, D = q.shape
    W, Hkv, Lcap, _ = k_prior.shape
    Lc = k_cur.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    r = np.arange(Hq * Sc, dtype=np.int64) if rows is None else np.ascontiguousarray(np.asarray(rows, np.int64))
    o = np.zeros((len(r), D))
    lse = np.zeros(len(r))
    _load().ora_dcp_prefill(_ptr(q), _ptr(k_prior), _ptr(v_prior), _ptr(k_cur), _ptr(v_cur), Hq, Hkv, Sc, D,
                            W, int(interleave), int(prior_tokens), Lcap, Lc, scale, int(part_rank), _ptr(r), len(r),
                            _ptr(o), _ptr(lse))
    if rows is None:
        return o.reshape(Hq, Sc, D), lse.reshape(Hq, Sc)
    return o, lse


def dcp_decode_paged(q, k_cache, v_cache, block_tables, interleave, seq_lens, scale=None):
    """DCP decode over paged caches.  q [N,Hq,D]; k/v cache [W,nblk,Hkv,bs,D];
    block_tables [W,N,max_blocks] int32; seq_lens [N].  Returns (o, lse)."""
    q = _f32(q)
    k_cache, v_cache = _f32(k_cache), _f32(v_cache)
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    N, Hq, D = q.shape
    W, nblk, Hkv, bs, _ = k_cache.shape
    max_blocks = bt.shape[2]
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int64))
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.zeros((N, Hq, D))
    lse = np.zeros((N, Hq))
    _load().ora_dcp_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), N, Hq, Hkv, nblk, bs, max_blocks,
                                 D, W, int(interleave), _ptr(sl), scale, _ptr(o), _ptr(lse))
    return o, lse


def qk_prologue(x, H, g=None, eps=1e-6, cos=None, sin=None, cp=1, layout=LAYOUT_CONTIGUOUS, norm=True):
    """Attention input [B,H,S,D] (fp64) of one projected tensor x [B,S,H*D]:
    whole-hidden RMS norm with gain g (norm=True), rotary turn of channel
    pairs by the per-position tables cos/sin [S, D/2] (if given), rows in the
    shard-major order of the layout."""
    x = _f32(x)
    B, S, HD = x.shape
    D = HD // H
    assert H * D == HD and D % 2 == 0 and S % cp == 0
    gp = None if g is None else _f32(g)
    cs = None if cos is None else _f32(cos)
    sn = None if sin is None else _f32(sin)
    out = np.zeros((B, H, S, D))
    _load().ora_qk_prologue(_ptr(x), _ptr(gp), float(eps), _ptr(cs), _ptr(sn), B, S, H, D, cp, int(layout),
                            1 if norm else 0, _ptr(out))
    return out
