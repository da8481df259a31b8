"""context_attention_gb300 -- GB300-native hot path of context-parallel attention.

A thin ctypes binding over ``libctxattn.so`` (the C ABI in include/ctxattn.h).
Every function here only checks tensors, allocates outputs and workspaces with
PyTorch (device memory and streams are PyTorch's job) and passes raw pointers
plus the current CUDA stream to the library; every step of the computation runs
in the library's CUDA kernels.  There is no CPU fallback: if the library is
missing or a call fails, a ``CtxAttnError`` is raised.

Python names mirror the C entry points without the ``ca_`` prefix.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "CtxAttnError", "build", "library_path",
    "ring_attn_fwd", "ring_attn_fwd_bounded", "ring_attn_fwd_kmax", "attn_partial_step", "lse_merge",
    "qkv_prologue", "key_max2", "const_max_bound",
    "ring_decode", "dcp_decode", "dcp_decode_noalloc", "dcp_decode_paged", "paged_kv_write", "dcp_prefill", "dcp_prefill_partial",
    "layout_to_shards", "layout_from_shards", "dcp_shard_kv",
    "layout_global_index", "layout_shard_row", "ring_kv_shard", "dcp_owner", "dcp_local_index",
    "dcp_local_to_global", "dcp_local_filled", "dcp_active_mask", "dcp_slot_mapping",
    "device_status", "selftest_wait_timeout",
    "ring_attn_fwd_workspace_size", "dcp_decode_workspace_size", "ring_decode_workspace_size",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libctxattn.so")
_lock = threading.Lock()
_lib = None

CA_OK = 0
STATUS = {0: "CA_OK", 1: "CA_ERR_INVALID_ARG", 2: "CA_ERR_SHAPE", 3: "CA_ERR_UNSUPPORTED",
          4: "CA_ERR_ALIGNMENT", 5: "CA_ERR_WORKSPACE", 6: "CA_ERR_CUDA", 7: "CA_ERR_TIMEOUT"}
DTYPE = {torch.float32: 0, torch.bfloat16: 1}
MODE = {"online_max": 0, "const_max": 1}
LAYOUT = {"contiguous": 0, "striped": 1}


class CtxAttnError(RuntimeError):
    """A libctxattn call returned an error status."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


def library_path() -> str:
    """Path of the in-tree libctxattn.so the binding loads."""
    return _LIB_PATH


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libctxattn.so in-tree for sm_103a (see _build.py)."""
    from . import _build

    return _build.build(force=force, verbose=verbose)


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise CtxAttnError("load libctxattn.so (not built: run context_attention_gb300.build())", 6)
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        sig = {
            "ca_status_string": ([I], ctypes.c_char_p),
            "ca_version": ([], I),
            "ca_ring_attn_fwd_workspace_size": ([I, I, I, I64, I, I, I], SZ),
            "ca_ring_attn_fwd": ([P, P, P, P, P, I, I, I, I, I64, I, I, I, I, I, F, P, SZ, P], I),
            "ca_ring_attn_fwd_bounded": ([P, P, P, P, P, P, I, I, I, I, I64, I, I, I, I, F, P], I),
            "ca_ring_attn_fwd_kmax": ([P, P, P, P, P, P, I, I, I, I, I64, I, I, I, I, F, P], I),
            "ca_key_max2": ([P, I, I, I, I64, I, P, P], I),
            "ca_qkv_prologue": ([P, P, P, P, P, F, P, P, I, I, I64, I, I, I, I, I, P, P, P, P, P], I),
            "ca_attn_partial_step": ([P, P, P, I, I, I, I, I64, I, I, I, I, I, I, I, F, P, P, P, P], I),
            "ca_lse_merge": ([P, P, I, I64, I, P, P, I, P, P], I),
            "ca_const_max_bound": ([P, P, I, I, I, I, I64, I, F, P, P, P], I),
            "ca_dcp_decode_workspace_size": ([I, I, I, I64, I, I, I], SZ),
            "ca_dcp_decode": ([P, P, P, I, I, I, I, I64, I, I, I, P, F, P, P, P, SZ, P], I),
            "ca_dcp_decode_noalloc": ([P, P, P, I, I, I, I, I64, I, I, I, P, F, P, P, P], I),
            "ca_ring_decode_workspace_size": ([I, I, I, I64, I, I], SZ),
            "ca_ring_decode": ([P, P, P, I, I, I, I, I64, I, I, I, P, F, P, P, P, SZ, P], I),
            "ca_dcp_decode_paged": ([P, P, P, P, I, I, I, I, I64, I, I64, I, I, I, P, F, P, P, P, SZ, P], I),
            "ca_paged_kv_write": ([P, P, P, P, P, I, I, I, I, I, I64, I, P], I),
            "ca_dcp_prefill": ([P, P, P, P, P, I, I, I, I64, I, I, I, I64, I64, I64, F, P, P, P], I),
            "ca_dcp_prefill_partial": ([P, P, P, P, P, I, I, I, I64, I, I, I, I64, I64, I64, I, F, P, P, P], I),
            "ca_layout_to_shards": ([P, P, I64, I64, I64, I, I, P], I),
            "ca_layout_from_shards": ([P, P, I64, I64, I64, I, I, P], I),
            "ca_dcp_shard_kv": ([P, P, I64, I64, I64, I, I, P], I),
            "ca_layout_global_index": ([I, I, I64, I64], I64),
            "ca_layout_shard_row": ([I, I, I64, I64], I64),
            "ca_ring_kv_shard": ([I, I, I], I),
            "ca_dcp_owner": ([I64, I, I], I),
            "ca_dcp_local_index": ([I64, I, I], I64),
            "ca_dcp_local_to_global": ([I64, I, I, I], I64),
            "ca_dcp_local_filled": ([I64, I, I, I, I], I64),
            "ca_dcp_active_mask": ([I64, I, I, I, I], I),
            "ca_dcp_slot_mapping": ([P, I64, P, I64, I, I, I, I, P], I),
            "ca_device_status": ([I], I),
            "ca_selftest_wait_timeout": ([ctypes.c_longlong, P], I),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != CA_OK:
        raise CtxAttnError(fn, status)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


FLOATS = tuple(DTYPE)


def _dims(t, name: str, ndim: int):
    """Shape of the tensor that fixes a call's problem sizes."""
    if not isinstance(t, torch.Tensor) or t.dim() != ndim:
        raise ValueError(f"{name} must be a {ndim}-d tensor")
    return tuple(t.shape)


def _args(*specs):
    """Check every tensor of one call before anything is launched.

    A spec is (tensor or None, name, shape, dtypes).  shape is a tuple whose
    None entries match any size, an int (that many elements, any shape) or
    None (unchecked); dtypes is one dtype, a tuple of them or None (any).  A
    None tensor is an optional operand left out and is skipped.  First the shapes and
    dtypes (the kernels read and write exactly the extents the sizes passed
    to the library give, so a mismatch would run past a buffer), then that
    all of them are contiguous CUDA tensors on one device."""
    given = [s for s in specs if s[0] is not None]
    for t, name, shape, dtypes in given:
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{name} must be a torch.Tensor")
        if isinstance(shape, int):
            if t.numel() != shape:
                raise ValueError(f"{name}: {t.numel()} elements, expected {shape}")
        elif shape is not None:
            if t.dim() != len(shape) or any(e is not None and e != n for e, n in zip(shape, t.shape)):
                want = "[" + ", ".join("*" if e is None else str(e) for e in shape) + "]"
                raise ValueError(f"{name}: shape {list(t.shape)}, expected {want}")
        dts = () if dtypes is None else dtypes if isinstance(dtypes, tuple) else (dtypes,)
        if dts and t.dtype not in dts:
            raise ValueError(f"{name}: dtype {t.dtype}, expected {' or '.join(str(d) for d in dts)}")
    dev = None
    for t, name, _, _ in given:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other operands on {dev}")


def _ws_bytes(workspace) -> int:
    return 0 if workspace is None else workspace.numel() * workspace.element_size()


def ring_attn_fwd_workspace_size(B, Hq, Hkv, S, D, cp_size, mode="online_max") -> int:
    """Workspace bytes ring_attn_fwd needs (const max: the key maximum kmax2; online max: 0)."""
    return int(_load().ca_ring_attn_fwd_workspace_size(B, Hq, Hkv, S, D, cp_size, MODE[mode]))


def ring_attn_fwd(q, k, v, cp_size, mode="online_max", causal=False, layout="contiguous",
                  softmax_scale=None, out=None, lse=None, return_lse=True, workspace=None):
    """Ring attention forward over cp_size virtual shards (shard-major rows).

    q [B,Hq,S,D], k/v [B,Hkv,S,D] (bf16 with D=128, or fp32 with D<=128).
    Returns (o, lse) with o [B,Hq,S,D] in q's dtype and lse [B,Hq,S] fp32."""
    lib = _load()
    B, Hq, S, D = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    _args((q, "q", None, FLOATS), (k, "k", (B, Hkv, S, D), q.dtype), (v, "v", (B, Hkv, S, D), q.dtype),
          (out, "out", (B, Hq, S, D), q.dtype), (lse if return_lse else None, "lse", (B, Hq, S), torch.float32),
          (workspace, "workspace", None, None))
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty(B, Hq, S, device=q.device, dtype=torch.float32)
    ws_bytes = int(lib.ca_ring_attn_fwd_workspace_size(B, Hq, Hkv, S, D, cp_size, MODE[mode]))
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, device=q.device, dtype=torch.uint8)
    st = lib.ca_ring_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse if return_lse else None),
                              DTYPE[q.dtype], B, Hq, Hkv, S, D, cp_size, MODE[mode], int(bool(causal)),
                              LAYOUT[layout], float(softmax_scale or 0.0),
                              _ptr(workspace) if ws_bytes else None,
                              _ws_bytes(workspace) if ws_bytes else 0, _stream(q))
    _check("ca_ring_attn_fwd", st)
    return out, (lse if return_lse else None)


def ring_attn_fwd_bounded(q, k, v, c, cp_size, causal=False, layout="contiguous", softmax_scale=None,
                          out=None, lse=None, return_lse=True):
    """Const-max ring attention with a caller-provided bound c [B,Hq,S] fp32."""
    lib = _load()
    B, Hq, S, D = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    c = c.contiguous() if isinstance(c, torch.Tensor) else c
    _args((q, "q", None, FLOATS), (k, "k", (B, Hkv, S, D), q.dtype), (v, "v", (B, Hkv, S, D), q.dtype),
          (c, "c", (B, Hq, S), torch.float32), (out, "out", (B, Hq, S, D), q.dtype),
          (lse if return_lse else None, "lse", (B, Hq, S), torch.float32))
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty(B, Hq, S, device=q.device, dtype=torch.float32)
    st = lib.ca_ring_attn_fwd_bounded(_ptr(q), _ptr(k), _ptr(v), _ptr(c), _ptr(out),
                                      _ptr(lse if return_lse else None), DTYPE[q.dtype], B, Hq, Hkv, S, D,
                                      cp_size, int(bool(causal)), LAYOUT[layout], float(softmax_scale or 0.0),
                                      _stream(q))
    _check("ca_ring_attn_fwd_bounded", st)
    return out, (lse if return_lse else None)


def ring_attn_fwd_kmax(q, k, v, kmax2, cp_size, causal=False, layout="contiguous", softmax_scale=None,
                       out=None, lse=None, return_lse=True):
    """Const-max ring attention with a caller-provided key maximum kmax2
    [B,Hkv] fp32 (max |k_j|^2 per head, e.g. from key_max2, or its max over
    processes); each row's bound is formed in the kernel."""
    lib = _load()
    B, Hq, S, D = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    kmax2 = kmax2.contiguous() if isinstance(kmax2, torch.Tensor) else kmax2
    _args((q, "q", None, FLOATS), (k, "k", (B, Hkv, S, D), q.dtype), (v, "v", (B, Hkv, S, D), q.dtype),
          (kmax2, "kmax2", (B, Hkv), torch.float32), (out, "out", (B, Hq, S, D), q.dtype),
          (lse if return_lse else None, "lse", (B, Hq, S), torch.float32))
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty(B, Hq, S, device=q.device, dtype=torch.float32)
    st = lib.ca_ring_attn_fwd_kmax(_ptr(q), _ptr(k), _ptr(v), _ptr(kmax2), _ptr(out),
                                   _ptr(lse if return_lse else None), DTYPE[q.dtype], B, Hq, Hkv, S, D,
                                   cp_size, int(bool(causal)), LAYOUT[layout], float(softmax_scale or 0.0),
                                   _stream(q))
    _check("ca_ring_attn_fwd_kmax", st)
    return out, (lse if return_lse else None)


def attn_partial_step(q_shard, k_shard, v_shard, q_rank, kv_rank, cp_size, mode="online_max",
                      causal=False, layout="contiguous", softmax_scale=None, c=None):
    """One ring step: queries of shard q_rank against the K/V of shard kv_rank.

    Returns (o_part fp32, lse_part fp32).  In const-max mode pass the shard's
    rows of the bound c; o_part is then the unnormalised sum."""
    lib = _load()
    B, Hq, Ls, D = _dims(q_shard, "q_shard", 4)
    Hkv = _dims(k_shard, "k_shard", 4)[1]
    if isinstance(c, torch.Tensor):
        c = c.contiguous()
    _args((q_shard, "q_shard", None, FLOATS), (k_shard, "k_shard", (B, Hkv, Ls, D), q_shard.dtype),
          (v_shard, "v_shard", (B, Hkv, Ls, D), q_shard.dtype), (c, "c", (B, Hq, Ls), torch.float32))
    o = torch.empty(B, Hq, Ls, D, device=q_shard.device, dtype=torch.float32)
    lse = torch.empty(B, Hq, Ls, device=q_shard.device, dtype=torch.float32)
    st = lib.ca_attn_partial_step(_ptr(q_shard), _ptr(k_shard), _ptr(v_shard), DTYPE[q_shard.dtype],
                                  B, Hq, Hkv, Ls, D, q_rank, kv_rank, cp_size, MODE[mode],
                                  int(bool(causal)), LAYOUT[layout], float(softmax_scale or 0.0),
                                  _ptr(c), _ptr(o), _ptr(lse), _stream(q_shard))
    _check("ca_attn_partial_step", st)
    return o, lse


def lse_merge(o_parts, lse_parts, c=None, out_dtype=torch.float32):
    """Merge n partials o_parts [n, ..., D], lse_parts [n, ...] (fp32)."""
    lib = _load()
    if not isinstance(o_parts, torch.Tensor) or o_parts.dim() < 2:
        raise ValueError("o_parts must be a tensor [n, ..., D]")
    if out_dtype not in DTYPE:
        raise ValueError(f"out_dtype {out_dtype} not supported (bf16 or fp32)")
    n, D = o_parts.shape[0], o_parts.shape[-1]
    R = o_parts[0].numel() // D if D else 0
    lse_parts = lse_parts.contiguous() if isinstance(lse_parts, torch.Tensor) else lse_parts
    c = c.contiguous() if isinstance(c, torch.Tensor) else c
    _args((o_parts, "o_parts", None, torch.float32), (lse_parts, "lse_parts", tuple(o_parts.shape[:-1]), torch.float32),
          (c, "c", R, torch.float32))
    o = torch.empty(o_parts.shape[1:], device=o_parts.device, dtype=out_dtype)
    lse = torch.empty(o_parts.shape[1:-1], device=o_parts.device, dtype=torch.float32)
    st = lib.ca_lse_merge(_ptr(o_parts), _ptr(lse_parts), n, R, D,
                          _ptr(c), _ptr(o), DTYPE[out_dtype],
                          _ptr(lse), _stream(o_parts))
    _check("ca_lse_merge", st)
    return o, lse


def qkv_prologue(x_q, x_k, Hq, Hkv, x_v=None, g_q=None, g_k=None, eps=1e-6, rope_cos=None, rope_sin=None,
                 cp_size=1, layout="contiguous", want_kmax2=True):
    """Attention inputs from projected activations x_q [B,S,Hq*D], x_k (and
    x_v) [B,S,Hkv*D] (bf16, token order): whole-hidden RMS norm with gains,
    rotary turn by per-position tables [S, D/2], heads split into [B,H,S,D]
    in the shard-major row order of the layout.  Returns (q, k, v or None,
    kmax2 [B,Hkv] or None)."""
    lib = _load()
    B, S, HqD = _dims(x_q, "x_q", 3)
    if Hq <= 0 or Hkv <= 0 or HqD % Hq:
        raise ValueError(f"x_q's last dimension {HqD} is not Hq={Hq} heads")
    D = HqD // Hq
    if (rope_cos is None) != (rope_sin is None):
        raise ValueError("rope_cos and rope_sin go together")
    _args((x_q, "x_q", None, FLOATS), (x_k, "x_k", (B, S, Hkv * D), x_q.dtype), (x_v, "x_v", (B, S, Hkv * D), x_q.dtype),
          (g_q, "g_q", Hq * D, torch.float32), (g_k, "g_k", Hkv * D, torch.float32),
          (rope_cos, "rope_cos", S * (D // 2), torch.float32), (rope_sin, "rope_sin", S * (D // 2), torch.float32))
    q = torch.empty(B, Hq, S, D, device=x_q.device, dtype=x_q.dtype)
    k = torch.empty(B, Hkv, S, D, device=x_q.device, dtype=x_q.dtype)
    v = None if x_v is None else torch.empty(B, Hkv, S, D, device=x_q.device, dtype=x_q.dtype)
    km = torch.empty(B, Hkv, device=x_q.device, dtype=torch.float32) if want_kmax2 else None
    st = lib.ca_qkv_prologue(_ptr(x_q), _ptr(x_k), _ptr(x_v), _ptr(g_q), _ptr(g_k), float(eps), _ptr(rope_cos),
                             _ptr(rope_sin), DTYPE[x_q.dtype], B, S, Hq, Hkv, D, cp_size, LAYOUT[layout], _ptr(q),
                             _ptr(k), _ptr(v), _ptr(km), _stream(x_q))
    _check("ca_qkv_prologue", st)
    return q, k, v, km


def key_max2(k, out=None):
    """kmax2 [B,Hkv] fp32: per head, the max over keys of |k_j|^2."""
    lib = _load()
    B, Hkv, S, D = _dims(k, "k", 4)
    _args((k, "k", None, FLOATS), (out, "out", (B, Hkv), torch.float32))
    if out is None:
        out = torch.empty(B, Hkv, device=k.device, dtype=torch.float32)
    st = lib.ca_key_max2(_ptr(k), DTYPE[k.dtype], B, Hkv, S, D, _ptr(out), _stream(k))
    _check("ca_key_max2", st)
    return out


def const_max_bound(q, k, softmax_scale=None):
    """Per-row const-max bound: returns (c [B,Hq,S] fp32, kmax2 [B,Hkv] fp32)."""
    lib = _load()
    B, Hq, S, D = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    _args((q, "q", None, FLOATS), (k, "k", (B, Hkv, S, D), q.dtype))
    c = torch.empty(B, Hq, S, device=q.device, dtype=torch.float32)
    kmax2 = torch.empty(B, Hkv, device=q.device, dtype=torch.float32)
    st = lib.ca_const_max_bound(_ptr(q), _ptr(k), DTYPE[q.dtype], B, Hq, Hkv, S, D,
                                float(softmax_scale or 0.0), _ptr(c), _ptr(kmax2), _stream(q))
    _check("ca_const_max_bound", st)
    return c, kmax2


def ring_decode_workspace_size(B, Hq, Hkv, S, D, cp_size):
    """Workspace bytes of ring_decode (its split-KV partials)."""
    return int(_load().ca_ring_decode_workspace_size(B, Hq, Hkv, S, D, cp_size))


def dcp_decode_workspace_size(N, Hq, Hkv, Lloc, D, dcp, interleave) -> int:
    """Workspace bytes of dcp_decode / dcp_decode_paged (its split-KV partials)."""
    return int(_load().ca_dcp_decode_workspace_size(N, Hq, Hkv, Lloc, D, dcp, interleave))


def dcp_decode(q, k_shards, v_shards, interleave, seq_lens=None, softmax_scale=None, out=None,
               lse=None, workspace=None):
    """DCP decode.  q [N,Hq,D]; k/v shards [dcp,N,Hkv,Lloc,D] (bf16, D=128).

    seq_lens: optional CUDA int32 [N].  Returns (o [N,Hq,D], lse [N,Hq])."""
    lib = _load()
    N, Hq, D = _dims(q, "q", 3)
    W, _, Hkv, Lloc, _ = _dims(k_shards, "k_shards", 5)
    _args((q, "q", None, FLOATS), (k_shards, "k_shards", (W, N, Hkv, Lloc, D), q.dtype),
          (v_shards, "v_shards", (W, N, Hkv, Lloc, D), q.dtype), (seq_lens, "seq_lens", (N,), torch.int32),
          (out, "out", (N, Hq, D), q.dtype), (lse, "lse", (N, Hq), torch.float32),
          (workspace, "workspace", None, None))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(N, Hq, device=q.device, dtype=torch.float32)
    ws_bytes = int(lib.ca_dcp_decode_workspace_size(N, Hq, Hkv, Lloc, D, W, interleave))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=q.device, dtype=torch.uint8)
    st = lib.ca_dcp_decode(_ptr(q), _ptr(k_shards), _ptr(v_shards), DTYPE[q.dtype], N, Hq, Hkv, Lloc,
                           D, W, interleave, _ptr(seq_lens), float(softmax_scale or 0.0), _ptr(out),
                           _ptr(lse), _ptr(workspace), _ws_bytes(workspace), _stream(q))
    _check("ca_dcp_decode", st)
    return out, lse


def ring_decode(q, k, v, cp_size, layout="contiguous", seq_lens=None, softmax_scale=None, out=None, lse=None,
                workspace=None):
    """Ring Pass-Q decode: one query token per sequence over the ring layout's
    KV cache.  q [B,Hq,D]; k/v [B,Hkv,S,D] shard-major (bf16, D=128).

    seq_lens: optional CUDA int32 [B] (cached tokens, default S).  Returns
    (o [B,Hq,D], lse [B,Hq])."""
    lib = _load()
    B, Hq, D = _dims(q, "q", 3)
    _, Hkv, S, _ = _dims(k, "k", 4)
    _args((q, "q", None, FLOATS), (k, "k", (B, Hkv, S, D), q.dtype), (v, "v", (B, Hkv, S, D), q.dtype),
          (seq_lens, "seq_lens", (B,), torch.int32), (out, "out", (B, Hq, D), q.dtype),
          (lse, "lse", (B, Hq), torch.float32), (workspace, "workspace", None, None))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, device=q.device, dtype=torch.float32)
    ws_bytes = int(lib.ca_ring_decode_workspace_size(B, Hq, Hkv, S, D, cp_size))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=q.device, dtype=torch.uint8)
    st = lib.ca_ring_decode(_ptr(q), _ptr(k), _ptr(v), DTYPE[q.dtype], B, Hq, Hkv, S, D, cp_size, LAYOUT[layout],
                            _ptr(seq_lens), float(softmax_scale or 0.0), _ptr(out), _ptr(lse), _ptr(workspace),
                            _ws_bytes(workspace), _stream(q))
    _check("ca_ring_decode", st)
    return out, lse


def dcp_decode_noalloc(q, k_shards, v_shards, interleave, seq_lens=None, softmax_scale=None, out=None,
                       lse=None):
    """DCP decode through the allocation-free entry point.

    For callers that cannot allocate device memory at call time (their
    framework's allocator owns all of it, or their enqueue path may not
    allocate): the library keeps the split-KV partials in a built-in 16 MiB
    scratch array instead of a workspace.  Pass ``out`` and ``lse`` to keep
    this call free of allocations on the Python side too.  Larger problems
    raise CtxAttnError (CA_ERR_WORKSPACE)."""
    lib = _load()
    N, Hq, D = _dims(q, "q", 3)
    W, _, Hkv, Lloc, _ = _dims(k_shards, "k_shards", 5)
    _args((q, "q", None, FLOATS), (k_shards, "k_shards", (W, N, Hkv, Lloc, D), q.dtype),
          (v_shards, "v_shards", (W, N, Hkv, Lloc, D), q.dtype), (seq_lens, "seq_lens", (N,), torch.int32),
          (out, "out", (N, Hq, D), q.dtype), (lse, "lse", (N, Hq), torch.float32))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(N, Hq, device=q.device, dtype=torch.float32)
    st = lib.ca_dcp_decode_noalloc(_ptr(q), _ptr(k_shards), _ptr(v_shards), DTYPE[q.dtype], N, Hq, Hkv, Lloc,
                                   D, W, interleave, _ptr(seq_lens), float(softmax_scale or 0.0), _ptr(out),
                                   _ptr(lse), _stream(q))
    _check("ca_dcp_decode_noalloc", st)
    return out, lse


def dcp_decode_paged(q, k_cache, v_cache, block_tables, interleave, seq_lens, softmax_scale=None, out=None,
                     lse=None, workspace=None):
    """DCP decode over paged caches.  q [N,Hq,D]; k/v cache [dcp,nblk,Hkv,bs,D];
    block_tables CUDA int32 [dcp,N,max_blocks]; seq_lens CUDA int32 [N]."""
    lib = _load()
    N, Hq, D = _dims(q, "q", 3)
    W, nblk, Hkv, bs, _ = _dims(k_cache, "k_cache", 5)
    max_blocks = _dims(block_tables, "block_tables", 3)[2]
    if seq_lens is None:
        raise ValueError("seq_lens is required for the paged cache")
    _args((q, "q", None, FLOATS), (k_cache, "k_cache", (W, nblk, Hkv, bs, D), q.dtype),
          (v_cache, "v_cache", (W, nblk, Hkv, bs, D), q.dtype),
          (block_tables, "block_tables", (W, N, max_blocks), torch.int32), (seq_lens, "seq_lens", (N,), torch.int32),
          (out, "out", (N, Hq, D), q.dtype), (lse, "lse", (N, Hq), torch.float32),
          (workspace, "workspace", None, None))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(N, Hq, device=q.device, dtype=torch.float32)
    ws_bytes = int(lib.ca_dcp_decode_workspace_size(N, Hq, Hkv, max_blocks * bs, D, W, interleave))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), device=q.device, dtype=torch.uint8)
    st = lib.ca_dcp_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), DTYPE[q.dtype], N, Hq,
                                 Hkv, nblk, bs, max_blocks, D, W, interleave, _ptr(seq_lens),
                                 float(softmax_scale or 0.0), _ptr(out), _ptr(lse), _ptr(workspace),
                                 _ws_bytes(workspace), _stream(q))
    _check("ca_dcp_decode_paged", st)
    return out, lse


def paged_kv_write(k_new, v_new, slots, k_cache, v_cache):
    """Write new tokens' K/V [T,Hkv,D] into the paged caches by slot mapping
    (slots: CUDA int64 [dcp, T], -1 = not owned)."""
    T, Hkv, D = _dims(k_new, "k_new", 3)
    W, nblk, _, bs, _ = _dims(k_cache, "k_cache", 5)
    _args((k_new, "k_new", None, FLOATS), (v_new, "v_new", (T, Hkv, D), k_new.dtype),
          (slots, "slots", (W, T), torch.int64), (k_cache, "k_cache", (W, nblk, Hkv, bs, D), k_new.dtype),
          (v_cache, "v_cache", (W, nblk, Hkv, bs, D), k_new.dtype))
    st = _load().ca_paged_kv_write(_ptr(k_new), _ptr(v_new), _ptr(slots), _ptr(k_cache), _ptr(v_cache),
                                   DTYPE[k_new.dtype], T, Hkv, D, W, nblk, bs, _stream(k_new))
    _check("ca_paged_kv_write", st)


def _prefill_dims(q, k_prior, v_prior, k_cur, v_cur, out=None, lse=None):
    """Sizes of a DCP prefill call, after checking its tensors."""
    Hq, Sc, D = _dims(q, "q", 3)
    W, Hkv, Lcap, _ = _dims(k_prior, "k_prior", 4)
    Lc = _dims(k_cur, "k_cur", 4)[2]
    _args((q, "q", None, FLOATS), (k_prior, "k_prior", (W, Hkv, Lcap, D), q.dtype),
          (v_prior, "v_prior", (W, Hkv, Lcap, D), q.dtype), (k_cur, "k_cur", (W, Hkv, Lc, D), q.dtype),
          (v_cur, "v_cur", (W, Hkv, Lc, D), q.dtype), (out, "out", (Hq, Sc, D), q.dtype),
          (lse, "lse", (Hq, Sc), torch.float32))
    return Hq, Sc, D, W, Hkv, Lcap, Lc


def dcp_prefill(q, k_prior, v_prior, k_cur, v_cur, interleave, prior_tokens, softmax_scale=None, out=None,
                lse=None):
    """DCP prefill of one chunk (online max).

    q [Hq,Sc,D]; prior shards [dcp,Hkv,Lcap,D]; current shards [dcp,Hkv,Lc,D]
    (bf16, D=128).  Returns (o [Hq,Sc,D] bf16, lse [Hq,Sc])."""
    lib = _load()
    Hq, Sc, D, W, Hkv, Lcap, Lc = _prefill_dims(q, k_prior, v_prior, k_cur, v_cur, out, lse)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, Sc, device=q.device, dtype=torch.float32)
    st = lib.ca_dcp_prefill(_ptr(q), _ptr(k_prior), _ptr(v_prior), _ptr(k_cur), _ptr(v_cur), DTYPE[q.dtype], Hq,
                            Hkv, Sc, D, W, interleave, int(prior_tokens), Lcap, Lc, float(softmax_scale or 0.0),
                            _ptr(out), _ptr(lse), _stream(q))
    _check("ca_dcp_prefill", st)
    return out, lse


def dcp_prefill_partial(q, k_prior, v_prior, k_cur, v_cur, interleave, prior_tokens, rank, softmax_scale=None):
    """One rank's DCP prefill partial: (o_part [Hq,Sc,D] fp32, lse_part [Hq,Sc])."""
    lib = _load()
    Hq, Sc, D, W, Hkv, Lcap, Lc = _prefill_dims(q, k_prior, v_prior, k_cur, v_cur)
    o = torch.empty(Hq, Sc, D, device=q.device, dtype=torch.float32)
    lse = torch.empty(Hq, Sc, device=q.device, dtype=torch.float32)
    st = lib.ca_dcp_prefill_partial(_ptr(q), _ptr(k_prior), _ptr(v_prior), _ptr(k_cur), _ptr(v_cur),
                                    DTYPE[q.dtype], Hq, Hkv, Sc, D, W, interleave, int(prior_tokens), Lcap, Lc,
                                    int(rank), float(softmax_scale or 0.0), _ptr(o), _ptr(lse), _stream(q))
    _check("ca_dcp_prefill_partial", st)
    return o, lse


def _rows(x: torch.Tensor):
    if not (x.is_cuda and x.is_contiguous() and x.dim() >= 3):
        raise ValueError("expected a contiguous CUDA tensor [..., S, D]")
    S = x.shape[-2]
    BH = x.numel() // (S * x.shape[-1])
    return BH, S, x.shape[-1] * x.element_size()


def layout_to_shards(x, cp_size, layout="contiguous"):
    """Rows of x [..., S, D] from global token order into shard-major order."""
    BH, S, rb = _rows(x)
    y = torch.empty_like(x)
    _check("ca_layout_to_shards", _load().ca_layout_to_shards(_ptr(x), _ptr(y), BH, S, rb, cp_size,
                                                               LAYOUT[layout], _stream(x)))
    return y


def layout_from_shards(y, cp_size, layout="contiguous"):
    """Inverse of layout_to_shards."""
    BH, S, rb = _rows(y)
    x = torch.empty_like(y)
    _check("ca_layout_from_shards", _load().ca_layout_from_shards(_ptr(y), _ptr(x), BH, S, rb, cp_size,
                                                                   LAYOUT[layout], _stream(y)))
    return x


def dcp_shard_kv(kv, dcp, interleave):
    """kv [N, Hkv, L, D] in global order -> shards [dcp, N, Hkv, L/dcp, D]."""
    BH, L, rb = _rows(kv)
    out = torch.empty((dcp,) + tuple(kv.shape[:-2]) + (L // dcp, kv.shape[-1]), device=kv.device,
                      dtype=kv.dtype)
    _check("ca_dcp_shard_kv", _load().ca_dcp_shard_kv(_ptr(kv), _ptr(out), BH, L, rb, dcp, interleave,
                                                       _stream(kv)))
    return out


# ------------------------------------------------------------- host index helpers
def layout_global_index(layout, cp_size, Ls, row) -> int:
    """Global token position of stored row r*Ls + a (contiguous: r*Ls + a; striped: a*cp + r)."""
    return int(_load().ca_layout_global_index(LAYOUT[layout], cp_size, Ls, row))


def layout_shard_row(layout, cp_size, Ls, token) -> int:
    """Stored row of a global token: the inverse of layout_global_index."""
    return int(_load().ca_layout_shard_row(LAYOUT[layout], cp_size, Ls, token))


def ring_kv_shard(rank, step, cp_size) -> int:
    """K/V shard that shard `rank` meets at ring step `step`: (rank - step) mod cp_size."""
    return int(_load().ca_ring_kv_shard(rank, step, cp_size))


def dcp_owner(pos, dcp, interleave) -> int:
    """DCP rank holding global position pos: (pos // interleave) mod dcp."""
    return int(_load().ca_dcp_owner(pos, dcp, interleave))


def dcp_local_index(pos, dcp, interleave) -> int:
    """Local slot of pos on its owner rank: (pos // (dcp*I))*I + pos % I."""
    return int(_load().ca_dcp_local_index(pos, dcp, interleave))


def dcp_local_to_global(local, rank, dcp, interleave) -> int:
    """Global position of local slot s on a rank: (s // I)*(dcp*I) + rank*I + s % I."""
    return int(_load().ca_dcp_local_to_global(local, rank, dcp, interleave))


def dcp_local_filled(N, dcp, interleave, block_size, rank) -> int:
    """Tokens among positions [0, N) a rank holds (the DCP page's local_filled formula)."""
    return int(_load().ca_dcp_local_filled(N, dcp, interleave, block_size, rank))


def dcp_active_mask(N, dcp, interleave, block_size, rank) -> int:
    """1 if `rank` owns the token at position N (the decoded token), else 0."""
    return int(_load().ca_dcp_active_mask(N, dcp, interleave, block_size, rank))


def dcp_slot_mapping(positions, block_table, block_size, dcp, rank, interleave):
    """Host slot mapping: -1 for positions `rank` does not own."""
    import numpy as np

    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
    bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
    out = np.zeros(len(pos), dtype=np.int64)
    st = _load().ca_dcp_slot_mapping(pos.ctypes.data, len(pos), bt.ctypes.data, len(bt), block_size,
                                      dcp, rank, interleave, out.ctypes.data)
    _check("ca_dcp_slot_mapping", st)
    return out


def selftest_wait_timeout(limit_cycles: int = 2_000_000):
    """Run the failure-path diagnostic on the current stream: one warp's
    bounded wait on a barrier nothing completes gives up after
    `limit_cycles` cycles and raises the device error word (read it with
    device_status())."""
    _check("ca_selftest_wait_timeout", _load().ca_selftest_wait_timeout(int(limit_cycles),
                                                                        torch.cuda.current_stream().cuda_stream))


def device_status(reset: bool = True) -> int:
    """Status of the device error word raised by bounded waits (0 = clean)."""
    return int(_load().ca_device_status(int(reset)))
