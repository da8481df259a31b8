"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random tensors and arranges them in the layouts the
library takes; it holds none of the attention arithmetic.  Both the CUDA path
and the CPU oracle receive the very same tensors from here.

Recipes (shapes follow the workloads on the pages on context parallelism):

* ``normal_qkv``: q, k, v ~ N(0, 1), [B, H, S, D] (k and v with Hkv heads).
* ``dit_qk``: the DiT workload of "Context Parallelism in vLLM Omni Neuron"
  (section "Self-Attention with Context Parallelism": QK RMSNorm over the whole
  hidden before the head split).  For each of q and k: activations
  x ~ N(0, 1) of shape [B, S, H*D], a per-channel gain g ~ 1 + 0.1*N(0, 1),
  y = x / sqrt(mean(x^2 over the hidden) + 1e-6) * g, split into H heads of D
  and transposed to [B, H, S, D].  No rotary embedding (a rotation keeps norms).
* ``sink_rows``: the "attention sinks" stress of the const-max page (section
  "Adapting this kernel"): round(0.01*S) token positions per batch element,
  picked by a seeded permutation, have their k rows scaled by 8 in every head.
* ``decode_inputs``: q [N, Hq, D] and interleaved K/V shards
  [W, N, Hkv, Lloc, D], all ~ N(0, 1).
* ``qkv_activations``: projected activations for the attention prologue:
  x_q [B, S, Hq*D], x_k, x_v [B, S, Hkv*D] ~ N(0, 1) bf16, per-channel gains
  1 + 0.1*N(0, 1) (fp32) for q and k, and rotary tables cos/sin [S, D/2] of
  the angles p * 10000^(-2i/D) (fp32).
"""
from __future__ import annotations

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, dtype=torch.float32, device="cpu") -> torch.Tensor:
    """N(0, 1) tensor drawn in fp32 from ``seed`` then cast to ``dtype``."""
    g = _gen(seed, device)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def normal_qkv(B, Hq, Hkv, S, D, seed, dtype=torch.float32, device="cpu"):
    """q [B,Hq,S,D], k and v [B,Hkv,S,D], all N(0,1), from one seed."""
    g = _gen(seed, device)
    q = torch.randn(B, Hq, S, D, generator=g, device=device).to(dtype)
    k = torch.randn(B, Hkv, S, D, generator=g, device=device).to(dtype)
    v = torch.randn(B, Hkv, S, D, generator=g, device=device).to(dtype)
    return q, k, v


def dit_qk(B, H, S, D, seed, dtype=torch.bfloat16, device="cpu", eps=1e-6):
    """q, k [B,H,S,D] from cross-head RMS-normalised N(0,1) activations, plus v."""
    g = _gen(seed, device)
    out = []
    for _ in range(2):
        x = torch.randn(B, S, H * D, generator=g, device=device)
        gain = 1.0 + 0.1 * torch.randn(H * D, generator=g, device=device)
        y = x * torch.rsqrt(x.pow(2).mean(dim=-1, keepdim=True) + eps) * gain
        out.append(y.view(B, S, H, D).transpose(1, 2).contiguous().to(dtype))
        del x, y
    v = torch.randn(B, H, S, D, generator=g, device=device).to(dtype)
    return out[0], out[1], v


def sink_rows(B, S, seed, frac=0.01, device="cpu"):
    """Per batch element, the sorted token rows chosen as key sinks."""
    g = _gen(seed, "cpu")
    n = int(round(frac * S))
    rows = [torch.randperm(S, generator=g)[:n].sort().values for _ in range(B)]
    return torch.stack(rows).to(device)


def apply_sinks(k: torch.Tensor, rows: torch.Tensor, factor: float = 8.0) -> torch.Tensor:
    """Scale the chosen token rows of k [B,H,S,D] by ``factor`` in every head."""
    k = k.clone()
    for b in range(k.shape[0]):
        k[b, :, rows[b].to(k.device), :] *= factor
    return k


def decode_inputs(N, Hq, Hkv, D, W, Lloc, seed, dtype=torch.bfloat16, device="cpu"):
    """q [N,Hq,D] and K/V shards [W,N,Hkv,Lloc,D], N(0,1)."""
    g = _gen(seed, device)
    q = torch.randn(N, Hq, D, generator=g, device=device).to(dtype)
    k = torch.empty(W, N, Hkv, Lloc, D, device=device, dtype=dtype)
    v = torch.empty(W, N, Hkv, Lloc, D, device=device, dtype=dtype)
    # drawn shard by shard to bound the fp32 staging memory
    for t in (k, v):
        for r in range(W):
            t[r].copy_(torch.randn(N, Hkv, Lloc, D, generator=g, device=device).to(dtype))
    return q, k, v


def dcp_prefill_inputs(Hq, Hkv, D, W, Sc, Lcap, Lc, seed, dtype=torch.bfloat16, device="cpu"):
    """q [Hq,Sc,D], prior shards [W,Hkv,Lcap,D] and current-chunk shards
    [W,Hkv,Lc,D], all N(0,1)."""
    g = _gen(seed, device)
    q = torch.randn(Hq, Sc, D, generator=g, device=device).to(dtype)
    kp = torch.randn(W, Hkv, Lcap, D, generator=g, device=device).to(dtype)
    vp = torch.randn(W, Hkv, Lcap, D, generator=g, device=device).to(dtype)
    kc = torch.randn(W, Hkv, Lc, D, generator=g, device=device).to(dtype)
    vc = torch.randn(W, Hkv, Lc, D, generator=g, device=device).to(dtype)
    return q, kp, vp, kc, vc


def rope_tables(S, D, base=10000.0, device="cpu"):
    """cos, sin [S, D/2] fp32 of the angles p * base^(-2i/D)."""
    p = torch.arange(S, dtype=torch.float64).view(S, 1)
    w = base ** (-2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
    ang = p * w.view(1, -1)
    return torch.cos(ang).float().to(device), torch.sin(ang).float().to(device)


def qkv_activations(B, S, Hq, Hkv, D, seed, device="cpu"):
    """x_q, x_k, x_v (bf16), g_q, g_k (fp32), cos, sin (fp32); see the module doc."""
    g = _gen(seed, device)
    x_q = torch.randn(B, S, Hq * D, generator=g, device=device).to(torch.bfloat16)
    x_k = torch.randn(B, S, Hkv * D, generator=g, device=device).to(torch.bfloat16)
    x_v = torch.randn(B, S, Hkv * D, generator=g, device=device).to(torch.bfloat16)
    g_q = 1.0 + 0.1 * torch.randn(Hq * D, generator=g, device=device)
    g_k = 1.0 + 0.1 * torch.randn(Hkv * D, generator=g, device=device)
    cos, sin = rope_tables(S, D, device=device)
    return x_q, x_k, x_v, g_q, g_k, cos, sin
