// merge.cu -- LSE merge of partial attention results.
//
// "DCP (Decode Context Parallelism)", section "Decode Compute Pattern" steps
// 5-7 and "Segmented Attention CP" step 6: partials (o_i, lse_i) combine with
// weight_i = exp(lse_i - lse_global), lse_global = ln sum_i exp(lse_i).
// "Kernel reference: ring_attention_const_max_fwd", sections "A static bound
// makes the ring reduction pure addition" and "Accumulate, then normalize
// once": with a shared bound c the unnormalised sums just add, and the row is
// normalised once with the 1e-37 clamp.
//
// One warp per output row; each lane owns 16-byte column chunks, so every
// partial row is read with fully coalesced 16-byte loads (HBM bound).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"

namespace ca {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float warp_max(float x) {
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// kMaxChunks: float4 chunks per lane (D <= 128 * kMaxChunks).
template <int kMaxChunks>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
lse_merge_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int n,
                 int64_t R, int D, const float* __restrict__ c, void* __restrict__ o, int out_bf16,
                 float* __restrict__ lse) {
  const int lane = threadIdx.x % 32;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + threadIdx.x / 32;
  if (row >= R) return;
  const int nch = D / 4;  // D % 4 == 0 is checked by the host

  float ref;  // c (const) or the max lse (online)
  float acc = 0.f;
  if (c) {
    ref = c[row];
    for (int i = lane; i < n; i += 32) acc += expf(lse_parts[(int64_t)i * R + row] - ref);
    acc = warp_sum(acc);
  } else {
    float mx = -INFINITY;
    for (int i = lane; i < n; i += 32) mx = fmaxf(mx, lse_parts[(int64_t)i * R + row]);
    ref = warp_max(mx);
    if (ref != -INFINITY) {
      for (int i = lane; i < n; i += 32) {
        const float li = lse_parts[(int64_t)i * R + row];
        if (li != -INFINITY) acc += expf(li - ref);
      }
      acc = warp_sum(acc);
    }
  }
  float out_lse, total_scale;
  bool empty;
  if (c) {
    out_lse = ref + logf(acc);
    total_scale = 1.f / fmaxf(acc, 1e-37f);
    empty = false;
  } else {
    empty = (ref == -INFINITY);
    out_lse = empty ? -INFINITY : ref + logf(acc);
    total_scale = 1.f;
  }

  float4 sum[kMaxChunks];
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j) sum[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!empty) {
    // partials in groups of 32: lane l holds the weight of partial g + l;
    // the rows of kUnroll partials are loaded before any is accumulated
    constexpr int kUnroll = 8;
    for (int g = 0; g < n; g += 32) {
      float wl = 0.f;
      if (g + lane < n) {
        const float li = lse_parts[(int64_t)(g + lane) * R + row];
        // const max: pure addition of unnormalised sums
        wl = c ? 1.f : (li == -INFINITY ? 0.f : expf(li - out_lse));
      }
      const int m = min(32, n - g);
      for (int i0 = 0; i0 < m; i0 += kUnroll) {
        float4 x[kUnroll][kMaxChunks];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const float4* src = reinterpret_cast<const float4*>(o_parts + ((int64_t)(g + i0 + u) * R + row) * D);
#pragma unroll
          for (int j = 0; j < kMaxChunks; ++j) {
            const int ch = lane + 32 * j;
            x[u][j] = (i0 + u < m && ch < nch) ? __ldg(src + ch) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const float w = __shfl_sync(0xffffffffu, wl, (i0 + u) & 31);
#pragma unroll
          for (int j = 0; j < kMaxChunks; ++j) {
            sum[j].x = fmaf(w, x[u][j].x, sum[j].x);
            sum[j].y = fmaf(w, x[u][j].y, sum[j].y);
            sum[j].z = fmaf(w, x[u][j].z, sum[j].z);
            sum[j].w = fmaf(w, x[u][j].w, sum[j].w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j) {
    const int ch = lane + 32 * j;
    if (ch >= nch) continue;
    float4 x = sum[j];
    x.x *= total_scale;
    x.y *= total_scale;
    x.z *= total_scale;
    x.w *= total_scale;
    if (out_bf16) {
      __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y);
      __nv_bfloat162 b = __floats2bfloat162_rn(x.z, x.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&a);
      u.y = *reinterpret_cast<uint32_t*>(&b);
      reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(o) + row * D)[ch] = u;
    } else {
      reinterpret_cast<float4*>(reinterpret_cast<float*>(o) + row * D)[ch] = x;
    }
  }
  if (lse && lane == 0) lse[row] = out_lse;
}

}  // namespace

cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int n, int64_t R,
                             int D, const float* c, void* o, int out_bf16, float* lse,
                             cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  const int64_t blocks = (R + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const unsigned g = (unsigned)blocks, t = kWarpsPerBlock * 32;
  if (D <= 128)
    lse_merge_kernel<1><<<g, t, 0, stream>>>(o_parts, lse_parts, n, R, D, c, o, out_bf16, lse);
  else if (D <= 256)
    lse_merge_kernel<2><<<g, t, 0, stream>>>(o_parts, lse_parts, n, R, D, c, o, out_bf16, lse);
  else
    lse_merge_kernel<4><<<g, t, 0, stream>>>(o_parts, lse_parts, n, R, D, c, o, out_bf16, lse);
  return cudaGetLastError();
}

}  // namespace ca
