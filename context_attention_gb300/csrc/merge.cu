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
// Each lane owns 16-byte column chunks, so every partial row is read with
// fully coalesced 16-byte loads.  Three orders of the same arithmetic: one
// warp per output row for partials that sit in L2 (the plain kernel) and
// for larger ones, HBM bound (the prefetching one); one block per row for a
// few rows with many partials (the wide kernel, a decode's).  A partial of
// zero weight -- its lse is -inf, or its weight underflows -- adds nothing
// and its o row is not used, so it may hold any bits: a decode leaves the
// rows of its empty slots unwritten.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

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

// kMaxChunks: float4 chunks per lane (D <= 128 * kMaxChunks).  For partials
// that sit in L2 (a decode's, read right after they were written): the
// row's weights first, then its partial rows eight at a time.
template <int kMaxChunks>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
lse_merge_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int n,
                 int64_t R, int D, const float* __restrict__ c, void* __restrict__ o, int out_bf16,
                 float* __restrict__ lse) {
  griddep_wait();
  griddep_launch_dependents();
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
        wl = li == -INFINITY ? 0.f : (c ? 1.f : expf(li - out_lse));
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
          if (w == 0.f) continue;  // a partial of no weight: its row is not used
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

// partial rows loaded together: 8 for D <= 128, fewer for wider rows so
// that a group stays 32 registers per lane
template <int kMaxChunks>
__host__ __device__ constexpr int group_of() { return 8 / kMaxChunks; }

// Loads the rows of partials g .. g + group - 1 (those below n) of `row`:
// lane l takes the 16-byte column chunks l, l + 32, ...
template <int kMaxChunks>
__device__ __forceinline__ void load_group(float4 (&x)[group_of<kMaxChunks>()][kMaxChunks],
                                           const float* __restrict__ o_parts, int g, int n, int64_t R,
                                           int64_t row, int D, int nch, int lane) {
#pragma unroll
  for (int u = 0; u < group_of<kMaxChunks>(); ++u) {
    const float4* src = reinterpret_cast<const float4*>(o_parts + ((int64_t)(g + u) * R + row) * D);
#pragma unroll
    for (int j = 0; j < kMaxChunks; ++j) {
      const int ch = lane + 32 * j;
      x[u][j] = (g + u < n && ch < nch) ? __ldg(src + ch) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// The same merge for partials larger than L2 (HBM bound): the first group
// of partial rows is requested before the row's log-sum-exp is reduced (the
// rows do not depend on the weights), so a row's two DRAM round trips
// overlap, and at D <= 128 three blocks fit on an SM (80 registers).
template <int kMaxChunks>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, kMaxChunks == 1 ? 3 : 1)
lse_merge_prefetch_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int n,
                 int64_t R, int D, const float* __restrict__ c, void* __restrict__ o, int out_bf16,
                 float* __restrict__ lse) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x % 32;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + threadIdx.x / 32;
  if (row >= R) return;
  const int nch = D / 4;  // D % 4 == 0 is checked by the host

  constexpr int kGroup = group_of<kMaxChunks>();
  float4 x[kGroup][kMaxChunks];
  load_group<kMaxChunks>(x, o_parts, 0, n, R, row, D, nch, lane);

  // lane l holds the lse of partial l (the first 32 partials)
  const float l0 = lane < n ? lse_parts[(int64_t)lane * R + row] : -INFINITY;
  float ref;  // c (const) or the max lse (online)
  float acc = 0.f;
  if (c) {
    ref = c[row];
    acc = lane < n ? expf(l0 - ref) : 0.f;
    for (int i = lane + 32; i < n; i += 32) acc += expf(lse_parts[(int64_t)i * R + row] - ref);
    acc = warp_sum(acc);
  } else {
    float mx = l0;
    for (int i = lane + 32; i < n; i += 32) mx = fmaxf(mx, lse_parts[(int64_t)i * R + row]);
    ref = warp_max(mx);
    if (ref != -INFINITY) {
      acc = l0 != -INFINITY ? expf(l0 - ref) : 0.f;
      for (int i = lane + 32; i < n; i += 32) {
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
    // lane l holds the weight of partial g + l of the current group of 32
    // (const max: pure addition of unnormalised sums)
    auto weight = [&](float li) { return li == -INFINITY ? 0.f : (c ? 1.f : expf(li - out_lse)); };
    float wl = lane < n ? weight(l0) : 0.f;
    for (int g = 0; g < n; g += kGroup) {
      if (g > 0) load_group<kMaxChunks>(x, o_parts, g, n, R, row, D, nch, lane);
      if (g > 0 && (g & 31) == 0) {
        const int i = g + lane;
        wl = i < n ? weight(lse_parts[(int64_t)i * R + row]) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const float w = __shfl_sync(0xffffffffu, wl, (g + u) & 31);
        if (w == 0.f) continue;  // a partial of no weight: its row is not used
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
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j) {
    const int ch = lane + 32 * j;
    if (ch >= nch) continue;
    float4 y = sum[j];
    y.x *= total_scale;
    y.y *= total_scale;
    y.z *= total_scale;
    y.w *= total_scale;
    if (out_bf16) {
      __nv_bfloat162 a = __floats2bfloat162_rn(y.x, y.y);
      __nv_bfloat162 b = __floats2bfloat162_rn(y.z, y.w);
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&a);
      u.y = *reinterpret_cast<uint32_t*>(&b);
      reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(o) + row * D)[ch] = u;
    } else {
      reinterpret_cast<float4*>(reinterpret_cast<float*>(o) + row * D)[ch] = y;
    }
  }
  if (lse && lane == 0) lse[row] = out_lse;
}

// The same merge for few rows with many partials (a decode's: tens to a few
// thousand rows): one block per row, its eight warps taking every eighth
// partial, so a row's partials are read in one or two round trips instead of
// one per group of eight; the warps' sums then add in shared memory in warp
// order.
template <int kMaxChunks>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
lse_merge_wide_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int n,
                      int64_t R, int D, const float* __restrict__ c, void* __restrict__ o,
                      int out_bf16, float* __restrict__ lse) {
  __shared__ float4 red[kWarpsPerBlock][32 * kMaxChunks];
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int64_t row = blockIdx.x;
  const int nch = D / 4;  // D % 4 == 0 is checked by the host

  // every warp reduces the row's log-sum-exp (the same loads and order)
  float ref;
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
    // warp w takes partials w, w + 8, ...: four of them loaded before any
    // is accumulated
    constexpr int kUnroll = 4;
    for (int i0 = warp; i0 < n; i0 += kUnroll * kWarpsPerBlock) {
      float4 x[kUnroll][kMaxChunks];
      float w[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = i0 + u * kWarpsPerBlock;
        const float4* src = reinterpret_cast<const float4*>(o_parts + ((int64_t)i * R + row) * D);
        const float li = i < n ? lse_parts[(int64_t)i * R + row] : -INFINITY;
        // const max: pure addition of unnormalised sums
        w[u] = (i < n && li != -INFINITY) ? (c ? 1.f : expf(li - out_lse)) : 0.f;
#pragma unroll
        for (int j = 0; j < kMaxChunks; ++j) {
          const int ch = lane + 32 * j;
          x[u][j] = (i < n && ch < nch) ? __ldg(src + ch) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (w[u] == 0.f) continue;  // a partial of no weight: its row is not used
#pragma unroll
        for (int j = 0; j < kMaxChunks; ++j) {
          sum[j].x = fmaf(w[u], x[u][j].x, sum[j].x);
          sum[j].y = fmaf(w[u], x[u][j].y, sum[j].y);
          sum[j].z = fmaf(w[u], x[u][j].z, sum[j].z);
          sum[j].w = fmaf(w[u], x[u][j].w, sum[j].w);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j) red[warp][lane + 32 * j] = sum[j];
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int j = 0; j < kMaxChunks; ++j) {
    const int ch = lane + 32 * j;
    if (ch >= nch) continue;
    float4 x = red[0][ch];
#pragma unroll
    for (int v = 1; v < kWarpsPerBlock; ++v) {
      const float4 y = red[v][ch];
      x.x += y.x;
      x.y += y.y;
      x.z += y.z;
      x.w += y.w;
    }
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

// Partials larger than this take the prefetching kernel (they stream from
// HBM); smaller ones, such as a decode's, are read from L2, where the plain
// kernel's order measured faster (32 x 2048 rows: 6.9 against 8.5 us).
constexpr size_t kPrefetchMergeBytes = (size_t)64 << 20;

// Rows up to this many with 16 or more partials take the wide kernel: one
// warp per row reads a row's partials eight at a time, one round trip each,
// which for the 32 rows of a one-sequence decode left 32 warps on the GPU
// (91.8 against 89.7 us for the whole decode).  At 2048 rows (64 sequences)
// the wide kernel's blocks need two waves and it was the slower one (17.4
// against 10.0 us a launch, cold cache under ncu).
constexpr int64_t kWideMergeRows = 1024;

template <typename Kernel>
static cudaError_t launch_merge(Kernel kernel, unsigned grid, unsigned threads, cudaStream_t stream,
                                const float* o_parts, const float* lse_parts, int n, int64_t R,
                                int D, const float* c, void* o, int out_bf16, float* lse) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, o_parts, lse_parts, n, R, D, c, o, out_bf16, lse);
}

cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int n, int64_t R,
                             int D, const float* c, void* o, int out_bf16, float* lse,
                             cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  const int64_t blocks = (R + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const unsigned g = (unsigned)blocks, t = kWarpsPerBlock * 32;
  const bool big = (size_t)n * (size_t)R * (size_t)D * sizeof(float) > kPrefetchMergeBytes;
#define CA_MERGE(K) launch_merge(K, g, t, stream, o_parts, lse_parts, n, R, D, c, o, out_bf16, lse)
  if (!big && R <= kWideMergeRows && n >= 16) {
    const unsigned gw = (unsigned)R;
#define CA_MERGE_W(K) launch_merge(K, gw, t, stream, o_parts, lse_parts, n, R, D, c, o, out_bf16, lse)
    return D <= 128 ? CA_MERGE_W(lse_merge_wide_kernel<1>)
                    : D <= 256 ? CA_MERGE_W(lse_merge_wide_kernel<2>) : CA_MERGE_W(lse_merge_wide_kernel<4>);
#undef CA_MERGE_W
  }
  if (big)
    return D <= 128 ? CA_MERGE(lse_merge_prefetch_kernel<1>)
                    : D <= 256 ? CA_MERGE(lse_merge_prefetch_kernel<2>) : CA_MERGE(lse_merge_prefetch_kernel<4>);
  return D <= 128 ? CA_MERGE(lse_merge_kernel<1>)
                  : D <= 256 ? CA_MERGE(lse_merge_kernel<2>) : CA_MERGE(lse_merge_kernel<4>);
#undef CA_MERGE
}

}  // namespace ca
