// layout.cu -- bit-exact row permutations between global token order and the
// shard-major storage of the virtual shards.
//
// Contiguous and striped layouts: "Context Parallelism in vLLM Omni Neuron"
// (section "Model Implementation": rank r holds [r*local_S, (r+1)*local_S))
// and "Sharding the Input" (striped attention: token t on device t mod cp).
// DCP interleave: "DCP (Decode Context Parallelism)", sections "Slot Mapping
// and KV Cache" (block b of I tokens on rank b mod W) and "Segmented
// Attention CP" (slot s of rank R is global (s/I)*(W*I) + R*I + s%I).
//
// Pure data movement: one thread per 16-byte chunk, consecutive threads on
// consecutive chunks of a row, so both reads and writes are coalesced.
#include <cuda_runtime.h>
#include <stdint.h>

#include "index_maps.cuh"
#include "internal.h"

namespace ca {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
permute_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t BH, int64_t S,
                    int64_t chunks, int cp, int layout, int to_shards) {
  const int64_t Ls = S / cp;
  const int64_t total = BH * S * chunks;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t ch = i % chunks;
    const int64_t row = i / chunks;
    const int64_t bh = row / S;
    const int64_t rho = row % S;  // stored (shard-major) row
    const int r = (int)(rho / Ls);
    const int64_t a = rho % Ls;
    const int64_t g = layout_global(layout, cp, Ls, r, a);
    const int64_t sr = bh * S + (to_shards ? g : rho);
    const int64_t dr = bh * S + (to_shards ? rho : g);
    dst[dr * chunks + ch] = src[sr * chunks + ch];
  }
}

__global__ void __launch_bounds__(kThreads)
dcp_shard_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t NH, int64_t L,
                 int64_t chunks, int W, int I) {
  const int64_t Lloc = L / W;
  const int64_t total = (int64_t)W * NH * Lloc * chunks;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t ch = i % chunks;
    const int64_t row = i / chunks;      // (R, nh, s)
    const int64_t s = row % Lloc;
    const int64_t nh = (row / Lloc) % NH;
    const int R = (int)(row / (Lloc * NH));
    const int64_t g = dcp_local_to_global(s, R, W, I);
    dst[row * chunks + ch] = src[(nh * L + g) * chunks + ch];
  }
}

int64_t grid_for(int64_t total) {
  int64_t blocks = (total + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  return blocks < cap ? blocks : cap;
}

}  // namespace

cudaError_t launch_permute_rows(const void* src, void* dst, int64_t BH, int64_t S,
                                int64_t row_bytes, int cp, int layout, int to_shards,
                                cudaStream_t stream) {
  const int64_t chunks = row_bytes / 16;
  const int64_t total = BH * S * chunks;
  if (total == 0) return cudaSuccess;
  permute_rows_kernel<<<(unsigned)grid_for(total), kThreads, 0, stream>>>(
      (const uint4*)src, (uint4*)dst, BH, S, chunks, cp, layout, to_shards);
  return cudaGetLastError();
}

cudaError_t launch_dcp_shard_rows(const void* src, void* dst, int64_t NH, int64_t L,
                                  int64_t row_bytes, int W, int I, cudaStream_t stream) {
  const int64_t chunks = row_bytes / 16;
  const int64_t total = NH * L * chunks;
  if (total == 0) return cudaSuccess;
  dcp_shard_kernel<<<(unsigned)grid_for(total), kThreads, 0, stream>>>(
      (const uint4*)src, (uint4*)dst, NH, L, chunks, W, I);
  return cudaGetLastError();
}

}  // namespace ca
