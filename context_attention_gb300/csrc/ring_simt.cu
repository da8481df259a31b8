// ring_simt.cu -- fp32 ring attention on the CUDA cores (true fp32 FMA).
//
// fp32 inputs must match the oracle to 1e-4, which the tensor cores' tf32
// path cannot do, so fp32 runs here: one warp per query row group, K/V tiles
// of 32 keys staged in shared memory, exact expf.  Same semantics as the
// tensor-core kernel: the ring schedule of "Kernel reference:
// ring_attention_const_max_fwd" (section "Overview": shard r meets shard
// r - t at step t), online max or the const-max bound (sections "Picking a
// max ..." and "Accumulate, then normalize once"), causal masking on global
// positions of the contiguous or striped layout ("Sharding the Input").
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "index_maps.cuh"
#include "internal.h"

namespace ca {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRows = kWarps * kRowsPerWarp;  // query rows per block
constexpr int kKeys = 32;                     // keys per staged tile
constexpr int kMaxD = 128;
constexpr int kDPer = kMaxD / 32;             // output columns per lane

__global__ void __launch_bounds__(kWarps * 32)
ring_simt_kernel(RingArgs a, int qblocks) {
  extern __shared__ float sm[];
  const int D = a.D;
  const int Ks = D + 1;  // padded K row stride (conflict-free column reads)
  float* sq = sm;                      // [kRows][D]
  float* sk = sq + kRows * D;          // [kKeys][D+1]
  float* sv = sk + kKeys * Ks;         // [kKeys][D]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r_store = blockIdx.x / qblocks;
  const int64_t a0 = (int64_t)(blockIdx.x % qblocks) * kRows;
  const int64_t bh = blockIdx.y;
  const int b = (int)(bh / a.Hq), h = (int)(bh % a.Hq);
  const int G = a.Hq / a.Hkv;
  const int64_t bhk = (int64_t)b * a.Hkv + h / G;
  const int r_log = a.q_rank_fixed >= 0 ? a.q_rank_fixed : r_store;
  const float* q = (const float*)a.q + (bh * a.Sq + (int64_t)r_store * a.Ls) * D;
  const float* kh = (const float*)a.k + bhk * a.Sk * D;
  const float* vh = (const float*)a.v + bhk * a.Sk * D;

  for (int i = threadIdx.x; i < kRows * D; i += blockDim.x) {
    int64_t row = a0 + i / D;
    sq[i] = row < a.Ls ? q[row * D + i % D] : 0.f;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], cst[kRowsPerWarp], o[kRowsPerWarp][kDPer];
  int64_t arow[kRowsPerWarp];
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    arow[rr] = a0 + warp * kRowsPerWarp + rr;
    m[rr] = -INFINITY;
    l[rr] = 0.f;
    cst[rr] = 0.f;
    if (a.mode == 1 && !a.kmax2 && arow[rr] < a.Ls)
      cst[rr] = a.c[bh * a.Sq + (int64_t)r_store * a.Ls + arow[rr]];
    for (int i = 0; i < kDPer; ++i) o[rr][i] = 0.f;
  }
  if (a.mode == 1 && a.kmax2) {
    // each row's bound from its staged q row: c = sqrt(scale^2 * kmax2 * |q|^2)
    __syncthreads();
    const float km = a.kmax2[bhk];
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const float* qr = sq + (warp * kRowsPerWarp + rr) * D;
      float ss = 0.f;
      for (int d = lane; d < D; d += 32) ss = fmaf(qr[d], qr[d], ss);
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      cst[rr] = sqrtf(a.scale * a.scale * km * ss);
    }
  }
  const int64_t a_last = min(a0 + kRows - 1, a.Ls - 1);
  const int nsteps = a.kv_rank_fixed >= 0 ? 1 : a.cp;

  for (int t = 0; t < nsteps; ++t) {
    const int s_log = a.kv_rank_fixed >= 0 ? a.kv_rank_fixed : ring_kv_shard(r_log, t, a.cp);
    const int s_store = a.kv_rank_fixed >= 0 ? 0 : s_log;
    const int64_t delta = a.causal ? causal_delta(a.layout, r_log, s_log) : kDeltaAll;
    if (delta == kDeltaNone) continue;
    int64_t kend = a.Ls;  // keys [0, kend) of the shard can be visible to this block
    if (delta != kDeltaAll) kend = min(kend, a_last - delta + 1);
    for (int64_t kb = 0; kb < kend; kb += kKeys) {
      __syncthreads();
      const float* kt = kh + ((int64_t)s_store * a.Ls + kb) * D;
      const float* vt = vh + ((int64_t)s_store * a.Ls + kb) * D;
      for (int i = threadIdx.x; i < kKeys * D; i += blockDim.x) {
        int j = i / D, d = i % D;
        bool in = kb + j < a.Ls;
        sk[j * Ks + d] = in ? kt[(int64_t)j * D + d] : 0.f;
        sv[j * D + d] = in ? vt[(int64_t)j * D + d] : 0.f;
      }
      __syncthreads();
      const int64_t bkey = kb + lane;
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const float* qr = sq + (warp * kRowsPerWarp + rr) * D;
        float dot = 0.f;
        for (int d = 0; d < D; ++d) dot = fmaf(qr[d], sk[lane * Ks + d], dot);
        float s = dot * a.scale;
        bool vis = bkey < a.Ls && (delta == kDeltaAll || bkey <= arow[rr] - delta);
        float p;
        if (a.mode == 1) {
          p = vis ? expf(s - cst[rr]) : 0.f;
        } else {
          float sm_ = vis ? s : -INFINITY;
          float tmax = sm_;
          for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
          float mnew = fmaxf(m[rr], tmax);
          float fac = (m[rr] == -INFINITY) ? 0.f : expf(m[rr] - mnew);
          if (mnew == -INFINITY) fac = 1.f;
          p = vis ? expf(s - mnew) : 0.f;
          l[rr] *= fac;
          for (int i = 0; i < kDPer; ++i) o[rr][i] *= fac;
          m[rr] = mnew;
        }
        float psum = p;
        for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l[rr] += psum;
        for (int j = 0; j < kKeys; ++j) {
          float pj = __shfl_sync(0xffffffffu, p, j);
          for (int i = 0; i < kDPer; ++i) {
            int d = lane + 32 * i;
            if (d < D) o[rr][i] = fmaf(pj, sv[j * D + d], o[rr][i]);
          }
        }
      }
    }
  }

  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    if (arow[rr] >= a.Ls) continue;
    const int64_t orow = bh * a.Sq + (int64_t)r_store * a.Ls + arow[rr];
    float lse, scl;
    if (a.mode == 1) {
      lse = cst[rr] + logf(l[rr]);
      scl = a.unnormalized ? 1.f : 1.f / fmaxf(l[rr], 1e-37f);
    } else if (l[rr] > 0.f) {
      lse = m[rr] + logf(l[rr]);
      scl = 1.f / l[rr];
    } else {
      lse = -INFINITY;
      scl = 0.f;
    }
    float* out = (float*)a.o + orow * D;
    for (int i = 0; i < kDPer; ++i) {
      int d = lane + 32 * i;
      if (d < D) out[d] = o[rr][i] * scl;
    }
    if (a.lse && lane == 0) a.lse[orow] = lse;
  }
}

}  // namespace

cudaError_t launch_ring_simt_f32(const RingArgs& a, cudaStream_t stream) {
  const int qblocks = (int)((a.Ls + kRows - 1) / kRows);
  dim3 grid((unsigned)(qblocks * a.q_shards), (unsigned)(a.B * a.Hq));
  size_t smem = sizeof(float) * ((size_t)kRows * a.D + (size_t)kKeys * (a.D + 1) + (size_t)kKeys * a.D);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  ring_simt_kernel<<<grid, kWarps * 32, smem, stream>>>(a, qblocks);
  return cudaGetLastError();
}

}  // namespace ca
