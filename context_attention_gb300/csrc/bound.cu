// bound.cu -- the const-max bound of "Kernel reference:
// ring_attention_const_max_fwd" (sections "Picking a max that is safe
// without measuring it", "Global key max", "Assembling the bound"):
//   kmax2[b, hk] = max over all S keys of the head of |k_j|^2
//   c[b, h, i]   = sqrt(scale^2 * kmax2[b, h / G] * |q_i|^2)
// Squares are summed in fp32; the square root is taken once per row.
// Both passes stream their input once with 16-byte loads: HBM bound.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace ca {
namespace {

constexpr int kThreads = 256;
constexpr int kKeyRowsPerBlock = 256;

// Sum of squares of one 16-byte chunk.
__device__ __forceinline__ float sumsq16(const uint4& u, bool bf16) {
  float s = 0.f;
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  if (bf16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
      s = fmaf(lo, lo, s);
      s = fmaf(hi, hi, s);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float x = __uint_as_float(w[i]);
      s = fmaf(x, x, s);
    }
  }
  return s;
}

// |row|^2 for row `row` of a matrix whose rows are `chunks` 16-byte chunks
// (tpr threads per row, tpr a power of two <= 32, chunks % tpr == 0), or of
// D scalar elements when chunks == 0.  Every lane of the warp must call it
// (the reduction shuffles use the full mask); lanes with valid == false
// contribute nothing and get 0.
__device__ __forceinline__ float row_sumsq(const uint8_t* base, int64_t row, bool valid, int D,
                                           int elem, int chunks, int tpr, int sub) {
  float s = 0.f;
  if (valid) {
    if (chunks > 0) {
      const uint4* p = reinterpret_cast<const uint4*>(base + row * (int64_t)D * elem);
      for (int c = sub; c < chunks; c += tpr) s += sumsq16(__ldg(p + c), elem == 2);
    } else {
      for (int d = sub; d < D; d += tpr) {
        float x;
        if (elem == 2) {
          x = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[row * D + d]);
        } else {
          x = reinterpret_cast<const float*>(base)[row * D + d];
        }
        s = fmaf(x, x, s);
      }
    }
  }
  for (int off = tpr / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off, tpr);
  return s;
}

// Row loops are arranged so that all lanes of a warp make the same number of
// trips: a warp owns whole groups of rows per trip and steps by whole warps,
// so the full-mask shuffles never see a lane missing.
//
// Key pass, vector path (rows of `chunks` 16-byte chunks, tpr lanes a row):
// a warp takes kLoads * 32 / tpr consecutive rows per trip and issues all
// kLoads row loads before reducing any, so each lane keeps kLoads 16-byte
// loads in flight.
constexpr int kLoads = 4;

template <int tpr>
__global__ void __launch_bounds__(kThreads)
kmax2_vec_kernel(const uint8_t* k, int64_t S, int D, int elem, int chunks,
                 int64_t rows_per_block, float* kmax2) {
  __shared__ float red[kThreads / 32];
  const int64_t bhk = blockIdx.y;
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int sub = lane % tpr;
  constexpr int rows_per_load = 32 / tpr;
  constexpr int rows_per_trip = kLoads * rows_per_load;
  const int64_t r0 = (int64_t)blockIdx.x * rows_per_block;
  const int64_t r1 = min(r0 + rows_per_block, S);
  const int64_t row_bytes = (int64_t)D * elem;
  const uint8_t* head = k + bhk * S * row_bytes;
  float mx = 0.f;
  for (int64_t base = r0 + (int64_t)warp * rows_per_trip; base < r1;
       base += (int64_t)(kThreads / 32) * rows_per_trip) {
    uint4 x[kLoads];
    float s[kLoads];
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      const int64_t r = base + i * rows_per_load + lane / tpr;
      x[i] = r < r1 ? __ldg(reinterpret_cast<const uint4*>(head + r * row_bytes) + sub)
                    : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
      const int64_t r = base + i * rows_per_load + lane / tpr;
      s[i] = sumsq16(x[i], elem == 2);
      if (r < r1)  // rows wider than tpr chunks
        for (int c = sub + tpr; c < chunks; c += tpr)
          s[i] += sumsq16(__ldg(reinterpret_cast<const uint4*>(head + r * row_bytes) + c), elem == 2);
    }
#pragma unroll
    for (int i = 0; i < kLoads; ++i) {
#pragma unroll
      for (int off = tpr / 2; off > 0; off >>= 1) s[i] += __shfl_xor_sync(0xffffffffu, s[i], off, tpr);
      mx = fmaxf(mx, s[i]);  // rows past r1 contribute 0, the neutral value
    }
  }
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int i = 0; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
    // squares are >= 0, so their bit patterns order like unsigned integers
    atomicMax(reinterpret_cast<unsigned*>(kmax2) + bhk, __float_as_uint(m));
  }
}

// Key pass, scalar path (rows whose byte length is not a multiple of 16).
__global__ void __launch_bounds__(kThreads)
kmax2_kernel(const uint8_t* k, int64_t S, int D, int elem, int chunks, int tpr,
             float* kmax2) {
  __shared__ float red[kThreads / 32];
  const int64_t bhk = blockIdx.y;
  const int rows_per_warp = 32 / tpr;
  const int rows_per_pass = kThreads / tpr;
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int sub = lane % tpr;
  const int64_t r0 = (int64_t)blockIdx.x * kKeyRowsPerBlock;
  const int64_t r1 = min(r0 + kKeyRowsPerBlock, S);
  float mx = 0.f;
  for (int64_t base = r0 + (int64_t)warp * rows_per_warp; base < r1; base += rows_per_pass) {
    const int64_t r = base + lane / tpr;
    const bool valid = r < r1;
    const float s = row_sumsq(k, bhk * S + r, valid, D, elem, chunks, tpr, sub);
    if (valid) mx = fmaxf(mx, s);
  }
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int i = 0; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
    atomicMax(reinterpret_cast<unsigned*>(kmax2) + bhk, __float_as_uint(m));
  }
}

__global__ void __launch_bounds__(kThreads)
bound_kernel(const uint8_t* q, int64_t rows, int64_t S, int Hq, int Hkv, int D, int elem,
             int chunks, int tpr, float scale, const float* kmax2, float* c) {
  const int rows_per_warp = 32 / tpr;
  const int rows_per_block = kThreads / tpr;
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int sub = lane % tpr;
  const int G = Hq / Hkv;
  for (int64_t base = (int64_t)blockIdx.x * rows_per_block + (int64_t)warp * rows_per_warp; base < rows;
       base += (int64_t)gridDim.x * rows_per_block) {
    const int64_t r = base + lane / tpr;
    const bool valid = r < rows;
    const float s = row_sumsq(q, r, valid, D, elem, chunks, tpr, sub);
    if (valid && sub == 0) {
      const int64_t bh = r / S;
      const int64_t b = bh / Hq, h = bh % Hq;
      const float km = kmax2[b * Hkv + h / G];
      c[r] = sqrtf(scale * scale * km * s);
    }
  }
}

void pick_vector(int D, int elem, int* chunks, int* tpr) {
  const int bytes = D * elem;
  *chunks = 0;
  *tpr = 32;
  if (bytes % 16 == 0) {
    int ch = bytes / 16;
    int t = 1;
    while (t * 2 <= 32 && ch % (t * 2) == 0) t *= 2;
    *chunks = ch;
    *tpr = t;
  }
}

}  // namespace

cudaError_t launch_key_max2(const void* k, int is_bf16, int B, int Hkv, int64_t S, int D,
                            float* kmax2, cudaStream_t stream) {
  const int elem = is_bf16 ? 2 : 4;
  int chunks, tpr;
  pick_vector(D, elem, &chunks, &tpr);
  cudaError_t e = cudaMemsetAsync(kmax2, 0, sizeof(float) * (size_t)B * Hkv, stream);
  if (e != cudaSuccess || S == 0) return e;
  if (chunks > 0) {
    // about four resident blocks per SM over all heads, whole warp trips per block
    const int64_t trip = (int64_t)(kThreads / 32) * kLoads * (32 / tpr);
    const int64_t want = (int64_t)device_sm_count() * 4;
    int64_t per_head = (want + (int64_t)B * Hkv - 1) / ((int64_t)B * Hkv);
    int64_t rows_per_block = (S + per_head - 1) / per_head;
    rows_per_block = ((rows_per_block + trip - 1) / trip) * trip;
    const int64_t nb = (S + rows_per_block - 1) / rows_per_block;
    dim3 g((unsigned)nb, (unsigned)(B * Hkv));
#define CA_KMAX2_VEC(T)                                                                 \
  case T:                                                                               \
    kmax2_vec_kernel<T><<<g, kThreads, 0, stream>>>((const uint8_t*)k, S, D, elem, chunks, \
                                                    rows_per_block, kmax2);             \
    break;
    switch (tpr) {
      CA_KMAX2_VEC(1)
      CA_KMAX2_VEC(2)
      CA_KMAX2_VEC(4)
      CA_KMAX2_VEC(8)
      CA_KMAX2_VEC(16)
      CA_KMAX2_VEC(32)
      default: return cudaErrorInvalidValue;
    }
#undef CA_KMAX2_VEC
  } else {
    dim3 g((unsigned)((S + kKeyRowsPerBlock - 1) / kKeyRowsPerBlock), (unsigned)(B * Hkv));
    kmax2_kernel<<<g, kThreads, 0, stream>>>((const uint8_t*)k, S, D, elem, chunks, tpr, kmax2);
  }
  return cudaGetLastError();
}

cudaError_t launch_const_max_bound(const void* q, const void* k, int is_bf16, int B, int Hq,
                                   int Hkv, int64_t S, int D, float scale, float* c,
                                   float* kmax2, cudaStream_t stream) {
  cudaError_t e = launch_key_max2(k, is_bf16, B, Hkv, S, D, kmax2, stream);
  if (e != cudaSuccess || S == 0) return e;
  const int elem = is_bf16 ? 2 : 4;
  int chunks, tpr;
  pick_vector(D, elem, &chunks, &tpr);
  const int64_t rows = (int64_t)B * Hq * S;
  const int rows_per_block = kThreads / tpr;
  int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  bound_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>((const uint8_t*)q, rows, S, Hq, Hkv,
                                                          D, elem, chunks, tpr, scale, kmax2, c);
  return cudaGetLastError();
}

}  // namespace ca
