// prologue.cu -- the pass that turns projected activations into the inputs
// of const-max ring attention ("Context Parallelism in vLLM Omni Neuron",
// section "Self-Attention with Context Parallelism": q and k are normalised
// over the whole hidden before the head split, rotary embeddings are applied
// per head at each token's position, and the heads are transposed to
// [B, H, S, D]), fused with the key half of the const-max bound ("Kernel
// reference: ring_attention_const_max_fwd", sections "Best practices" and
// "Transpose prologue with fused norms": the per-head max of |k|^2 is
// reduced off the tiles the prologue already holds).
//
// One warp per token row of one tensor; a warp walks the q, k, v rows of a
// run of tokens.  Each warp streams its rows through a few shared-memory
// buffers of its own with 1-D bulk copies (cp.async.bulk, completing on one
// mbarrier per buffer), so whole rows are in flight while other rows are
// processed, and both passes over a q or k row read shared memory: HBM sees
// each input byte once and the load pipe stays full with few warps.
// Lanes take 16-byte chunks lane, lane + 32, ... (8 channels):
//   q, k:  y = x * rsqrt(mean(x^2) + eps) * g, then each channel pair
//          (2i, 2i+1) of a head turns by the token's angle (cos/sin tables
//          [S, D/2]), rounded to bf16 (packed f32x2 arithmetic);
//   v:     copied into the head-major layout.
// The output row of token p is its shard-major row in the chosen layout
// (contiguous: p; striped: (p mod cp) * S/cp + p div cp).  For k, |k_row|^2
// of each head is summed from the rounded bf16 values (the ones attention
// reads), kept as a per-warp running max in shared memory and merged into
// kmax2[b, h] with one atomicMax per head whenever the warp's tokens move
// to another batch element.
#include <atomic>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "index_maps.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ca {
namespace {

constexpr int kMaxWarps = 18;     // per block (one block per SM)
constexpr int kMaxHeads = 128;    // H * D <= 8192 and D >= 64
constexpr int kMaxBufs = 4;       // row buffers per warp

struct PrologueTensor {
  const uint4* x;      // [B, S, H*D] bf16
  const float* g;      // [H*D] or null (gain 1)
  uint4* out;          // [B, H, S, D] bf16
  int H;
  int norm;            // 1: RMS norm + rotation; 0: copy (value)
  int key;             // 1: reduce |k|^2 per head into kmax2
};

struct PrologueArgs {
  PrologueTensor t[3];
  int ntensors;
  int B, D;
  int64_t S;
  int cp, layout;
  float eps;
  const float* cs;     // [S, D/2] or null
  const float* sn;
  float* kmax2;        // [B, Hkv] or null
  int64_t jobs_per_warp;  // tokens per warp
  int nbuf;            // row buffers per warp (1..kMaxBufs)
  uint32_t buf_bytes;  // bytes per buffer (>= the longest row, multiple of 128)
  uint32_t gain_floats;  // gains staged in shared memory (q's then k's)
  unsigned* err;       // device error word
};

// Dynamic shared memory: per-warp key-head maxima, per-warp buffer barriers,
// the block's abort flag, the gains (fp32, q's then k's), then the row
// buffers (128-byte aligned).
__host__ __device__ constexpr uint32_t pro_head_bytes(int warps) {
  return (uint32_t)((warps * kMaxHeads * 4 + warps * kMaxBufs * 8 + 4 + 127) / 128 * 128);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2u(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// The bf16 pair of a 32-bit word as an fp32 pair (exact).
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(uint64_t v) {
  float lo, hi;
  f2u(v, lo, hi);
  return pack2(lo, hi);
}
// Sum of squares of the 8 channels of a chunk, as two partial sums.
__device__ __forceinline__ uint64_t sumsq_chunk(const uint4& u, uint64_t acc) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint64_t v = bf2_to_f2(w[e]);
    acc = f2fma(v, v, acc);
  }
  return acc;
}
__device__ __forceinline__ float f2sum(uint64_t v) {
  float lo, hi;
  f2u(v, lo, hi);
  return lo + hi;
}

constexpr int kGroup = 4;   // chunks per lane per step (output pass)

// kD: head dimension (64 or 128), a constant so that chunk -> (head, offset)
// is a shift and a mask.
template <int kD>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
prologue_kernel(const PrologueArgs a) {
  extern __shared__ __align__(128) uint8_t psm[];
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const int warps = blockDim.x / 32;
  float* kmx = reinterpret_cast<float*>(psm) + warp * kMaxHeads;
  uint64_t* wbar = reinterpret_cast<uint64_t*>(psm + warps * kMaxHeads * 4) + warp * kMaxBufs;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(psm + warps * kMaxHeads * 4 + warps * kMaxBufs * 8);
  float* gsm = reinterpret_cast<float*>(psm + pro_head_bytes(warps));
  const uint32_t gain_bytes = (a.gain_floats * 4 + 127) / 128 * 128;
  uint8_t* wbuf = psm + pro_head_bytes(warps) + gain_bytes + (size_t)warp * a.nbuf * a.buf_bytes;
  const int64_t gwarp = (int64_t)blockIdx.x * warps + warp;
  const int64_t ntok = (int64_t)a.B * a.S;
  const int64_t j0 = min(gwarp * a.jobs_per_warp, ntok);
  const int64_t j1 = min(j0 + a.jobs_per_warp, ntok);
  constexpr int cph = kD / 8;  // chunks per head
  const int64_t Ls = a.S / a.cp;
  if (threadIdx.x == 0) *abort_flag = 0;
  for (int h = lane; h < kMaxHeads; h += 32) kmx[h] = 0.f;
  if (lane == 0) {
    for (int i = 0; i < a.nbuf; ++i) mbar_init(smem_u32(&wbar[i]), 1);
    fence_barrier_init();
  }
  // the gains, read by every chunk of every q and k row, live in shared
  // memory (the row buffers leave little L1)
  const uint32_t glen_q = a.t[0].g ? (uint32_t)a.t[0].H * kD : 0u;
  const uint32_t glen_k = a.t[1].g ? (uint32_t)a.t[1].H * kD : 0u;
  for (uint32_t i = threadIdx.x * 4; i < glen_q; i += blockDim.x * 4)
    *reinterpret_cast<float4*>(gsm + i) = __ldg(reinterpret_cast<const float4*>(a.t[0].g + i));
  for (uint32_t i = threadIdx.x * 4; i < glen_k; i += blockDim.x * 4)
    *reinterpret_cast<float4*>(gsm + glen_q + i) = __ldg(reinterpret_cast<const float4*>(a.t[1].g + i));
  const float* gain_q = glen_q ? gsm : nullptr;
  const float* gain_k = glen_k ? gsm + glen_q : nullptr;
  __syncthreads();
  int cur_b = -1;
  // merge the warp's running key-head maxima of batch element cur_b
  auto flush = [&]() {
    if (cur_b >= 0 && a.kmax2) {
      __syncwarp();
      for (int h = lane; h < a.t[1].H; h += 32) {
        // squares are >= 0: float bits order like unsigned integers
        atomicMax(reinterpret_cast<unsigned*>(a.kmax2) + (int64_t)cur_b * a.t[1].H + h,
                  __float_as_uint(kmx[h]));
        kmx[h] = 0.f;
      }
      __syncwarp();
    }
  };
  // row indices fit 32 bits (the host checks B * S * tensors < 2^31), so the
  // per-row index arithmetic stays in cheap 32-bit divisions
  const uint32_t nt = (uint32_t)a.ntensors, S32 = (uint32_t)a.S, cp32 = (uint32_t)a.cp;
  const int64_t jbeg = j0 * a.ntensors, jend = j1 * a.ntensors;
  // row jt into buffer `slot` (lane 0)
  auto issue = [&](int64_t jt, int slot) {
    const uint32_t ju = (uint32_t)jt;
    const uint32_t tok32 = ju / nt;
    const PrologueTensor& T = a.t[ju - tok32 * nt];
    const uint32_t bytes = (uint32_t)T.H * kD * 2;
    const uint32_t bar = smem_u32(&wbar[slot]);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load_1d(smem_u32(wbuf + (size_t)slot * a.buf_bytes), T.x + (int64_t)tok32 * (T.H * cph), bytes, bar);
  };
  if (lane == 0)
    for (int i = 0; i < a.nbuf && jbeg + i < jend; ++i) issue(jbeg + i, i);
  int64_t n = 0;  // rows consumed
  bool ok = true;
  for (int64_t jt = jbeg; jt < jend; ++jt, ++n) {
    const uint32_t ju = (uint32_t)jt;
    const uint32_t tok32 = ju / nt;
    const int t = (int)(ju - tok32 * nt);  // q, k, then v of the token
    const int b = (int)(tok32 / S32);
    const uint32_t p32 = tok32 - (uint32_t)b * S32;
    const int64_t p = p32;  // token (global position)
    if (b != cur_b) {
      flush();
      cur_b = b;
    }
    const int slot = (int)(n % a.nbuf);
    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&wbar[slot]), (uint32_t)((n / a.nbuf) & 1), abort_flag, a.err));
    if (!ok) break;
    const uint4* xr = reinterpret_cast<const uint4*>(wbuf + (size_t)slot * a.buf_bytes);
    const PrologueTensor& T = a.t[t];
    const int nchunks = T.H * cph;
    const int rounds = (nchunks + 31) / 32;
    // stored row of token p: contiguous p; striped (p mod cp) * Ls + p div cp
    int64_t orow = p;
    if (a.layout == kLayoutStriped) {
      const uint32_t a_sh = p32 / cp32;
      orow = (int64_t)(p32 - a_sh * cp32) * Ls + a_sh;
    }
    uint4* orow_base = T.out + ((int64_t)b * T.H * a.S + orow) * cph;  // head 0 of the row
    const int64_t head_stride = a.S * cph;                              // uint4 per head
    if (!T.norm) {
#pragma unroll 4
      for (int c = lane; c < nchunks; c += 32) orow_base[(c / cph) * head_stride + c % cph] = xr[c];
    } else {
      // pass 1: sum of squares
      uint64_t ss2 = f2(0.f, 0.f);
#pragma unroll 4
      for (int c = lane; c < nchunks; c += 32) ss2 = sumsq_chunk(xr[c], ss2);
      float ss = f2sum(ss2);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float rstd = rsqrtf(ss / (float)(T.H * kD) + a.eps);
      const uint64_t rstd2 = f2(rstd, rstd);
      // a lane's chunks c = lane + 32 i all sit at the same offset in their
      // head (cph divides 32), so its rotation angles are loaded once per row
      const int d0 = (lane % cph) * 8;
      float cc[4] = {1.f, 1.f, 1.f, 1.f}, sv[4] = {0.f, 0.f, 0.f, 0.f};
      if (a.cs) {
        const float4 c4 = __ldg(reinterpret_cast<const float4*>(a.cs + p * (kD / 2) + d0 / 2));
        const float4 s4 = __ldg(reinterpret_cast<const float4*>(a.sn + p * (kD / 2) + d0 / 2));
        cc[0] = c4.x; cc[1] = c4.y; cc[2] = c4.z; cc[3] = c4.w;
        sv[0] = s4.x; sv[1] = s4.y; sv[2] = s4.z; sv[3] = s4.w;
      }
      const float* gs = t == 0 ? gain_q : t == 1 ? gain_k : nullptr;
      // pass 2: normalise, gain, turn, round, store (and key-head norms)
      for (int i0 = 0; i0 < rounds; i0 += kGroup) {
        float hsq[kGroup];
#pragma unroll
        for (int g = 0; g < kGroup; ++g) {
          const int c = lane + 32 * (i0 + g);
          hsq[g] = 0.f;
          if (c >= nchunks) continue;
          const uint4 u = xr[c];
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
          uint64_t y[4];
          if (gs) {
            const float4 g0 = *reinterpret_cast<const float4*>(gs + c * 8);
            const float4 g1 = *reinterpret_cast<const float4*>(gs + c * 8 + 4);
            const uint64_t gg[4] = {f2(g0.x, g0.y), f2(g0.z, g0.w), f2(g1.x, g1.y), f2(g1.z, g1.w)};
#pragma unroll
            for (int e = 0; e < 4; ++e) y[e] = f2mul(f2mul(bf2_to_f2(w[e]), rstd2), gg[e]);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) y[e] = f2mul(bf2_to_f2(w[e]), rstd2);
          }
          if (a.cs) {
            // (y0, y1) -> (y0 c - y1 s, y0 s + y1 c) = (y0, y1) * c + (-y1, y0) * s
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float y0, y1;
              f2u(y[e], y0, y1);
              y[e] = f2fma(y[e], f2(cc[e], cc[e]), f2mul(f2(-y1, y0), f2(sv[e], sv[e])));
            }
          }
          const uint4 o = make_uint4(f2_to_bf2(y[0]), f2_to_bf2(y[1]), f2_to_bf2(y[2]), f2_to_bf2(y[3]));
          orow_base[(c / cph) * head_stride + c % cph] = o;
          if (T.key) hsq[g] = f2sum(sumsq_chunk(o, f2(0.f, 0.f)));
        }
        if (T.key) {
          // |k|^2 of each head: the cph lanes holding its chunks in a round (32
          // is a multiple of cph, so heads never straddle rounds); the shuffle
          // trees of the group's rounds are independent and interleave
#pragma unroll
          for (int off = 8; off > 0; off >>= 1)
            if (off < cph) {
#pragma unroll
              for (int g = 0; g < kGroup; ++g) hsq[g] += __shfl_xor_sync(0xffffffffu, hsq[g], off, cph);
            }
#pragma unroll
          for (int g = 0; g < kGroup; ++g) {
            const int c = lane + 32 * (i0 + g);
            if (c < nchunks && (c % cph) == 0) kmx[c / cph] = fmaxf(kmx[c / cph], hsq[g]);
          }
        }
      }
    }
    // the buffer is free once every lane has read it: refill it with the
    // row nbuf ahead (generic-proxy reads before the async-proxy write)
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && jt + a.nbuf < jend) issue(jt + a.nbuf, slot);
  }
  if (!ok) {
    // error path: let this warp's copies still in flight land before exit
    volatile int never = 0;
    if (lane == 0)
      for (int64_t m = n; m < n + a.nbuf && jbeg + m < jend; ++m)
        mbar_wait(smem_u32(&wbar[m % a.nbuf]), (uint32_t)((m / a.nbuf) & 1), &never, a.err);
    __syncwarp();
    return;
  }
  flush();
}

}  // namespace

cudaError_t launch_qkv_prologue(const QkvPrologueArgs& q, cudaStream_t stream) {
  if (q.D != 64 && q.D != 128) return cudaErrorInvalidValue;
  PrologueArgs a;
  const void* xs[3] = {q.x_q, q.x_k, q.x_v};
  const float* gs[3] = {q.g_q, q.g_k, nullptr};
  void* outs[3] = {q.q, q.k, q.v};
  const int hs[3] = {q.Hq, q.Hkv, q.Hkv};
  a.ntensors = 0;
  int max_h = 0;
  for (int i = 0; i < 3; ++i) {
    if (!xs[i]) continue;
    PrologueTensor& T = a.t[a.ntensors++];
    T.x = static_cast<const uint4*>(xs[i]);
    T.g = gs[i];
    T.out = static_cast<uint4*>(outs[i]);
    T.H = hs[i];
    T.norm = i < 2;
    T.key = i == 1;
    if (hs[i] > max_h) max_h = hs[i];
  }
  if (max_h * q.D > kMaxHeads * 64 || max_h > kMaxHeads) return cudaErrorInvalidValue;
  a.B = q.B;
  a.D = q.D;
  a.S = q.S;
  a.cp = q.cp;
  a.layout = q.layout;
  a.eps = q.eps;
  a.cs = q.cos;
  a.sn = q.sin;
  a.kmax2 = q.kmax2;
  if (q.kmax2) {
    cudaError_t e = cudaMemsetAsync(q.kmax2, 0, sizeof(float) * (size_t)q.B * q.Hkv, stream);
    if (e != cudaSuccess) return e;
  }
  const int64_t ntok = (int64_t)q.B * q.S;
  if (ntok == 0) return cudaSuccess;
  a.err = q.err;
  // one block per SM; buffers sized for the longest row.  Long rows get one
  // buffer per warp (the next row is requested as soon as the current one has
  // been read): more warps, each with one row in flight, outrun fewer warps
  // that prefetch deeper.  Short rows get more buffers, so that a warp keeps
  // about 8 KB or more in flight.  Warps: as many as shared memory holds, up
  // to ~160 KB of rows in flight per SM (measured: beyond that the extra
  // copies only queue in the memory system and the kernel slows down).
  const uint32_t row_bytes = (uint32_t)max_h * q.D * 2;
  a.buf_bytes = (row_bytes + 127) / 128 * 128;
  a.nbuf = a.buf_bytes >= 8192 ? 1 : a.buf_bytes >= 4096 ? 2 : kMaxBufs;
  constexpr uint32_t kSmemBudget = 232448;  // per block, opt-in maximum
  a.gain_floats = (uint32_t)((q.g_q ? q.Hq : 0) + (q.g_k ? q.Hkv : 0)) * q.D;
  const uint32_t gain_bytes = (a.gain_floats * 4 + 127) / 128 * 128;
  int warps = kMaxWarps;
  while (warps > 1 && (uint32_t)warps * a.nbuf * a.buf_bytes > 160u * 1024u) --warps;
  while (warps > 1 && pro_head_bytes(warps) + gain_bytes + (uint32_t)warps * a.nbuf * a.buf_bytes > kSmemBudget)
    --warps;
  const uint32_t smem = pro_head_bytes(warps) + gain_bytes + (uint32_t)warps * a.nbuf * a.buf_bytes;
  const int64_t total = (int64_t)device_sm_count() * warps;
  a.jobs_per_warp = (ntok + total - 1) / total;
  const int64_t nwarps = (ntok + a.jobs_per_warp - 1) / a.jobs_per_warp;
  const unsigned blocks = (unsigned)((nwarps + warps - 1) / warps);
  auto kern = q.D == 128 ? prologue_kernel<128> : prologue_kernel<64>;
  static std::atomic<int> attr_set[64][2];  // idempotent once-per-device setup
  int dev = 0;
  cudaGetDevice(&dev);
  const int di = q.D == 128;
  if (dev >= 0 && dev < 64 && !attr_set[dev][di]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
    if (e != cudaSuccess) return e;
    attr_set[dev][di] = 1;
  }
  kern<<<blocks, warps * 32, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ca
