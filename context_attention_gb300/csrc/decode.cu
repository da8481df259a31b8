// decode.cu -- split-KV decode over interleaved DCP shards, and over the ring
// layout's shards (Ring Pass-Q decode, "Sharding the Input": the KV cache stays
// where the sharded prefill put it and the query visits every shard).
//
// "DCP (Decode Context Parallelism)", section "Decode Compute Pattern": the
// gathered query heads of a sequence attend to each rank's local KV shard and
// produce a partial output plus its log-sum-exp; the partials are combined by
// the LSE merge (merge.cu).  Section "local_filled Computation" fixes how
// many local slots of rank r hold tokens of a sequence of length N; every one
// of them is visible to the decoded token (its own K/V sits on its owner).
//
// One GPU holds all shards (dcp ranks, or the cp shards of the ring layout,
// whose valid slots and rows differ only in pair_of and seg_tokens).  The
// work is the 128-token stages of every (shard r, sequence n, KV head) pair,
// cut into segments, each one CTA's share of one pair (SegWalk):
//  - with many pairs, each pair's stages form splits of 32 stages (4096
//    tokens) dealt to the CTAs round robin, so the CTAs stream neighbouring
//    parts of the cache at any moment (at 64 sequences, contiguous ranges
//    over the whole cache measured 1-2 % slower);
//  - with few pairs (a handful of sequences), the stages, pair after pair,
//    are cut into one contiguous range per CTA, the ranges differing by at
//    most one stage.  Dealt splits left 104 of 152 CTAs a second 4096-token
//    split at one sequence, where a CTA streams at most ~60 GB/s: the
//    ranges took two sequences from 172.7 to 160.4 us and one from 92.8 to
//    88.7 us.
// Each segment yields one partial per query head, in its pair's slot.  The
// scan is HBM bound: a TMA producer warp streams 128-token stages (K and V,
// 64 KB, each one box holding both 64-column halves of its rows) through a
// 3-stage ring; four consumer warps each take 32 tokens of a stage.  The G
// query heads that share a KV head are the N side of warp-level bf16 MMAs
// (m16n8k16, fp32 accumulate): S^T = K Q^T per 16 tokens, then O^T += V^T P^T,
// with P moved from the accumulator layout to the operand layout by
// movmatrix.  Row maxima use a lazy rescale: the reference moves only when a
// 16-token group's maximum passes it by more than 8 (log2); the rescale of
// the register-resident O is cheap here.  Each head keeps two row sums: of p
// as computed (for the log-sum-exp) and of p rounded to bf16 as the PV MMA
// consumes it (O is divided by this one, so the weights in O and in its
// normaliser are the same and o is a convex combination of V rows).  At the
// end of a segment the four warps' partial states are LSE-merged in shared
// memory and one partial (o, lse) per query head is written.
#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "index_maps.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace ca {
namespace {

constexpr int kTok = 128;                      // tokens per stage
constexpr int kD = 128;
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr uint32_t kBox = kTok * 64 * 2;       // 16 KB: 128 tokens x 64 columns
constexpr uint32_t kStageBytes = 4 * kBox;     // K halves, V halves
constexpr int kMaxG = 8;

constexpr uint32_t kSmemStages = 0;
constexpr uint32_t kSmemMergeO = kStages * kStageBytes;                    // [warps][8][128] f32
constexpr uint32_t kSmemMergeML = kSmemMergeO + kConsumerWarps * kMaxG * kD * 4;  // [warps][8] m, l, lr
constexpr uint32_t kSmemBar = kSmemMergeML + kConsumerWarps * kMaxG * 3 * 4;
constexpr uint32_t kSmemAbort = kSmemBar + (2 * kStages + 1) * 8;
constexpr uint32_t kSmemUsed = kSmemAbort + 4;
constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecParams {
  DecodeArgs a;
  int G;
  uint32_t units;            // pairs * stages, or pairs * splits when dealt (< 2^31)
  uint32_t range_q, range_r;  // units / ctas, units % ctas
  float scale_log2;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One CTA's share of one pair: stages [s0, s1) of pair p, i.e. the pair's
// local slots [t0, t0 + ntok) that hold tokens (none when the segment lies
// past the shard's valid length).
struct Seg {
  int r, n, hkv;
  int64_t t0, ntok;  // first local slot, number of valid tokens
  int64_t row0;      // first row in the [W*N*Hkv*Lloc, D] view (contiguous caches)
  int slot;          // partial slot of the segment within its pair
  bool last;         // the segment ends the pair (its CTA writes the unused slots)
};

// Integer work per segment is 32-bit: a unit, a pair, a slot or a position
// is below 2^31 (the host rejects caches of 2^31 rows or more), and a 64-bit
// division costs ~350 cycles; the first segment's nine of them held every
// CTA's first load back by ~1.5 us.
//
// CTA c deals with units [c * U / C, (c + 1) * U / C), computed as
// c * (U / C) + c * (U % C) / C with the quotient and remainder from the
// host; unit x is on CTA ((x + 1) * C - 1) / U, the last c whose range
// starts at or before x.
__device__ __forceinline__ uint32_t range_begin(const DecParams& P, uint32_t c) {
  return c * P.range_q + (c * P.range_r) / (uint32_t)P.a.ctas;
}
__device__ __forceinline__ uint32_t cta_of_unit(const DecParams& P, uint32_t x) {
  return (uint32_t)((((uint64_t)x + 1) * (uint64_t)P.a.ctas - 1) / P.units);
}

// The pair's valid local slots and first cache row of its slot t0.
__device__ __forceinline__ void pair_of(const DecParams& P, uint32_t pair, Seg& S, int* valid) {
  const DecodeArgs& a = P.a;
  S.hkv = (int)(pair % (uint32_t)a.Hkv);
  const uint32_t rest = pair / (uint32_t)a.Hkv;
  S.n = (int)(rest % (uint32_t)a.N);
  S.r = (int)(rest / (uint32_t)a.N);
  const int Lloc = (int)a.Lloc;
  const int seq = a.seq_lens ? a.seq_lens[S.n] : a.W * Lloc;
  const int v = a.ring_layout < 0 ? dcp_local_filled_t<int>(seq, a.W, a.I, a.I, S.r)
                                  : ring_shard_filled_t<int>(seq, a.W, Lloc, a.ring_layout, S.r);
  *valid = v > Lloc ? Lloc : v;
}

// Segment stages [s0, s1) of the pair: tokens [s0 * 128, min(s1 * 128, valid)).
__device__ __forceinline__ void seg_tokens(const DecParams& P, uint32_t s0, uint32_t s1, int valid,
                                           Seg& S) {
  const DecodeArgs& a = P.a;
  S.t0 = (int64_t)s0 * kTok;
  const int64_t t1 = (int64_t)s1 * kTok < valid ? (int64_t)s1 * kTok : valid;
  S.ntok = t1 > S.t0 ? t1 - S.t0 : 0;
  S.row0 = a.ring_layout < 0 ? (((int64_t)S.r * a.N + S.n) * a.Hkv + S.hkv) * a.Lloc + S.t0
                              : (((int64_t)S.n * a.Hkv + S.hkv) * a.W + S.r) * a.Lloc + S.t0;
}

// Walks one CTA's segments in order; the producer and the consumers each
// run one and see the same sequence.
struct SegWalk {
  uint32_t u, u_end;
};
__device__ __forceinline__ SegWalk seg_walk(const DecParams& P) {
  const DecodeArgs& a = P.a;
  SegWalk w;
  if (a.dealt) {
    w.u = blockIdx.x;
    w.u_end = P.units;
  } else {
    w.u = range_begin(P, blockIdx.x);
    w.u_end = range_begin(P, blockIdx.x + 1);
  }
  return w;
}
__device__ __forceinline__ bool seg_next(const DecParams& P, SegWalk& w, Seg& S) {
  if (w.u >= w.u_end) return false;
  const DecodeArgs& a = P.a;
  int valid;
  if (a.dealt) {
    // unit = (pair, split): a split of split_stages stages, its own slot
    const uint32_t slots = (uint32_t)a.slots, ss = (uint32_t)a.split_stages, SP = (uint32_t)a.stages;
    const uint32_t pair = w.u / slots, split = w.u % slots;
    pair_of(P, pair, S, &valid);
    const uint32_t s0 = split * ss;
    const uint32_t s1 = s0 + ss < SP ? s0 + ss : SP;
    seg_tokens(P, s0, s1, valid, S);
    S.slot = (int)split;
    S.last = false;
    w.u += (uint32_t)a.ctas;
    return true;
  }
  const uint32_t SP = (uint32_t)a.stages;
  const uint32_t pair = w.u / SP, pu0 = pair * SP;
  const uint32_t s1u = w.u_end < pu0 + SP ? w.u_end : pu0 + SP;
  pair_of(P, pair, S, &valid);
  seg_tokens(P, w.u - pu0, s1u - pu0, valid, S);
  // a pair that starts inside this CTA's range has this CTA as its first
  S.slot = w.u == pu0 ? 0 : (int)(blockIdx.x - cta_of_unit(P, pu0));
  S.last = s1u == pu0 + SP;
  w.u = s1u;
  return true;
}

template <bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
dcp_decode_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                  const DecParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = (uint64_t*)(smem + kSmemBar);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[kStages + s]); };
  const uint32_t merge_bar = smem_u32(&bars[2 * kStages]);
  volatile int* abort_flag = (volatile int*)(smem + kSmemAbort);
  float* mo = (float*)(smem + kSmemMergeO);
  float* mml = (float*)(smem + kSmemMergeML);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const DecodeArgs& a = P.a;
  unsigned* err = a.err;

  // the LSE merge that follows may be scheduled now: its blocks fit beside
  // this CTA and wait for this grid to finish before they read a partial
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kConsumerWarps);
    }
    mbar_init(merge_bar, kConsumerWarps);
    fence_barrier_init();
  }
  __syncthreads();
  // launched as a programmatic dependent: the set-up above overlapped the
  // previous kernel on the stream (a previous decode's merge, which may still
  // read this workspace); no global memory is touched before that kernel has
  // completed.  Back-to-back decodes of one sequence: 84.5 -> 82.4 us.
  griddep_wait();

  if (warp == kProducerWarp && kPaged) {
    // Paged cache: a stage's 128 slots are up to 128/bs blocks scattered over
    // the cache.  Lane i fetches block i of the stage through the block table
    // and loads its K rows, then its V rows, each as one box holding both
    // 64-column halves ([half][row], 2 * bs * 128 bytes at a 1024-byte-
    // aligned offset, so every 128-byte row keeps the 128B swizzle of its
    // row index): two boxes per block instead of four halved the TMA
    // operations per stage and raised the paged decode from 6.77 to
    // 7.37 TB/s, the contiguous decode's rate.
    const uint64_t policy = l2_policy_evict_first();
    const uint32_t box_bytes = (uint32_t)a.bs * 128;
    uint64_t pos = 0;
    bool ok = true;
    SegWalk walk = seg_walk(P);
    Seg I;
    while (ok && seg_next(P, walk, I)) {
      const int nst = (int)((I.ntok + kTok - 1) / kTok);
      const int32_t* bt = a.block_tables + ((int64_t)I.r * a.N + I.n) * a.max_blocks;
      for (int st = 0; st < nst; ++st) {
        const int slot = (int)(pos % kStages);
        const int64_t first = I.t0 + (int64_t)st * kTok;  // first local slot of the stage
        const int64_t nvalid = min((int64_t)kTok, I.ntok - (int64_t)st * kTok);
        const int nb = (int)((nvalid + a.bs - 1) / a.bs);
        // the stage's block ids, read before waiting for the slot so that
        // their latency overlaps the wait
        const int64_t blk = lane < nb ? (int64_t)__ldg(bt + first / a.bs + lane) : 0;
        ok = __all_sync(0xffffffffu, mbar_wait(empty(slot), (uint32_t)(((pos / kStages) & 1) ^ 1),
                                               abort_flag, err));
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(full(slot), (uint32_t)nb * 4 * box_bytes);
        __syncwarp();
        if (lane < nb) {
          const int row = (int)((((int64_t)I.r * a.nblk + blk) * a.Hkv + I.hkv) * a.bs);
          // block `lane` at rows [2 * lane * bs, 2 * (lane + 1) * bs) of the
          // stage's K (then V) region: its two halves, one after the other
          const uint32_t dst = sbase + kSmemStages + slot * kStageBytes + (uint32_t)lane * 2 * box_bytes;
          tma_load_3d_hint(dst, &tk, full(slot), 0, row, 0, policy);
          tma_load_3d_hint(dst + 2 * kBox, &tv, full(slot), 0, row, 0, policy);
        }
        ++pos;
      }
    }
    if (!ok && lane == 0) {
      for (uint64_t p = pos > kStages ? pos - kStages : 0; p < pos; ++p) {
        volatile int never = 0;
        mbar_wait(full((int)(p % kStages)), (uint32_t)((p / kStages) & 1), &never, err);
      }
    }
  } else if (warp == kProducerWarp) {
    if (lane == 0) {
      prefetch_tensormap(&tk);
      prefetch_tensormap(&tv);
      const uint64_t policy = l2_policy_evict_first();
      uint64_t pos = 0;
      bool ok = true;
      SegWalk walk = seg_walk(P);
      Seg I;
      while (ok && seg_next(P, walk, I)) {
        const int nst = (int)((I.ntok + kTok - 1) / kTok);
        for (int st = 0; st < nst; ++st) {
          const int slot = (int)(pos % kStages);
          ok = mbar_wait(empty(slot), (uint32_t)(((pos / kStages) & 1) ^ 1), abort_flag, err);
          if (!ok) break;
          mbar_arrive_expect_tx(full(slot), kStageBytes);
          const int row = (int)(I.row0 + (int64_t)st * kTok);
          const uint32_t dst = sbase + kSmemStages + slot * kStageBytes;
          tma_load_3d_hint(dst, &tk, full(slot), 0, row, 0, policy);
          tma_load_3d_hint(dst + 2 * kBox, &tv, full(slot), 0, row, 0, policy);
          ++pos;
        }
      }
      if (!ok) {
        for (uint64_t p = pos > kStages ? pos - kStages : 0; p < pos; ++p) {
          volatile int never = 0;
          mbar_wait(full((int)(p % kStages)), (uint32_t)((p / kStages) & 1), &never, err);
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;  // fragment row / column group
    const int G = P.G;
    // Where token tok's 64-column half h sits in a stage's K (or V) region:
    // (tok + (tok & bmask)) * 128 + h * hstride, each 128-byte row swizzled
    // (16-byte chunk c stored at c ^ (tok & 7)).  Both kinds of cache load
    // boxes holding both 64-column halves of their rows, [half][row]:
    // contiguous caches one box for the stage's 128 rows (bmask 0, hstride =
    // kBox), paged caches one per block of bs rows (bmask = ~(bs - 1),
    // hstride = bs * 128).
    const int bmask = kPaged ? ~(a.bs - 1) : 0;
    const uint32_t hstride = kPaged ? (uint32_t)a.bs * 128 : kBox;
    auto half_row = [&](int tok, int h) {
      return (uint32_t)(tok + (tok & bmask)) * 128 + (uint32_t)h * hstride;
    };
    uint64_t pos = 0;
    uint32_t merges = 0;  // phases completed on merge_bar
    bool ok = true;
    SegWalk walk = seg_walk(P);
    Seg I;
    while (ok && seg_next(P, walk, I)) {
      const int64_t R = (int64_t)a.N * a.Hq;
      const int64_t orow0 = (int64_t)I.n * a.Hq + (int64_t)I.hkv * G;  // first q head row
      if (I.slot < 0 || I.slot >= a.slots) {
        // a slot outside the pair's bound (the host sized it otherwise):
        // reported, nothing written
        if (threadIdx.x == 0) {
          *abort_flag = 1;
          atomicOr(err, kErrBadLaunch);
        }
        ok = false;
        break;
      }
      const int pidx = I.r * a.slots + I.slot;
      // the pair's slots that no segment reaches carry no weight
      if (I.last) {
        for (int idx = threadIdx.x; idx < (a.slots - 1 - I.slot) * G; idx += kConsumerWarps * 32) {
          const int sl = I.slot + 1 + idx / G, h = idx % G;
          a.lse_parts[((int64_t)I.r * a.slots + sl) * R + orow0 + h] = -INFINITY;
        }
      }
      if (I.ntok == 0) {
        // no valid token in the segment: a partial of no weight (the merge
        // does not read the o row of a partial whose lse is -inf)
        for (int h = threadIdx.x; h < G; h += kConsumerWarps * 32)
          a.lse_parts[(int64_t)pidx * R + orow0 + h] = -INFINITY;
        continue;
      }
      // Q^T operand fragments (B of S^T = K Q^T): head g, d = 16kk + 2t (+8)
      uint32_t qf[kD / 16][2];
      {
        const __nv_bfloat16* qh = (const __nv_bfloat16*)a.q + (orow0 + g) * kD;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          qf[kk][0] = g < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 2 * t) : 0u;
          qf[kk][1] = g < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 8 + 2 * t) : 0u;
        }
      }
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, lr0 = 0.f, lr1 = 0.f;
      float acc[kD / 16][4];
#pragma unroll
      for (int mb = 0; mb < kD / 16; ++mb) acc[mb][0] = acc[mb][1] = acc[mb][2] = acc[mb][3] = 0.f;

      const int nst = (int)((I.ntok + kTok - 1) / kTok);
      for (int st = 0; st < nst; ++st) {
        const int slot = (int)(pos % kStages);
        ok = __all_sync(0xffffffffu,
                        mbar_wait(full(slot), (uint32_t)((pos / kStages) & 1), abort_flag, err));
        if (!ok) break;
        const uint32_t kb = sbase + kSmemStages + slot * kStageBytes;
        const uint32_t vb = kb + 2 * kBox;
        const int64_t base = (int64_t)st * kTok;
        const int wt = warp * 32;  // first token of this warp in the stage
        const int64_t nvalid = I.ntok - base;  // valid tokens in this stage (may exceed 128)
        bool wrote = false;
        if (nvalid < wt + 32) {
          // zero the V rows past the valid slots: unused cache slots may hold
          // any bit pattern, and 0 * NaN would poison the accumulators
          const int first = (int)max((int64_t)wt, nvalid);
          const int nrows = wt + 32 - first;
          uint8_t* vrow = smem + kSmemStages + slot * kStageBytes + 2 * kBox;
          for (int idx = lane; idx < nrows * 16; idx += 32) {
            const int tok = first + idx / 16, part = idx % 16;
            *reinterpret_cast<uint4*>(vrow + half_row(tok, part / 8) + (part % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          wrote = true;
          __syncwarp();
        }
#pragma unroll 1
        for (int gi = 0; gi < 2; ++gi) {
          const int tb = wt + 16 * gi;
          if (tb >= nvalid) break;
          float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const int tok = tb + (lane & 7) + 8 * ((lane >> 3) & 1);
            const int ch = 2 * kk + (lane >> 4);  // 16-byte chunk along D (0..15)
            uint32_t af[4];
            ldsm_x4(kb + half_row(tok, ch >> 3) + (uint32_t)(((ch & 7) ^ (tok & 7)) << 4), af);
            mma_bf16(c, af, qf[kk][0], qf[kk][1]);
          }
          const bool va = tb + g < nvalid, vb_ = tb + g + 8 < nvalid;
          const float x0 = va ? c[0] * P.scale_log2 : -INFINITY;
          const float x1 = va ? c[1] * P.scale_log2 : -INFINITY;
          const float x2 = vb_ ? c[2] * P.scale_log2 : -INFINITY;
          const float x3 = vb_ ? c[3] * P.scale_log2 : -INFINITY;
          float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
          }
          if (mx0 > m0 + 8.f || (m0 == -INFINITY && mx0 != -INFINITY)) {
            const float f = m0 == -INFINITY ? 0.f : ex2(m0 - mx0);
            l0 *= f;
            lr0 *= f;
#pragma unroll
            for (int mb = 0; mb < kD / 16; ++mb) {
              acc[mb][0] *= f;
              acc[mb][2] *= f;
            }
            m0 = mx0;
          }
          if (mx1 > m1 + 8.f || (m1 == -INFINITY && mx1 != -INFINITY)) {
            const float f = m1 == -INFINITY ? 0.f : ex2(m1 - mx1);
            l1 *= f;
            lr1 *= f;
#pragma unroll
            for (int mb = 0; mb < kD / 16; ++mb) {
              acc[mb][1] *= f;
              acc[mb][3] *= f;
            }
            m1 = mx1;
          }
          const float r0 = m0 == -INFINITY ? 0.f : m0;
          const float r1 = m1 == -INFINITY ? 0.f : m1;
          const float p0 = ex2(x0 - r0), p1 = ex2(x1 - r1), p2 = ex2(x2 - r0), p3 = ex2(x3 - r1);
          const uint32_t w01 = pack_bf16x2(p0, p1), w23 = pack_bf16x2(p2, p3);
          l0 += p0 + p2;
          l1 += p1 + p3;
          lr0 += __uint_as_float(w01 << 16) + __uint_as_float(w23 << 16);
          lr1 += __uint_as_float(w01 & 0xFFFF0000u) + __uint_as_float(w23 & 0xFFFF0000u);
          const uint32_t pb0 = movm_t(w01);
          const uint32_t pb1 = movm_t(w23);
#pragma unroll
          for (int mb = 0; mb < kD / 16; ++mb) {
            const int q4 = lane >> 3;
            const int tok = tb + 8 * (q4 >> 1) + (lane & 7);
            const int ch = 2 * mb + (q4 & 1);
            uint32_t af[4];
            ldsm_x4_t(vb + half_row(tok, ch >> 3) + (uint32_t)(((ch & 7) ^ (tok & 7)) << 4), af);
            mma_bf16(acc[mb], af, pb0, pb1);
          }
        }
        // generic-proxy writes to the slot must be ordered before the next
        // TMA (async proxy) writes into it
        if (wrote) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(slot));
        ++pos;
      }
      if (!ok) break;
      // ------------------------------------------------ merge the four warps
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        lr0 += __shfl_xor_sync(0xffffffffu, lr0, o);
        lr1 += __shfl_xor_sync(0xffffffffu, lr1, o);
      }
      float* mow = mo + warp * kMaxG * kD;
      float* mlw = mml + warp * kMaxG * 3;
      if (lane < 4) {
        mlw[3 * (2 * t) + 0] = m0;
        mlw[3 * (2 * t) + 1] = l0;
        mlw[3 * (2 * t) + 2] = lr0;
        mlw[3 * (2 * t + 1) + 0] = m1;
        mlw[3 * (2 * t + 1) + 1] = l1;
        mlw[3 * (2 * t + 1) + 2] = lr1;
      }
#pragma unroll
      for (int mb = 0; mb < kD / 16; ++mb) {
        const int d = 16 * mb + g;
        mow[(2 * t) * kD + d] = acc[mb][0];
        mow[(2 * t + 1) * kD + d] = acc[mb][1];
        mow[(2 * t) * kD + d + 8] = acc[mb][2];
        mow[(2 * t + 1) * kD + d + 8] = acc[mb][3];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(merge_bar);
      ok = __all_sync(0xffffffffu, mbar_wait(merge_bar, merges & 1, abort_flag, err));
      ++merges;
      if (!ok) break;
      for (int idx = threadIdx.x; idx < G * kD; idx += kConsumerWarps * 32) {
        const int h = idx / kD, d = idx % kD;
        float M = -INFINITY;
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mml[w * kMaxG * 3 + 3 * h]);
        float L = 0.f, Lr = 0.f, O = 0.f;
        if (M != -INFINITY) {
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = mml[w * kMaxG * 3 + 3 * h];
            if (mw == -INFINITY) continue;
            const float f = ex2(mw - M);
            L += mml[w * kMaxG * 3 + 3 * h + 1] * f;
            Lr += mml[w * kMaxG * 3 + 3 * h + 2] * f;
            O += mo[(w * kMaxG + h) * kD + d] * f;
          }
        }
        const int64_t prow = (int64_t)pidx * R + orow0 + h;
        a.o_parts[prow * kD + d] = L > 0.f ? O / Lr : 0.f;
        if (d == 0) a.lse_parts[prow] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
      }
      // every warp has read the shared partials before the next segment rewrites them
      __syncwarp();
      if (lane == 0) mbar_arrive(merge_bar);
      ok = __all_sync(0xffffffffu, mbar_wait(merge_bar, merges & 1, abort_flag, err));
      ++merges;
    }
  }
  __syncthreads();
}

}  // namespace

DecodeGeometry dcp_decode_geometry(int64_t pairs, int64_t Lloc, int max_ctas) {
  DecodeGeometry g;
  g.stages = (Lloc + kTok - 1) / kTok;
  g.dealt = pairs >= kDecodeDealPairs;
  g.split_stages = 32;  // 4096 tokens
  if (g.dealt) {
    g.slots = (int)((g.stages + g.split_stages - 1) / g.split_stages);
    g.units = pairs * g.slots;
  } else {
    g.units = pairs * g.stages;
  }
  const int64_t c = g.units < max_ctas ? g.units : max_ctas;
  g.ctas = (int)(c > 0 ? c : 0);
  if (g.dealt) return g;
  if (g.ctas == 0) {
    g.slots = 1;
    return g;
  }
  // every range holds at least U / C units, so a pair of SP units meets at
  // most (SP - 2) / (U / C) + 2 ranges: one at each end, the rest inside it
  const int64_t minlen = g.units / g.ctas;
  g.slots = (int)((g.stages - 1) / minlen + 2);
  if (g.slots > g.stages) g.slots = (int)g.stages;
  return g;
}

template <bool kPaged>
static cudaError_t launch_decode(const DecParams& P, const CUtensorMap& tk, const CUtensorMap& tv,
                                 cudaStream_t stream) {
  static std::atomic<int> attr_set[64];  // idempotent once-per-device setup
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(dcp_decode_kernel<kPaged>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)P.a.ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dcp_decode_kernel<kPaged>, tk, tv, P);
}

cudaError_t launch_dcp_decode_partials(const DecodeArgs& a, cudaStream_t stream) {
  DecParams P;
  P.a = a;
  P.G = a.Hq / a.Hkv;
  const int64_t units = (int64_t)a.W * a.N * a.Hkv * (a.dealt ? a.slots : a.stages);
  if (units >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;  // the host's row bound keeps it below
  P.units = (uint32_t)units;
  P.range_q = a.ctas > 0 ? P.units / (uint32_t)a.ctas : 0;
  P.range_r = a.ctas > 0 ? P.units % (uint32_t)a.ctas : 0;
  P.scale_log2 = a.scale * kLog2e;
  if (P.units == 0 || a.ctas <= 0) return cudaSuccess;
  CUtensorMap tk, tv;
  if (a.paged) {
    const uint64_t rows = (uint64_t)a.W * a.nblk * a.Hkv * a.bs;
    // one box per (block, head): both 64-column halves of its bs rows
    if (!encode_bf16_halves_sw128(&tk, a.k, rows, (uint32_t)a.bs) ||
        !encode_bf16_halves_sw128(&tv, a.v, rows, (uint32_t)a.bs))
      return cudaErrorInvalidValue;
    return launch_decode<true>(P, tk, tv, stream);
  }
  const uint64_t rows = (uint64_t)a.W * a.N * a.Hkv * a.Lloc;
  if (!encode_bf16_halves_sw128(&tk, a.k, rows, (uint32_t)kTok) ||
      !encode_bf16_halves_sw128(&tv, a.v, rows, (uint32_t)kTok))
    return cudaErrorInvalidValue;
  return launch_decode<false>(P, tk, tv, stream);
}

// Slot-mapping write of new tokens' K/V into the paged caches: token t goes
// to rank r's slot slots[r*T + t] (block slot / bs, offset slot % bs) unless
// that slot is -1 (the rank does not own the token).  Bit-exact copies of
// 16-byte chunks; one thread per chunk.
__global__ void __launch_bounds__(256)
paged_kv_write_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                      const int64_t* __restrict__ slots, uint4* __restrict__ k_cache,
                      uint4* __restrict__ v_cache, int T, int Hkv, int chunks, int W, int64_t nblk,
                      int bs) {
  const int64_t total = (int64_t)W * T * Hkv * chunks;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % chunks);
    const int h = (int)((i / chunks) % Hkv);
    const int64_t rt = i / ((int64_t)chunks * Hkv);  // r*T + t
    const int t = (int)(rt % T);
    const int r = (int)(rt / T);
    const int64_t slot = slots[rt];
    if (slot < 0 || slot / bs >= nblk) continue;
    const int64_t dst = ((((int64_t)r * nblk + slot / bs) * Hkv + h) * bs + slot % bs) * chunks + c;
    const int64_t src = ((int64_t)t * Hkv + h) * chunks + c;
    k_cache[dst] = k_new[src];
    v_cache[dst] = v_new[src];
  }
}

cudaError_t launch_paged_kv_write(const void* k_new, const void* v_new, const int64_t* slots,
                                  void* k_cache, void* v_cache, int T, int Hkv, int D, int W,
                                  int64_t nblk, int bs, int elem_bytes, cudaStream_t stream) {
  const int chunks = D * elem_bytes / 16;
  const int64_t total = (int64_t)W * T * Hkv * chunks;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  paged_kv_write_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      (const uint4*)k_new, (const uint4*)v_new, slots, (uint4*)k_cache, (uint4*)v_cache, T, Hkv,
      chunks, W, nblk, bs);
  return cudaGetLastError();
}

}  // namespace ca
