// ring_tc.cu -- bf16 ring attention on the 5th-generation tensor cores.
//
// What it computes ("Kernel reference: ring_attention_const_max_fwd",
// sections "Overview", "Design", "Accumulate, then normalize once"; "Sharding
// the Input" for causal/striped; "DCP (Decode Context Parallelism)" for the
// LSE form of a partial): the query rows of virtual shard r stay resident
// while the K/V of shard (r - t) mod cp is visited at ring step t; every
// step's scores are shifted either by the running row maximum (online max) or
// by the static per-row bound c_i (const max), exponentiated, summed and
// multiplied into V, and everything accumulates in fp32 across all steps.
//
// How (one GPU, GB300): a persistent kernel, one CTA per SM.  A work unit is
// two 128-row query tiles of one (batch, shard): the same rows of two query
// heads that share a KV head when the GQA group size is even, else two
// consecutive row blocks of one head.  Warp roles:
//   warps 0-3, 4-7   softmax warpgroups, one per query tile: each thread owns
//                    one query row (one TMEM lane) -- it reads its S row from
//                    TMEM, applies mask, shift and exp2, keeps the row sum in
//                    a register, writes P (bf16) back over S in TMEM, and at
//                    the end normalises O and writes o and lse;
//   warp 8           TMA producer: Q tiles, then K and V tiles of the unit's
//                    ring steps, through a 5-slot ring of 32 KB buffers --
//                    first, step by step, the tiles every row of the unit
//                    sees whole, then the tiles a causal or ragged-end mask
//                    crosses, which the softmax runs in a loop of their own;
//   warp 9           tcgen05 issuer: the whole warp walks the schedule (its
//                    descriptors stay warp-uniform) and lane 0 issues
//                    S_i = Q_i K^T and O_i += P_i V for both tiles,
//                    interleaved so that one tile's softmax overlaps the other
//                    tile's matrix products.
// TMEM (512 columns): S0, S1 (fp32, 128 each; P aliases their first 64), O0,
// O1 (fp32, 128 each).  The accumulators never leave TMEM until the unit ends.
//
// Online max uses a lazy rescale: a row's reference maximum only moves when
// a tile's maximum exceeds it by more than kRescaleThreshold (log2 units), so
// O is rescaled in TMEM only on those rare tiles; bf16 P keeps fp32's range,
// so P may grow far above 1 meanwhile.  Const max never rescales: merging the
// ring steps is pure addition.
#include <atomic>
#include <type_traits>
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

constexpr int kBM = 128;     // query rows per tile
constexpr int kBN = 128;     // keys per tile
constexpr int kD = 128;      // head dimension
constexpr int kUnitRows = 2 * kBM;
constexpr int kNSlot = 5;    // K/V ring slots
constexpr uint32_t kTileBytes = kBM * kD * 2;  // 32 KB
constexpr uint32_t kBoxBytes = kTileBytes / 2;  // one 64-column half
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;

constexpr uint32_t kSmemQ = 0;
constexpr uint32_t kSmemKV = 2 * kTileBytes;
constexpr uint32_t kSmemBar = kSmemKV + kNSlot * kTileBytes;
// barrier indices
// Loads land on "group" barriers, one per tile: a unit's Q tiles and K_0 on
// q_full; V_j together with K_(j+1) on tile_full[(t) % kNGroup], t the
// CTA's running tile index.  The issuing thread then waits once per tile for
// both operands of PV(j) and S(j+1).
constexpr int kNGroup = 4;
constexpr int kBarKvFull = 0;  // kNGroup tile barriers
constexpr int kBarKvEmpty = kBarKvFull + kNGroup;
constexpr int kBarQFull = kBarKvEmpty + kNSlot;
constexpr int kBarQEmpty = kBarQFull + 1;
constexpr int kBarSFull = kBarQEmpty + 1;   // 2
constexpr int kBarPFull = kBarSFull + 2;    // 2
constexpr int kBarOFull = kBarPFull + 2;    // 2
constexpr int kBarDrain = kBarOFull + 2;    // error path: the MMAs issued so far completed
constexpr int kNumBars = kBarDrain + 1;
constexpr uint32_t kSmemTmemSlot = kSmemBar + 8 * kNumBars;
constexpr uint32_t kSmemAbort = kSmemTmemSlot + 4;
constexpr uint32_t kSmemUsed = kSmemAbort + 4;
constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;  // slack for 1024-byte alignment
static_assert(kSmemAlloc <= 232448, "dynamic shared memory per block");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // + 128*i
constexpr uint32_t kColO = 256;  // + 128*i

constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kD, false, true);

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Online max: the reference moves only when a row's maximum passes it by
// more than this (log2 units).  P is bf16, which has fp32's exponent range,
// and a tile's P is kept only when its maximum lies at most 64 above the
// reference, so P <= 2^64 and O, l stay far from fp32 overflow; a high
// threshold saves the O rescales that rows with a few very loud keys would
// otherwise trigger again and again.
constexpr float kRescaleThreshold = 48.0f;
constexpr int kMaxRanks = 8;               // segmented schedule

struct TcParams {
  RingArgs a;
  // A unit's two 128-row query tiles: the same rows of two query heads that
  // share a KV head (hp = 1, when the GQA group size is even), else two
  // consecutive row blocks of one head.  Paired heads see the same causal
  // limits and the same K/V tiles, so neither tile runs key tiles that lie
  // wholly past its diagonal; a 256-row unit's first tile runs one such
  // tile per ring step.
  int hp;
  int unit_rows;    // query rows per unit and head: 128 (hp) or 256
  int qblocks;      // units per stored q shard and head (slot)
  int64_t units;    // total work units
  int64_t per_head; // units per head slot: (b, h), or (b, head pair) when hp
  int nsteps;
  int nkt;          // key tiles per shard
  float scale_log2;
  // Segmented schedule (DCP prefill): the keys of rank R come in two
  // segments -- its prior cache slots [0, lp[R]) and its current-chunk
  // tokens [0, lc[R]) -- read through per-rank tensor maps; current token j
  // is visible to query row a iff j <= local_filled(a + 1, W, I, I, R) - 1.
  int seg;          // 0: ring schedule over virtual shards, 1: segmented
  int W, I;         // DCP degree and interleave (segmented)
  int part_rank;    // segmented: -1 = all ranks, else only this rank
  int64_t lp[kMaxRanks], lc[kMaxRanks];
};

// Tensor maps of one launch: q, then (K, V) per key source.  The ring
// schedule uses one 2-D source (all shards of a head, rows of the stored
// tensor); the segmented schedule uses 3-D sources [Hkv, rows, D] per rank
// and segment (prior = 2R, current = 2R + 1) whose row extent is the rank's
// valid count, so TMA fills rows past it with zeros.
struct TcMaps {
  CUtensorMap q;
  CUtensorMap kv[2 * 2 * kMaxRanks];
};

struct Unit {
  int64_t bh, bh1;  // b * Hq + head of query tile 0 and of query tile 1
  int b, h;
  int64_t bhk;
  int r_store, r_log;
  int64_t qrow0;  // first local query row of the unit
};

// Units of one (batch, head) are consecutive (their K/V stay hot in L2) and
// heaviest first: contiguous causal work grows with the shard index and then
// the row block; striped causal work grows with the row block only (every
// shard pair has a diagonal); non-causal units are all equal.
__device__ __forceinline__ Unit unit_of(const TcParams& P, int64_t u) {
  Unit U;
  const int64_t slot = u / P.per_head;  // (b, h) or (b, head pair)
  const int64_t rem = P.per_head - 1 - (u % P.per_head);
  if (P.a.causal && P.a.layout == kLayoutContiguous) {
    U.r_store = (int)(rem / P.qblocks);
    U.qrow0 = (rem % P.qblocks) * P.unit_rows;
  } else {
    U.r_store = (int)(rem % P.a.q_shards);
    U.qrow0 = (rem / P.a.q_shards) * P.unit_rows;
  }
  if (P.hp) {
    U.b = (int)(slot / (P.a.Hq / 2));
    U.h = (int)(slot % (P.a.Hq / 2)) * 2;
    U.bh = (int64_t)U.b * P.a.Hq + U.h;
    U.bh1 = U.bh + 1;
  } else {
    U.bh = U.bh1 = slot;
    U.b = (int)(slot / P.a.Hq);
    U.h = (int)(slot % P.a.Hq);
  }
  U.bhk = (int64_t)U.b * P.a.Hkv + U.h / (P.a.Hq / P.a.Hkv);
  U.r_log = P.a.q_rank_fixed >= 0 ? P.a.q_rank_fixed : U.r_store;
  return U;
}

// Head (b * Hq + h) and first local query row of query tile i of a unit.
__device__ __forceinline__ int64_t tile_bh(const Unit& U, int i) { return i ? U.bh1 : U.bh; }
__device__ __forceinline__ int64_t tile_row0(const TcParams& P, const Unit& U, int i) {
  return U.qrow0 + (P.hp ? 0 : (int64_t)i * kBM);
}
// TMA row of query tile i's first row in the [B * Hq * Sq, D] view of q.
__device__ __forceinline__ int tile_qrow(const TcParams& P, const Unit& U, int i) {
  return (int)(tile_bh(U, i) * P.a.Sq + (int64_t)U.r_store * P.a.Ls + tile_row0(P, U, i));
}

// The k-th unit of this CTA: units are dealt to CTAs in a snake order
// (0..G-1, then G-1..0, ...) which, on a heaviest-first unit list, evens out
// the per-CTA work of causal runs.  Returns >= P.units when none is left.
__device__ __forceinline__ int64_t unit_at(const TcParams& P, int64_t k) {
  const int64_t G = gridDim.x;
  return k * G + ((k & 1) ? (G - 1 - (int64_t)blockIdx.x) : (int64_t)blockIdx.x);
}

// One step of a unit's key sequence: which source the keys come from, where
// they start, how many there are, and how the causal rule limits them.
enum { kMaskNone = 0, kMaskDelta = 1, kMaskDcp = 2 };
struct Step {
  int nk;         // key tiles that can be visible to some row of the unit
  int src;        // key source: tensor maps kv[2*src] (K), kv[2*src+1] (V)
  int64_t row0;   // ring: TMA row of key 0; segmented: 0 (rows are per source)
  int64_t nkeys;  // keys in the step (ragged end)
  int mask;       // kMaskNone / kMaskDelta / kMaskDcp
  int64_t delta;  // kMaskDelta: key b visible to row a iff b <= a - delta
  int rank;       // kMaskDcp: rank whose current tokens these are
};

// kSegMode 0: the ring schedule only; 1: the segmented schedule when P.seg.
template <int kSegMode>
__device__ __forceinline__ Step step_info(const TcParams& P, const Unit& U, int t) {
  Step st;
  const int64_t a_max = min(U.qrow0 + P.unit_rows - 1, P.a.Ls - 1);
  if (kSegMode != 0 && P.seg) {
    const int R = P.part_rank >= 0 ? P.part_rank : (t >> 1);
    st.rank = R;
    st.row0 = 0;
    st.delta = 0;
    if ((t & 1) == 0) {  // prior slots: all before the chunk, all visible
      st.src = 2 * R;
      st.nkeys = P.lp[R];
      st.mask = kMaskNone;
      st.nk = (int)((st.nkeys + kBN - 1) / kBN);
    } else {             // current chunk tokens of rank R: causal by global position
      st.src = 2 * R + 1;
      st.nkeys = P.lc[R];
      st.mask = kMaskDcp;
      int64_t jmax = dcp_local_filled(a_max + 1, P.W, P.I, P.I, R) - 1;
      if (jmax > st.nkeys - 1) jmax = st.nkeys - 1;
      st.nk = jmax < 0 ? 0 : (int)(jmax / kBN + 1);
    }
    return st;
  }
  const int s_log = P.a.kv_rank_fixed >= 0 ? P.a.kv_rank_fixed : ring_kv_shard(U.r_log, t, P.a.cp);
  const int s_store = P.a.kv_rank_fixed >= 0 ? 0 : s_log;
  st.src = 0;
  st.rank = 0;
  st.row0 = U.bhk * P.a.Sk + (int64_t)s_store * P.a.Ls;
  st.nkeys = P.a.Ls;
  st.delta = P.a.causal ? causal_delta(P.a.layout, U.r_log, s_log) : kDeltaAll;
  st.mask = st.delta == kDeltaAll ? kMaskNone : kMaskDelta;
  if (st.delta == kDeltaNone) {
    st.nk = 0;
  } else if (st.delta == kDeltaAll) {
    st.nk = P.nkt;
  } else {
    const int64_t bmax = a_max - st.delta;
    st.nk = bmax < 0 ? 0 : (int)min((int64_t)P.nkt, bmax / kBN + 1);
  }
  return st;
}

template <int kSegMode>
__device__ __forceinline__ int unit_tiles(const TcParams& P, const Unit& U) {
  int n = 0;
  for (int t = 0; t < P.nsteps; ++t) n += step_info<kSegMode>(P, U, t).nk;
  return n;
}

// Last key of step `st` visible to query row a (may be < 0: none).
template <int kSegMode>
__device__ __forceinline__ int64_t step_row_limit(const TcParams& P, const Step& st, int64_t a) {
  int64_t lim = st.nkeys - 1;
  if (st.mask == kMaskDelta) {
    lim = min(lim, a - st.delta);
  } else if (kSegMode != 0 && st.mask == kMaskDcp) {
    lim = min(lim, dcp_local_filled(a + 1, P.W, P.I, P.I, st.rank) - 1);
  }
  return lim;
}

// Walks the (step, key tile) sequence of a unit.  kPhased: first the tiles
// that every row of the unit sees whole, step by step, then, step by step,
// the rest (a row's last visible key grows with the row, so those are the
// tail of each step's range, found from the unit's first row): the softmax
// runs the two phases in separate loops, the first without the masked code.
template <int kSegMode, bool kPhased>
struct TileIter {
  int t, kt, kend;
  int phase;
  bool new_step;  // true on the first tile of a step within a phase
  Step st;
  __device__ __forceinline__ void seek(const TcParams& P, const Unit& U) {
    if constexpr (!kPhased) {
      kt = 0;
      while (t < P.nsteps) {
        st = step_info<kSegMode>(P, U, t);
        if (st.nk > 0) return;
        ++t;
      }
    } else {
      for (;;) {
        if (t >= P.nsteps) {
          if (phase == 1) return;
          phase = 1;
          t = 0;
        }
        st = step_info<kSegMode>(P, U, t);
        if (st.nk > 0) {
          const int64_t lo = step_row_limit<kSegMode>(P, st, U.qrow0);
          const int km = lo < 0 ? 0 : (int)min((int64_t)st.nk, (lo + 1) / kBN);
          const int k0 = phase == 0 ? 0 : km, k1 = phase == 0 ? km : st.nk;
          if (k0 < k1) {
            kt = k0;
            kend = k1;
            return;
          }
        }
        ++t;
      }
    }
  }
  __device__ __forceinline__ void begin(const TcParams& P, const Unit& U) {
    t = 0;
    phase = 0;
    new_step = true;
    seek(P, U);
  }
  __device__ __forceinline__ void next(const TcParams& P, const Unit& U) {
    new_step = false;
    if (++kt < (kPhased ? kend : st.nk)) return;
    ++t;
    new_step = true;
    seek(P, U);
  }
};

// S_i = Q_i K^T: eight K=16 MMAs.  Both operands are K-major 128-byte
// swizzled tiles stored as two 64-column halves, so the k-th MMA starts 32 B
// further along inside a half (+2 in 16-byte descriptor units) and the second
// half 16 KB further (+1024).  All eight issue from one asm block with the
// descriptors advanced by 64-bit adds, keeping the issuing thread's own
// instruction count (and so its share of contended issue slots) small.  The
// whole warp executes the block with warp-uniform operands; only lane 0
// issues.
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint64_t qdesc, uint64_t kdesc) {
  asm volatile(
      "{\n\t"
      ".reg .pred pf, pt, pl;\n\t"
      ".reg .b32 ln;\n\t"
      "mov.u32 ln, %%laneid;\n\t"
      "setp.eq.u32 pl, ln, 0;\n\t"
      ".reg .b64 a, b;\n\t"
      "setp.ne.b32 pf, %3, %3;\n\t"
      "setp.eq.b32 pt, %3, %3;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
      "add.s64 a, %1, 2;\n\tadd.s64 b, %2, 2;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 4;\n\tadd.s64 b, %2, 4;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 6;\n\tadd.s64 b, %2, 6;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 1024;\n\tadd.s64 b, %2, 1024;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 1026;\n\tadd.s64 b, %2, 1026;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 1028;\n\tadd.s64 b, %2, 1028;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
      "add.s64 a, %1, 1030;\n\tadd.s64 b, %2, 1030;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, pt;\n\t"
      "}" ::"r"(d_tmem),
      "l"(qdesc), "l"(kdesc), "n"(kIdescS)
      : "memory");
}

// O_i (+)= P_i V: eight K=16 MMAs with P (bf16, two values per 32-bit TMEM
// column) as the TMEM A operand, +8 columns per MMA, and V as the MN-major
// B operand, +16 rows = +2048 B (+128 descriptor units) per MMA.
// `acc` = 0 makes the first MMA overwrite O (first tile of a unit).
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t vdesc,
                                         uint32_t acc) {
  asm volatile(
      "{\n\t"
      ".reg .pred pa, pt, pl;\n\t"
      ".reg .b32 ln;\n\t"
      "mov.u32 ln, %%laneid;\n\t"
      "setp.eq.u32 pl, ln, 0;\n\t"
      ".reg .b64 b;\n\t"
      ".reg .b32 a;\n\t"
      "setp.ne.b32 pa, %3, 0;\n\t"
      "setp.eq.b32 pt, %3, %3;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, pa;\n\t"
      "add.s32 a, %1, 8;\n\tadd.s64 b, %2, 128;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, pt;\n\t"
      "add.s32 a, %1, 16;\n\tadd.s64 b, %2, 256;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, pt;\n\t"
      "add.s32 a, %1, 24;\n\tadd.s64 b, %2, 384;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, pt;\n\t"
      "add.s32 a, %1, 32;\n\tadd.s64 b, %2, 512;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, pt;\n\t"
      "add.s32 a, %1, 40;\n\tadd.s64 b, %2, 640;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, pt;\n\t"
      "add.s32 a, %1, 48;\n\tadd.s64 b, %2, 768;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, pt;\n\t"
      "add.s32 a, %1, 56;\n\tadd.s64 b, %2, 896;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, pt;\n\t"
      "}" ::"r"(d_tmem),
      "r"(p_tmem), "l"(vdesc), "r"(acc), "n"(kIdescPV)
      : "memory");
}

// Orders every use of registers filled by tcgen05.ld after the wait::ld that
// makes them valid (the compiler sees the wait as unrelated to them).
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; i += 8)
    asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]),
                 "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7]));
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <bool kMask>
__device__ __forceinline__ float chunk_max(const uint32_t (&r)[32], int col0, int vis_max, float mx) {
  if (kMask) {
#pragma unroll
    for (int x = 0; x < 32; ++x)
      mx = fmaxf(mx, col0 + x > vis_max ? -INFINITY : __uint_as_float(r[x]));
    return mx;
  }
  float a = mx, b = __uint_as_float(r[0]);
#pragma unroll
  for (int x = 1; x < 31; x += 2) {
    a = max3(a, __uint_as_float(r[x]), __uint_as_float(r[x + 1]));
  }
  return max3(a, b, __uint_as_float(r[31]));
}

// Row maximum of the 128 raw scores of this thread's TMEM lane; loads are
// software-pipelined so that one 32-column load is in flight while the
// previous one is reduced.
template <bool kMask>
__device__ __forceinline__ float row_max_from_tmem(uint32_t tS, int vis_max) {
  uint32_t ra[32], rb[32];
  float mx = -INFINITY;
  tmem_ld32(tS, ra);
  tmem_ld_wait();
  reg_fence(ra);
  tmem_ld32(tS + 32, rb);
  mx = chunk_max<kMask>(ra, 0, vis_max, mx);
  tmem_ld_wait();
  reg_fence(rb);
  tmem_ld32(tS + 64, ra);
  mx = chunk_max<kMask>(rb, 32, vis_max, mx);
  tmem_ld_wait();
  reg_fence(ra);
  tmem_ld32(tS + 96, rb);
  mx = chunk_max<kMask>(ra, 64, vis_max, mx);
  tmem_ld_wait();
  reg_fence(rb);
  return chunk_max<kMask>(rb, 96, vis_max, mx);
}

// 4x4 transpose of 16-byte blocks inside each group of four lanes.  On
// entry a[k] is block k of this lane's 64 bytes; on exit a[i] is block
// (lane % 4) of the 64 bytes lane (lane & ~3) + i held.  Four lanes then
// write four consecutive blocks of one row: whole 32-byte sectors.
__device__ __forceinline__ uint4 shfl_xor_u4(uint4 v, int m) {
  v.x = __shfl_xor_sync(0xffffffffu, v.x, m);
  v.y = __shfl_xor_sync(0xffffffffu, v.y, m);
  v.z = __shfl_xor_sync(0xffffffffu, v.z, m);
  v.w = __shfl_xor_sync(0xffffffffu, v.w, m);
  return v;
}
__device__ __forceinline__ void quad_transpose(uint4 (&a)[4], int lane) {
  const bool b1 = (lane & 2) != 0, b0 = (lane & 1) != 0;
  // exchange the off-diagonal 2x2 blocks with lane ^ 2
  uint4 r0 = shfl_xor_u4(b1 ? a[0] : a[2], 2);
  uint4 r1 = shfl_xor_u4(b1 ? a[1] : a[3], 2);
  if (b1) {
    a[0] = r0;
    a[1] = r1;
  } else {
    a[2] = r0;
    a[3] = r1;
  }
  // exchange inside each 2x2 block with lane ^ 1
  r0 = shfl_xor_u4(b0 ? a[0] : a[1], 1);
  r1 = shfl_xor_u4(b0 ? a[2] : a[3], 1);
  if (b0) {
    a[0] = r0;
    a[2] = r1;
  } else {
    a[1] = r0;
    a[3] = r1;
  }
}

// Packed fp32 pair arithmetic (one instruction for two lanes of data), used
// to keep the softmax's instruction count low: the softmax warps share issue
// slots with the single thread that issues the tensor-core MMAs.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// The two row sums of a softmax row.  `l` sums p as computed (fp32): it gives
// the log-sum-exp.  `lr` is the sum O is divided by.  On a tile that needs a
// mask (a causal diagonal, a shard's ragged end), for a warp holding a row
// that sees fewer than kRoundedSumKeys keys in all, lr sums p as the PV
// product consumes it, rounded to bf16, so that every weight in the
// numerator is matched by the same weight in the denominator ("Accumulate,
// then normalize once": the accumulator and its row sum come from one set of
// weights): the rows that see only a handful of keys -- where one weight's
// rounding error would otherwise move o by up to 2^-8 |o| -- get o as an
// exact convex combination of their V rows up to fp32 accumulation.
// Elsewhere lr takes the fp32 p like l: there a row's weight is spread over
// a thousand keys or more, and forming the rounded sum on every tile costs
// 8-14 % of the kernel's throughput (the softmax warps' issue slots are the
// bound); on the masked tiles of many-key rows it cost striped causal 0.75 %.
constexpr int64_t kRoundedSumKeys = 1024;

struct RowSums {
  uint64_t l2, lr2;  // packed pairs of partial sums
};

// Adds the two bf16 halves of w, widened exactly, into the pair sum lr2.
__device__ __forceinline__ void add_bf16_pair(uint64_t& lr2, uint32_t w) {
  lr2 = f2_add(lr2, f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)));
}

// p for one pair of scores: sums it into `rs` (lr too when kInl) and returns
// it as a packed bf16 pair (lo = p0).
template <bool kInl>
__device__ __forceinline__ uint32_t exp_pair(float s0, float s1, uint64_t sl2_2, uint64_t nref_2,
                                             RowSums& rs) {
  float a0, a1;
  f2_unpack(f2_fma(f2_pack(s0, s1), sl2_2, nref_2), a0, a1);
  const float p0 = ex2(a0), p1 = ex2(a1);
  const uint32_t w = pack_bf16x2(p0, p1);
  rs.l2 = f2_add(rs.l2, f2_pack(p0, p1));
  if (kInl) add_bf16_pair(rs.lr2, w);
  return w;
}

// 32 scores -> 16 packed bf16 pairs of p = 2^(s*sl2 - ref), written to TMEM
// columns [16*ch, 16*ch + 16) of the row and kept in pk; adds the chunk's p
// into `rs`.
template <bool kMask, bool kInl>
__device__ __forceinline__ void exp_chunk(const uint32_t (&r)[32], int ch, int vis_max,
                                          uint64_t sl2_2, uint64_t nref_2, RowSums& rs,
                                          uint32_t tS) {
  uint32_t pk[16];
#pragma unroll
  for (int x = 0; x < 16; ++x) {
    float s0 = __uint_as_float(r[2 * x]), s1 = __uint_as_float(r[2 * x + 1]);
    if (kMask) {
      if (ch * 32 + 2 * x > vis_max) s0 = -INFINITY;
      if (ch * 32 + 2 * x + 1 > vis_max) s1 = -INFINITY;
    }
    pk[x] = exp_pair<kInl>(s0, s1, sl2_2, nref_2, rs);
  }
  tmem_st16(tS + ch * 16, pk);
}

// A tile's (l, lr): on an unmasked tile lr is l itself.
template <bool kInl>
__device__ __forceinline__ float2 tile_sums(const RowSums& rs) {
  float lo, hi;
  f2_unpack(rs.l2, lo, hi);
  const float l = lo + hi;
  if (!kInl) return make_float2(l, l);
  f2_unpack(rs.lr2, lo, hi);
  return make_float2(l, lo + hi);
}

// Online max, speculative single pass over one S row of an unmasked tile:
// p = 2^(s*sl2 - m) against the row's current reference m, packed into
// registers (pk) and summed into rs, while the row maximum of the raw scores
// is tracked.  Nothing is written to TMEM, so if the maximum turns out to lie
// more than 64 (log2) above the reference the caller still has S to start
// over from.  (Masked tiles have their own single pass, spec_row_masked.)
__device__ __forceinline__ float spec_row(uint32_t tS, uint64_t sl2_2, uint64_t nref_2,
                                          uint32_t (&pk)[64], RowSums& rs) {
  uint32_t ra[32], rb[32];
  float mx = -INFINITY;
  auto chunk = [&](const uint32_t(&r)[32], int ch) {
    mx = chunk_max<false>(r, ch * 32, kBN - 1, mx);
#pragma unroll
    for (int x = 0; x < 16; ++x)
      pk[16 * ch + x] = exp_pair<false>(__uint_as_float(r[2 * x]), __uint_as_float(r[2 * x + 1]), sl2_2,
                                        nref_2, rs);
  };
  tmem_ld32(tS, ra);
  tmem_ld_wait();
  reg_fence(ra);
  tmem_ld32(tS + 32, rb);
  chunk(ra, 0);
  tmem_ld_wait();
  reg_fence(rb);
  tmem_ld32(tS + 64, ra);
  chunk(rb, 1);
  tmem_ld_wait();
  reg_fence(ra);
  tmem_ld32(tS + 96, rb);
  chunk(ra, 2);
  tmem_ld_wait();
  reg_fence(rb);
  chunk(rb, 3);
  return mx;
}

// Pass 2 over one S row: exp, row sums, P (bf16) back into TMEM and kept in
// pk, with the next 32-column load in flight while the current chunk is
// processed.  P block ch overwrites S columns [16ch, 16ch+16), which were
// already read.  Returns the tile's (l, lr) sums (lr only when kInl).
// A chunk of a masked tile, classified across the warp: where every row of
// the warp sees all 32 columns the unmasked code runs, where none sees any
// the chunk's P is zero (no exp, nothing summed), and only a chunk that the
// warp's visibility limits cross is masked element by element.  On a
// diagonal tile the limits of a warp's 32 consecutive rows span 32
// consecutive columns, so at most two of a row's four chunks are masked.
template <bool kInl>
__device__ __forceinline__ void exp_chunk_masked(const uint32_t (&r)[32], int ch, int vis_max,
                                                 uint64_t sl2_2, uint64_t nref_2, RowSums& rs,
                                                 uint32_t tS) {
  if (__all_sync(0xffffffffu, ch * 32 + 31 <= vis_max)) {
    exp_chunk<false, kInl>(r, ch, vis_max, sl2_2, nref_2, rs, tS);
  } else if (__all_sync(0xffffffffu, ch * 32 > vis_max)) {
    const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    tmem_st16(tS + ch * 16, z);
  } else {
    exp_chunk<true, kInl>(r, ch, vis_max, sl2_2, nref_2, rs, tS);
  }
}

// The chunk of a masked tile (kMask) or of an unmasked one.
template <bool kMask, bool kInl>
__device__ __forceinline__ void exp_chunk_any(const uint32_t (&r)[32], int ch, int vis_max,
                                              uint64_t sl2_2, uint64_t nref_2, RowSums& rs,
                                              uint32_t tS) {
  if (kMask)
    exp_chunk_masked<kInl>(r, ch, vis_max, sl2_2, nref_2, rs, tS);
  else
    exp_chunk<false, false>(r, ch, vis_max, sl2_2, nref_2, rs, tS);
}

// Pass 2 over one S row: exp, row sums, P (bf16) back into TMEM, with the
// next 32-column load in flight while the current chunk is processed.  P
// block ch overwrites S columns [16ch, 16ch+16), which were already read.
// Returns the tile's (l, lr) sums.
template <bool kMask, bool kInl = kMask>
__device__ __forceinline__ float2 exp_row_to_tmem(uint32_t tS, int vis_max, float sl2, float ref) {
  uint32_t ra[32], rb[32];
  const uint64_t sl2_2 = f2_pack(sl2, sl2), nref_2 = f2_pack(-ref, -ref);
  RowSums rs{f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
  tmem_ld32(tS, ra);
  tmem_ld_wait();
  reg_fence(ra);
  tmem_ld32(tS + 32, rb);
  exp_chunk_any<kMask, kInl>(ra, 0, vis_max, sl2_2, nref_2, rs, tS);
  tmem_ld_wait();
  reg_fence(rb);
  tmem_ld32(tS + 64, ra);
  exp_chunk_any<kMask, kInl>(rb, 1, vis_max, sl2_2, nref_2, rs, tS);
  tmem_ld_wait();
  reg_fence(ra);
  tmem_ld32(tS + 96, rb);
  exp_chunk_any<kMask, kInl>(ra, 2, vis_max, sl2_2, nref_2, rs, tS);
  tmem_ld_wait();
  reg_fence(rb);
  exp_chunk_any<kMask, kInl>(rb, 3, vis_max, sl2_2, nref_2, rs, tS);
  return tile_sums<kInl>(rs);
}

// O *= f for this thread's row, out of line: the deferred reference move of
// the online softmax is rare, and keeping its code out of the hot loop keeps
// that loop's instructions in the instruction cache.
__device__ __noinline__ void rescale_o_row(uint32_t tO, float f) {
#pragma unroll 1
  for (int ch = 0; ch < kD / 32; ++ch) {
    uint32_t r[32];
    tmem_ld32(tO + ch * 32, r);
    tmem_ld_wait();
    reg_fence(r);
#pragma unroll
    for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * f);
    tmem_st32(tO + ch * 32, r);
  }
  tmem_st_wait();
}

// The masked row passes, out of line: masked tiles are a few per cent of a
// causal problem's tiles, and keeping their code out of line keeps the loop
// over them compact (same-process A/B, when masked and unmasked tiles shared
// one loop: causal contiguous 22.03 -> 21.29 ms, striped 22.56 -> 22.11 ms,
// DCP prefill 10.67 -> 10.39 ms).  Const max runs every masked tile through
// the exp pass; online max runs both passes on a unit's first tile and on the
// rare tile whose maximum outruns the speculative pass.
__device__ __noinline__ float row_max_masked(uint32_t tS, int vis_max) {
  return row_max_from_tmem<true>(tS, vis_max);
}
__device__ __noinline__ float2 exp_row_masked(uint32_t tS, int vis_max, float sl2, float ref) {
  return exp_row_to_tmem<true, true>(tS, vis_max, sl2, ref);
}
// The same without the rounded row sum, for rows that see many keys in all.
__device__ __noinline__ float2 exp_row_masked_plain(uint32_t tS, int vis_max, float sl2, float ref) {
  return exp_row_to_tmem<true, false>(tS, vis_max, sl2, ref);
}

// Online max, speculative single pass over one S row of a masked tile (the
// masked counterpart of spec_row, inlined only into the loop over a unit's
// masked tiles): each 32-column chunk is classified across the warp as in
// exp_chunk_masked, p is formed against the current reference m and kept in
// registers while the visible maximum is tracked.  If no row of the warp has
// its maximum more than 64 (log2) above m, P is written to TMEM and (l, lr,
// pending reference move as int bits, 1) is returned; otherwise nothing is
// written and .w is 0, and the caller takes the two-pass path over the
// intact S.  lr sums the bf16-rounded p when kInl.
template <bool kInl>
__device__ __forceinline__ float4 spec_row_masked(uint32_t tS, int vis_max, float sl2, float m) {
  const uint64_t sl2_2 = f2_pack(sl2, sl2), nref_2 = f2_pack(-m, -m);
  RowSums rs{f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
  uint32_t pk[64];
  uint32_t ra[32], rb[32];
  float mx = -INFINITY;
  auto chunk = [&](const uint32_t(&r)[32], int ch) {
    if (__all_sync(0xffffffffu, ch * 32 + 31 <= vis_max)) {
      mx = chunk_max<false>(r, ch * 32, kBN - 1, mx);
#pragma unroll
      for (int x = 0; x < 16; ++x)
        pk[16 * ch + x] = exp_pair<kInl>(__uint_as_float(r[2 * x]), __uint_as_float(r[2 * x + 1]), sl2_2,
                                         nref_2, rs);
    } else if (__all_sync(0xffffffffu, ch * 32 > vis_max)) {
#pragma unroll
      for (int x = 0; x < 16; ++x) pk[16 * ch + x] = 0u;
    } else {
      mx = chunk_max<true>(r, ch * 32, vis_max, mx);
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        float s0 = __uint_as_float(r[2 * x]), s1 = __uint_as_float(r[2 * x + 1]);
        if (ch * 32 + 2 * x > vis_max) s0 = -INFINITY;
        if (ch * 32 + 2 * x + 1 > vis_max) s1 = -INFINITY;
        pk[16 * ch + x] = exp_pair<kInl>(s0, s1, sl2_2, nref_2, rs);
      }
    }
  };
  tmem_ld32(tS, ra);
  tmem_ld_wait();
  reg_fence(ra);
  tmem_ld32(tS + 32, rb);
  chunk(ra, 0);
  tmem_ld_wait();
  reg_fence(rb);
  tmem_ld32(tS + 64, ra);
  chunk(rb, 1);
  tmem_ld_wait();
  reg_fence(ra);
  tmem_ld32(tS + 96, rb);
  chunk(ra, 2);
  tmem_ld_wait();
  reg_fence(rb);
  chunk(rb, 3);
  const float jump = mx * sl2 - m;
  if (!__all_sync(0xffffffffu, !(jump > 64.f))) return make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) tmem_st16(tS + ch * 16, &pk[16 * ch]);
  const float2 t = tile_sums<kInl>(rs);
  const int pend = jump > kRescaleThreshold ? (int)ceilf(jump) : 0;
  return make_float4(t.x, t.y, __int_as_float(pend), 1.f);
}

// kConst: the const-max instantiation (no running maximum) or the online-max
// one; each compiles only its own softmax.  kMaskable: false for problems
// where no tile needs a mask (not causal, not segmented, shards of whole
// 128-key tiles), which then run without the masked softmax's code: on the
// DiT workload 3.353 -> 3.274 ms, online max 10.93 -> 10.41 ms, bit for bit
// the same output (the kernel is sensitive to the size of its hot code).
// kSegMode: 0 compiles the segmented schedule's branches out (the unmasked
// instantiations; online max 10.37 -> 10.12 ms), 1 decides them by P.seg.
// Compiling them out of the masked instantiations as well, with a third one
// for the segmented schedule, made causal and DCP prefill ~1 % slower.
template <bool kConst, bool kMaskable, int kSegMode>
__global__ void __launch_bounds__(kThreads, 1)
ring_tc_kernel(const __grid_constant__ TcMaps maps, const TcParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = (uint64_t*)(smem + kSmemBar);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  uint32_t* tmem_slot = (uint32_t*)(smem + kSmemTmemSlot);
  volatile int* abort_flag = (volatile int*)(smem + kSmemAbort);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  unsigned* err = P.a.err;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kNGroup; ++s) mbar_init(bar(kBarKvFull + s), 1);
    for (int s = 0; s < kNSlot; ++s) mbar_init(bar(kBarKvEmpty + s), 1);  // arrived by softmax warpgroup 1
    mbar_init(bar(kBarQFull), 1);
    // the Q tiles are released by softmax warpgroup 1 after the last S MMA
    // and, when the softmax warps read them for the row bounds, by each of
    // those eight warps too
    mbar_init(bar(kBarQEmpty), (P.a.mode == 1 && P.a.kmax2) ? 1 + 8 : 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarPFull + i), kBM);
      mbar_init(bar(kBarOFull + i), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tensormap(&maps.q);
    prefetch_tensormap(&maps.kv[0]);
    prefetch_tensormap(&maps.kv[1]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    int64_t kvh_of = 0;  // key/value head of the current unit (3-D maps)
    if (lane == 0) {
      uint32_t uc = 0;
      uint64_t pos = 0, gt = 0;
      uint64_t armed = 0;    // tile barriers armed so far (running tile index)
      uint32_t q_armed = 0;  // times q_full was armed
      bool ok = true;
      // wait until ring position `pos + d` is free
      auto slot_free = [&](uint64_t d) -> bool {
        const uint64_t p = pos + d;
        return mbar_wait(bar(kBarKvEmpty + (int)(p % kNSlot)), (uint32_t)(((p / kNSlot) & 1) ^ 1),
                         abort_flag, err);
      };
      // K (kv = 0) or V (kv = 1) tile kt of step `st` into ring position
      // `pos`, completing on barrier `fb`
      auto load_kv = [&](const Step& st, int kt, int kv, uint32_t fb) {
        const int slot = (int)(pos % kNSlot);
        const CUtensorMap* m = &maps.kv[2 * st.src + kv];
        const int krow = (int)(st.row0 + (int64_t)kt * kBN);
        for (int hx = 0; hx < 2; ++hx) {
          const uint32_t dst = sbase + kSmemKV + slot * kTileBytes + hx * kBoxBytes;
          if (kSegMode != 0 && P.seg)
            tma_load_3d(dst, m, fb, hx * 64, krow, (int)kvh_of);
          else
            tma_load_2d(dst, m, fb, hx * 64, krow);
        }
        ++pos;
      };
      // Every barrier is armed only once all slots its copies go to are
      // free, so an armed barrier always completes.
      for (int64_t k = 0, u = unit_at(P, 0); u < P.units && ok; ++k, u = unit_at(P, k)) {
        const Unit U = unit_of(P, u);
        const int n = unit_tiles<kSegMode>(P, U);
        if (n == 0) continue;
        kvh_of = U.bhk;
        ok = mbar_wait(bar(kBarQEmpty), (uc & 1) ^ 1, abort_flag, err) && slot_free(0);
        if (!ok) break;
        TileIter<kSegMode, kMaskable> it;
        it.begin(P, U);
        // Q tiles and K_0 on q_full
        mbar_arrive_expect_tx(bar(kBarQFull), 3 * kTileBytes);
        ++q_armed;
        for (int i = 0; i < 2; ++i)
          for (int hx = 0; hx < 2; ++hx)
            tma_load_2d(sbase + kSmemQ + i * kTileBytes + hx * kBoxBytes, &maps.q, bar(kBarQFull),
                        hx * 64, tile_qrow(P, U, i));
        load_kv(it.st, it.kt, 0, bar(kBarQFull));
        // the next unit's Q tiles come from HBM: start them towards L2 now
        if (unit_at(P, k + 1) < P.units) {
          const Unit N = unit_of(P, unit_at(P, k + 1));
          for (int i = 0; i < 2; ++i)
            for (int hx = 0; hx < 2; ++hx) tma_prefetch_2d(&maps.q, hx * 64, tile_qrow(P, N, i));
        }
        // V_j and K_(j+1) on the tile barrier of tile j.  The barrier's
        // previous phase (tile t - kNGroup) was waited for by the issuing
        // thread before it consumed the older tiles whose slots are free now.
        for (int j = 0; j < n; ++j) {
          const uint64_t t = gt + j;
          const uint32_t fb = bar(kBarKvFull + (int)(t % kNGroup));
          const Step stj = it.st;
          const int ktj = it.kt;
          it.next(P, U);
          const bool more = j + 1 < n;
          ok = slot_free(0) && (!more || slot_free(1));
          if (!ok) break;
          mbar_arrive_expect_tx(fb, (more ? 2u : 1u) * kTileBytes);
          ++armed;
          load_kv(stj, ktj, 1, fb);
          if (more) load_kv(it.st, it.kt, 0, fb);
        }
        gt += n;
        ++uc;
      }
      if (!ok) {
        // error path: let the copies already in flight land before exit
        volatile int never = 0;
        for (uint64_t t = armed > kNGroup ? armed - kNGroup : 0; t < armed; ++t)
          mbar_wait(bar(kBarKvFull + (int)(t % kNGroup)), (uint32_t)((t / kNGroup) & 1), &never, err);
        if (q_armed) mbar_wait(bar(kBarQFull), (q_armed - 1) & 1, &never, err);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the schedule, so every descriptor and TMEM
    // address stays warp-uniform; lane 0 alone issues the MMAs and commits.
    {
      uint32_t uc = 0;
      uint64_t pos = 0, gt = 0;
      bool ok = true;
      // base descriptors; a slot's tiles are kTileBytes (2048 units) apart
      const uint64_t qdesc0 = smem_desc_sw128(sbase + kSmemQ, 16, 1024);
      const uint64_t qdesc1 = smem_desc_sw128(sbase + kSmemQ + kTileBytes, 16, 1024);
      const uint64_t kvdesc = smem_desc_sw128(sbase + kSmemKV, 16, 1024);
      const uint64_t vdesc = smem_desc_sw128(sbase + kSmemKV, kBoxBytes, 1024);
      auto kd = [&](int slot) { return kvdesc + (uint64_t)(slot * (kTileBytes >> 4)); };
      auto vd = [&](int slot) { return vdesc + (uint64_t)(slot * (kTileBytes >> 4)); };
      const uint32_t tS0 = tmem + kColS, tS1 = tmem + kColS + 128, tO0 = tmem + kColO,
                     tO1 = tmem + kColO + 128;
      for (int64_t k = 0, u = unit_at(P, 0); u < P.units && ok; ++k, u = unit_at(P, k)) {
        const Unit U = unit_of(P, u);
        const int n = unit_tiles<kSegMode>(P, U);
        if (n == 0) continue;
        // Q tiles and K_0
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarQFull), uc & 1, abort_flag, err));
        if (!ok) break;
        tc_fence_after();
        int kslot = (int)(pos % kNSlot);
        issue_s(tS0, qdesc0, kd(kslot));
        tc_commit_lane0(bar(kBarSFull + 0));
        issue_s(tS1, qdesc1, kd(kslot));
        tc_commit_lane0(bar(kBarSFull + 1));
        ++pos;
        for (int j = 0; j < n && ok; ++j) {
          const int vslot = (int)(pos % kNSlot);
          // V_j and K_(j+1)
          const uint64_t t = gt + j;
          ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarKvFull + (int)(t % kNGroup)), (uint32_t)((t / kNGroup) & 1), abort_flag, err));
          if (!ok) break;
          const uint32_t pph = (uint32_t)((gt + j) & 1);
          ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarPFull + 0), pph, abort_flag, err));
          if (!ok) break;
          tc_fence_after();
          issue_pv(tO0, tS0, vd(vslot), j > 0);
          ++pos;
          const bool more = j + 1 < n;
          if (more) {
            kslot = (int)(pos % kNSlot);
            issue_s(tS0, qdesc0, kd(kslot));
            tc_commit_lane0(bar(kBarSFull + 0));
          } else {
            tc_commit_lane0(bar(kBarOFull + 0));
          }
          ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarPFull + 1), pph, abort_flag, err));
          if (!ok) break;
          tc_fence_after();
          issue_pv(tO1, tS1, vd(vslot), j > 0);
          if (more) {
            issue_s(tS1, qdesc1, kd(kslot));
            tc_commit_lane0(bar(kBarSFull + 1));
            ++pos;
          } else {
            tc_commit_lane0(bar(kBarOFull + 1));
          }
        }
        gt += n;
        ++uc;
      }
      if (!ok) {
        // error path: MMAs already issued still write TMEM; wait (bounded)
        // for all of them before the TMEM is freed
        tc_commit_lane0(bar(kBarDrain));
        volatile int never = 0;
        mbar_wait(bar(kBarDrain), 0, &never, err);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int i = warp / 4;                 // query tile of this warpgroup
    const int quarter = warp % 4;           // TMEM lane quarter
    const int tid = quarter * 32 + lane;    // row within the tile
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS + 128u * i;
    const uint32_t tO = tmem + lane_base + kColO + 128u * i;
    constexpr bool const_max = kConst;
    // Softmax warpgroup 1's first thread releases the K/V ring slots and the
    // Q tiles: the issuing thread commits s_full[1] after S1(j), which it
    // issues after S0(j), PV0(j-1) and PV1(j-1), so once s_full[1] of tile j
    // has completed, K_j, V_(j-1) and (on the last tile) Q are no longer read
    // by any MMA.  Moving these arrivals off the issuing thread saves it two
    // commits per tile.
    const bool releaser = (i == 1 && tid == 0);
    uint64_t kvpos = 0;  // ring position of K_0 of the current unit
    uint32_t uc = 0;
    uint64_t gt = 0;
    bool ok = true;
    for (int64_t k = 0, u = unit_at(P, 0); u < P.units && ok; ++k, u = unit_at(P, k)) {
      const Unit U = unit_of(P, u);
      const int n = unit_tiles<kSegMode>(P, U);
      const int64_t a_row = tile_row0(P, U, i) + tid;
      const bool valid = a_row < P.a.Ls;
      const int64_t orow = tile_bh(U, i) * P.a.Sq + (int64_t)U.r_store * P.a.Ls + a_row;
      if (n == 0) {
        if (valid) {
          if (P.a.out_f32) {
            float4* dst = (float4*)((float*)P.a.o + orow * kD);
            for (int c = 0; c < kD / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          } else {
            uint4* dst = (uint4*)((__nv_bfloat16*)P.a.o + orow * kD);
            for (int c = 0; c < kD / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          }
          if (P.a.lse) P.a.lse[orow] = -INFINITY;
        }
        continue;
      }
      // Rows that see few keys in all form the rounded sum on their masked
      // tiles (causal ring: a row sees its global position + 1 keys, else
      // all of them; the segmented and single-step schedules always do)
      bool few_keys = true;
      if (kMaskable && !P.seg && P.a.kv_rank_fixed < 0) {
        const int64_t keys = P.a.causal ? layout_global(P.a.layout, P.a.cp, P.a.Ls, U.r_log, a_row) + 1
                                        : (int64_t)P.a.cp * P.a.Ls;
        few_keys = __any_sync(0xffffffffu, valid && keys < kRoundedSumKeys);
      }
      float c_nat = 0.f;
      if (const_max && P.a.kmax2) {
        // the row's bound from its q row in the Q tile: |q|^2 summed in fp32
        // (the order of the 16-byte chunks is the swizzled one; a sum does
        // not care), c = sqrt(scale^2 * kmax2 * |q|^2)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarQFull), uc & 1, abort_flag, err));
        if (!ok) break;
        float ss = 0.f;
#pragma unroll
        for (int hx = 0; hx < 2; ++hx) {
          const uint4* row =
              reinterpret_cast<const uint4*>(smem + kSmemQ + i * kTileBytes + hx * kBoxBytes + tid * 128);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint4 w = row[ch];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float lo = __uint_as_float(ws[e] << 16), hi = __uint_as_float(ws[e] & 0xFFFF0000u);
              ss = fmaf(lo, lo, ss);
              ss = fmaf(hi, hi, ss);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarQEmpty));
        const float km = P.a.kmax2[U.bhk];
        c_nat = sqrtf(P.a.scale * P.a.scale * km * ss);
      } else if (const_max && valid) {
        c_nat = P.a.c[orow];
      }
      const float c_log2 = c_nat * kLog2e;
      float m = -INFINITY;  // reference max, log2 units (online mode)
      int pend = 0;         // reference move (log2 units) due before the next tile
      float l = 0.f;   // row sum of p as computed (log-sum-exp)
      float lr = 0.f;  // row sum of p rounded to bf16 (normalisation)
      // the key tile each softmax step is on: only the masked path needs it
      TileIter<kSegMode, kMaskable> it;
      if (kMaskable) it.begin(P, U);
      int64_t row_lim = 0;
      // one key tile; kM: the masked softmax compiled in (phase 1 tiles)
      auto tile = [&](int j, auto masked) -> bool {
        constexpr bool kM = decltype(masked)::value;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(kBarSFull + i), (uint32_t)((gt + j) & 1), abort_flag, err));
        if (!ok) return false;
        tc_fence_after();
        if (releaser) {
          const uint64_t kp = kvpos + 2 * (uint64_t)j;  // K_j
          mbar_arrive(bar(kBarKvEmpty + (int)(kp % kNSlot)));
          if (j > 0) mbar_arrive(bar(kBarKvEmpty + (int)((kp - 1) % kNSlot)));  // V_(j-1)
          if (j == n - 1) mbar_arrive(bar(kBarQEmpty));
        }
        // last visible column of this tile for this row
        int vis_max = kBN - 1;
        if constexpr (kM) {
          if (it.new_step) row_lim = step_row_limit<kSegMode>(P, it.st, a_row);
          const int64_t lim = row_lim - (int64_t)it.kt * kBN;
          vis_max = (int)max((int64_t)-1, min(lim, (int64_t)(kBN - 1)));
        }
        const bool need_mask = kM && __any_sync(0xffffffffu, vis_max < kBN - 1);
        // O *= f for this row (online max: the reference moved up)
        auto rescale_o = [&](float f) {
#pragma unroll 1
          for (int ch = 0; ch < kD / 32; ++ch) {
            uint32_t r[32];
            tmem_ld32(tO + ch * 32, r);
            tmem_ld_wait();
            reg_fence(r);
#pragma unroll
            for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * f);
            tmem_st32(tO + ch * 32, r);
          }
          tmem_st_wait();
        };
        float mref;
        bool p_done = false;  // P already in TMEM and its sums in tl, tlr
        float tl = 0.f, tlr = 0.f;  // the tile's l and lr
        if (!const_max && __any_sync(0xffffffffu, pend > 0)) {
          // the reference move left by the previous tile (whose PV has
          // completed: it precedes this tile's S in the MMA order)
          const float fac = pend > 0 ? __int_as_float((127 - pend) << 23) : 1.f;
          rescale_o_row(tO, fac);
          l *= fac;
          lr *= fac;
          m += (float)pend;
          pend = 0;
        }
        if (const_max) {
          mref = c_log2;
        } else if (need_mask && j > 0 && !__any_sync(0xffffffffu, m == -INFINITY)) {
          // a masked tile after the first: the single pass, with the mask
          const float4 r = few_keys ? spec_row_masked<true>(tS, vis_max, P.scale_log2, m)
                                    : spec_row_masked<false>(tS, vis_max, P.scale_log2, m);
          if (r.w != 0.f) {
            tl = r.x;
            tlr = r.y;
            pend = __float_as_int(r.z);
            p_done = true;
          }
          mref = m;
        } else if (!need_mask && j > 0 && !__any_sync(0xffffffffu, m == -INFINITY)) {
          // within a unit the row maximum rarely moves past the lazy-rescale
          // threshold: try the single pass against the current reference
          const uint64_t sl2_2 = f2_pack(P.scale_log2, P.scale_log2), nref_2 = f2_pack(-m, -m);
          RowSums rs{f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
          uint32_t pk[64];
          const float mx = spec_row(tS, sl2_2, nref_2, pk, rs);
          // how far the tile's maximum lies above the reference.  Up to 64
          // (log2) this tile's P, l and O stay far from fp32 overflow against
          // the old reference, so P is kept; past the lazy-rescale threshold
          // the reference then moves up by a whole number of log2 units
          // before the next tile (O, l scale by an exact power of two)
          const float jump = mx * P.scale_log2 - m;
          if (__all_sync(0xffffffffu, !(jump > 64.f))) {
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) tmem_st16(tS + ch * 16, &pk[16 * ch]);
            const float2 t = tile_sums<false>(rs);
            tl = t.x;
            tlr = t.y;
            if (jump > kRescaleThreshold) pend = (int)ceilf(jump);  // 49 .. 64
            p_done = true;
          }
          mref = m;
        }
        if (!const_max && !p_done) {
          // pass 1: row maximum straight from TMEM; the next 32-column load is
          // in flight while the current one is reduced
          float mx = need_mask ? row_max_masked(tS, vis_max) : row_max_from_tmem<false>(tS, vis_max);
          mx *= P.scale_log2;
          float fac = 1.f;
          bool need_o = false;
          if (mx > m + kRescaleThreshold || (m == -INFINITY && mx != -INFINITY)) {
            fac = (m == -INFINITY) ? 0.f : ex2(m - mx);
            need_o = (m != -INFINITY) && (j > 0);
            l *= fac;
            lr *= fac;
            m = mx;
          }
          if (__any_sync(0xffffffffu, need_o)) rescale_o(need_o ? fac : 1.f);
          mref = (m == -INFINITY) ? 0.f : m;
        }
        // pass 2: p = 2^(s*scale*log2e - ref), row sum, bf16 P written over
        // the S columns already consumed (P column block ch < S block ch+1)
        if (!p_done) {
          const float2 t = need_mask ? (few_keys ? exp_row_masked(tS, vis_max, P.scale_log2, mref)
                                                 : exp_row_masked_plain(tS, vis_max, P.scale_log2, mref))
                                     : exp_row_to_tmem<false>(tS, vis_max, P.scale_log2, mref);
          tl = t.x;
          tlr = t.y;
        }
        l += tl;
        lr += tlr;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + i));
        if (kMaskable) it.next(P, U);
        return true;
      };
      int j = 0;
      if (kMaskable)
        for (; j < n && it.phase == 0; ++j)
          if (!tile(j, std::false_type{})) break;
      if (ok)
        for (; j < n; ++j)
          if (!tile(j, std::integral_constant<bool, kMaskable>{})) break;
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarOFull + i), uc & 1, abort_flag, err));
      if (!ok) break;
      tc_fence_after();
      if (releaser) mbar_arrive(bar(kBarKvEmpty + (int)((kvpos + 2 * (uint64_t)n - 1) % kNSlot)));  // V_(n-1)
      kvpos += 2 * (uint64_t)n;
      // O is divided by the sum of the weights it was accumulated with (lr);
      // the log-sum-exp comes from the unrounded sum l.  An unnormalised
      // const-max partial carries O * l / lr, so that the merge, which
      // divides by the steps' summed l, still gives each step's O / lr its
      // weight l.
      float inv, lse;
      if (const_max) {
        inv = P.a.unnormalized ? (lr > 0.f ? l / lr : 1.f) : 1.f / fmaxf(lr, 1e-37f);
        lse = c_nat + logf(l);
      } else if (l > 0.f) {
        inv = 1.f / lr;
        lse = (m + log2f(l)) * kLn2;
      } else {
        inv = 0.f;
        lse = -INFINITY;
      }
      // the output row: the next 32 columns load from TMEM while the current
      // ones are scaled, transposed inside lane quads and stored
      {
        const int qd = lane & 3;
        uint32_t ra[32], rb[32];
        auto emit = [&](const uint32_t(&r)[32], int ch) {
          if (P.a.out_f32) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint4 a4[4];
#pragma unroll
              for (int x = 0; x < 4; ++x)
                a4[x] = make_uint4(__float_as_uint(__uint_as_float(r[16 * h + 4 * x]) * inv),
                                   __float_as_uint(__uint_as_float(r[16 * h + 4 * x + 1]) * inv),
                                   __float_as_uint(__uint_as_float(r[16 * h + 4 * x + 2]) * inv),
                                   __float_as_uint(__uint_as_float(r[16 * h + 4 * x + 3]) * inv));
              quad_transpose(a4, lane);
#pragma unroll
              for (int x = 0; x < 4; ++x)
                if (a_row - qd + x < P.a.Ls)
                  *(uint4*)((float*)P.a.o + (orow - qd + x) * kD + ch * 32 + h * 16 + qd * 4) = a4[x];
            }
          } else {
            uint4 a4[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              uint32_t w[4];
#pragma unroll
              for (int y = 0; y < 4; ++y)
                w[y] = pack_bf16x2(__uint_as_float(r[8 * x + 2 * y]) * inv,
                                   __uint_as_float(r[8 * x + 2 * y + 1]) * inv);
              a4[x] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            quad_transpose(a4, lane);
#pragma unroll
            for (int x = 0; x < 4; ++x)
              if (a_row - qd + x < P.a.Ls)
                *(uint4*)((__nv_bfloat16*)P.a.o + (orow - qd + x) * kD + ch * 32 + qd * 8) = a4[x];
          }
        };
        tmem_ld32(tO, ra);
        tmem_ld_wait();
        reg_fence(ra);
        tmem_ld32(tO + 32, rb);
        emit(ra, 0);
        tmem_ld_wait();
        reg_fence(rb);
        tmem_ld32(tO + 64, ra);
        emit(rb, 1);
        tmem_ld_wait();
        reg_fence(ra);
        tmem_ld32(tO + 96, rb);
        emit(ra, 2);
        tmem_ld_wait();
        reg_fence(rb);
        emit(rb, 3);
      }
      if (valid && P.a.lse) P.a.lse[orow] = lse;
      gt += n;
      ++uc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

template <bool kConst, bool kMaskable, int kSegMode>
static cudaError_t launch_tc_mode(const TcMaps& maps, const TcParams& P, cudaStream_t stream) {
  static std::atomic<int> attr_set[64];  // idempotent once-per-device setup
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(ring_tc_kernel<kConst, kMaskable, kSegMode>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  const int sms = device_sm_count();
  const int64_t grid = P.units < sms ? P.units : sms;
  ring_tc_kernel<kConst, kMaskable, kSegMode><<<(unsigned)grid, kThreads, kSmemAlloc, stream>>>(maps, P);
  return cudaGetLastError();
}

// A tile needs a mask only under a causal limit, in the segmented schedule or
// at a shard end that is not a whole 128-key tile; other problems take the
// instantiation without the masked softmax.
static cudaError_t launch_tc(const TcMaps& maps, const TcParams& P, cudaStream_t stream) {
  const bool maskable = P.a.causal || P.seg || P.a.Ls % kBN != 0;
  if (P.a.mode == 1)
    return maskable ? launch_tc_mode<true, true, 1>(maps, P, stream)
                    : launch_tc_mode<true, false, 0>(maps, P, stream);
  return maskable ? launch_tc_mode<false, true, 1>(maps, P, stream)
                  : launch_tc_mode<false, false, 0>(maps, P, stream);
}

static void init_common(TcParams& P, const RingArgs& a) {
  P.a = a;
  P.hp = (a.Hq / a.Hkv) % 2 == 0;
  P.unit_rows = P.hp ? kBM : kUnitRows;
  P.qblocks = (int)((a.Ls + P.unit_rows - 1) / P.unit_rows);
  P.per_head = (int64_t)a.q_shards * P.qblocks;
  P.units = (int64_t)a.B * (P.hp ? a.Hq / 2 : a.Hq) * P.per_head;
  P.nkt = (int)((a.Ls + kBN - 1) / kBN);
  P.scale_log2 = a.scale * kLog2e;
  P.seg = 0;
  P.W = 1;
  P.I = 1;
  P.part_rank = -1;
  for (int r = 0; r < kMaxRanks; ++r) P.lp[r] = P.lc[r] = 0;
}

cudaError_t launch_ring_tc_bf16(const RingArgs& a, cudaStream_t stream) {
  if (a.D != kD) return cudaErrorInvalidValue;
  TcParams P;
  init_common(P, a);
  P.nsteps = a.kv_rank_fixed >= 0 ? 1 : a.cp;
  if (P.units == 0) return cudaSuccess;
  TcMaps maps;
  if (!encode_bf16_2d_sw128(&maps.q, a.q, (uint64_t)a.B * a.Hq * a.Sq, kD, kBM, 64) ||
      !encode_bf16_2d_sw128(&maps.kv[0], a.k, (uint64_t)a.B * a.Hkv * a.Sk, kD, kBN, 64) ||
      !encode_bf16_2d_sw128(&maps.kv[1], a.v, (uint64_t)a.B * a.Hkv * a.Sk, kD, kBN, 64))
    return cudaErrorInvalidValue;
  return launch_tc(maps, P, stream);
}

cudaError_t launch_dcp_prefill_tc(const DcpPrefillArgs& d, cudaStream_t stream) {
  static_assert(kDcpPrefillMaxRanks == kMaxRanks, "rank limit");
  if (d.D != kD || d.W < 1 || d.W > kMaxRanks) return cudaErrorInvalidValue;
  RingArgs a;
  a.q = d.q;
  a.k = nullptr;
  a.v = nullptr;
  a.B = 1;
  a.Hq = d.Hq;
  a.Hkv = d.Hkv;
  a.D = d.D;
  a.Sq = d.Sc;
  a.Sk = 0;
  a.Ls = d.Sc;
  a.cp = 1;
  a.q_shards = 1;
  a.q_rank_fixed = 0;
  a.kv_rank_fixed = -1;
  a.causal = 0;  // causality comes from the segments' global positions
  a.layout = 0;
  a.mode = 0;
  a.scale = d.scale;
  a.c = nullptr;
  a.o = d.o;
  a.out_f32 = d.out_f32;
  a.unnormalized = 0;
  a.lse = d.lse;
  a.err = d.err;
  TcParams P;
  init_common(P, a);
  P.seg = 1;
  P.W = d.W;
  P.I = d.I;
  P.part_rank = d.part_rank;
  P.nsteps = d.part_rank >= 0 ? 2 : 2 * d.W;
  if (P.units == 0) return cudaSuccess;
  TcMaps maps;
  if (!encode_bf16_2d_sw128(&maps.q, d.q, (uint64_t)d.Hq * d.Sc, kD, kBM, 64))
    return cudaErrorInvalidValue;
  for (int r = 0; r < d.W; ++r) {
    P.lp[r] = dcp_local_filled(d.P, d.W, d.I, d.I, r);
    P.lc[r] = dcp_local_filled(d.Sc, d.W, d.I, d.I, r);
    if (P.lp[r] > d.Lcap) P.lp[r] = d.Lcap;
    if (P.lc[r] > d.Lc) P.lc[r] = d.Lc;
    const uint64_t rp = P.lp[r] > 0 ? (uint64_t)P.lp[r] : 1, rc = P.lc[r] > 0 ? (uint64_t)P.lc[r] : 1;
    const char* kp = (const char*)d.k_prior + (size_t)r * d.Hkv * d.Lcap * d.D * 2;
    const char* vp = (const char*)d.v_prior + (size_t)r * d.Hkv * d.Lcap * d.D * 2;
    const char* kc = (const char*)d.k_cur + (size_t)r * d.Hkv * d.Lc * d.D * 2;
    const char* vc = (const char*)d.v_cur + (size_t)r * d.Hkv * d.Lc * d.D * 2;
    if (!encode_bf16_3d_sw128(&maps.kv[4 * r + 0], kp, d.Hkv, rp, kD, (uint64_t)d.Lcap * kD, kBN, 64) ||
        !encode_bf16_3d_sw128(&maps.kv[4 * r + 1], vp, d.Hkv, rp, kD, (uint64_t)d.Lcap * kD, kBN, 64) ||
        !encode_bf16_3d_sw128(&maps.kv[4 * r + 2], kc, d.Hkv, rc, kD, (uint64_t)d.Lc * kD, kBN, 64) ||
        !encode_bf16_3d_sw128(&maps.kv[4 * r + 3], vc, d.Hkv, rc, kD, (uint64_t)d.Lc * kD, kBN, 64))
      return cudaErrorInvalidValue;
  }
  return launch_tc(maps, P, stream);
}

}  // namespace ca
