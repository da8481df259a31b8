// index_maps.cuh -- closed-form index maps of context parallelism, shared by
// the host API and the kernels (__host__ __device__, integer only, bit-exact).
//
// Layouts of the virtual shards ("Context Parallelism in vLLM Omni Neuron",
// section "Model Implementation": rank r holds tokens [r*local_S,
// (r+1)*local_S); "Sharding the Input", striped attention: token t goes to
// device t mod cp).  Storage is shard-major: row r*Ls + a is local token a of
// shard r.
//
// DCP interleave ("DCP (Decode Context Parallelism)", sections "Slot Mapping
// and KV Cache", "local_filled Computation", "Active Token Handling and
// dcp_active_mask", "Segmented Attention CP"): blocks of I tokens are dealt to
// W ranks round robin; local slot s of rank R is global (s/I)*(W*I) + R*I +
// s%I.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define CA_HD __host__ __device__ __forceinline__
#else
#define CA_HD inline
#endif

namespace ca {

enum { kLayoutContiguous = 0, kLayoutStriped = 1 };

// Global token position of stored row (r, a).
CA_HD int64_t layout_global(int layout, int cp, int64_t Ls, int r, int64_t a) {
  return layout == kLayoutStriped ? a * cp + r : (int64_t)r * Ls + a;
}

// Stored (shard, local) of a global token.
CA_HD void layout_locate(int layout, int cp, int64_t Ls, int64_t t, int* r,
                         int64_t* a) {
  if (layout == kLayoutStriped) {
    *r = (int)(t % cp);
    *a = t / cp;
  } else {
    *r = (int)(t / Ls);
    *a = t % Ls;
  }
}

// Ring schedule: shard met by `rank` at `step`.
CA_HD int ring_kv_shard(int rank, int step, int cp) {
  int s = (rank - step) % cp;
  return s < 0 ? s + cp : s;
}

// Causal rule between the queries of shard r and the keys of shard s, as a
// threshold on local indices: key b is visible to query a iff b <= a - delta.
//   contiguous: s < r -> every key (delta = -inf), s > r -> none (+inf),
//               s == r -> b <= a (delta = 0);
//   striped:    global b*cp + s <= a*cp + r  <=>  b <= a - (s > r ? 1 : 0).
// kDeltaAll / kDeltaNone stand for -inf / +inf.
constexpr int64_t kDeltaAll = -(int64_t(1) << 62);
constexpr int64_t kDeltaNone = (int64_t(1) << 62);
CA_HD int64_t causal_delta(int layout, int r, int s) {
  if (layout == kLayoutStriped) return s > r ? 1 : 0;
  if (s < r) return kDeltaAll;
  if (s > r) return kDeltaNone;
  return 0;
}

// DCP ownership and local slots.
CA_HD int dcp_owner(int64_t pos, int W, int I) { return (int)((pos / I) % W); }
CA_HD int64_t dcp_local_index(int64_t pos, int W, int I) {
  return (pos / ((int64_t)W * I)) * I + pos % I;
}
CA_HD int64_t dcp_local_to_global(int64_t s, int R, int W, int I) {
  return (s / I) * ((int64_t)W * I) + (int64_t)R * I + s % I;
}

// local_filled, evaluated as the DCP page prints it.  T is the integer type
// of the arithmetic: int64_t on the host; the decode kernel takes int, whose
// divisions cost a tenth of 64-bit ones, for its positions are below 2^31
// (the host rejects caches of 2^31 rows or more).
template <typename T>
CA_HD T dcp_local_filled_t(T N, T W, T I, T block_size, T R) {
  const T vblock = block_size * W;
  const T stride = I * W;
  const T rank_start = R * I;
  T filled = (N / vblock) * block_size;
  const T remaining = N - (N / vblock) * vblock;
  filled += (remaining / stride) * I;
  const T leftover = remaining - (remaining / stride) * stride;
  T extra = leftover - rank_start;
  if (extra < 0) extra = 0;
  if (extra > I) extra = I;
  return filled + extra;
}
CA_HD int64_t dcp_local_filled(int64_t N, int W, int I, int block_size, int R) {
  return dcp_local_filled_t<int64_t>(N, W, I, block_size, R);
}

// Slots of ring-layout shard r (Ls rows) that hold one of the global
// positions [0, N): contiguous shard r holds [r*Ls, (r+1)*Ls); striped shard
// r holds r, r + cp, r + 2 cp, ... ("Sharding the Input").  T as above.
template <typename T>
CA_HD T ring_shard_filled_t(T N, T cp, T Ls, int layout, T r) {
  T n;
  if (layout == kLayoutStriped)
    n = N > r ? (N - r + cp - 1) / cp : 0;
  else
    n = N - r * Ls;
  if (n < 0) n = 0;
  if (n > Ls) n = Ls;
  return n;
}
CA_HD int64_t ring_shard_filled(int64_t N, int cp, int64_t Ls, int layout, int r) {
  return ring_shard_filled_t<int64_t>(N, cp, Ls, layout, r);
}

// dcp_active_mask as the DCP page prints it.
CA_HD int dcp_active_mask(int64_t N, int W, int I, int block_size, int R) {
  const int64_t vblock = (int64_t)block_size * W;
  const int64_t pos_in_vblock = N - (N / vblock) * vblock;
  const int owner = (int)((pos_in_vblock / I) % W);
  return owner == R ? 1 : 0;
}

}  // namespace ca
