/*
 * oracle.c -- plain, slow, fp64 CPU oracle for context-parallel attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no source,
 * header, table or helper with the CUDA library in context_attention_gb300/,
 * and the CUDA library never calls it.
 *
 * Every value is computed in double precision from the stored input values
 * (fp32 arrays; bf16 inputs are passed already widened, which is exact).
 * Nothing here is blocked, fused or reordered beyond what the definitions
 * below state: each function is the definition written out.
 *
 * Sources (pages on context parallelism):
 *  - "Kernel reference: ring_attention_const_max_fwd", sections "Overview"
 *    (ring schedule, step t on rank r uses the K/V of rank r-t), "Picking a
 *    max that is safe without measuring it" (c_i = scale*|q_i|*max_j|k_j|),
 *    "A static bound makes the ring reduction pure addition" and "Accumulate,
 *    then normalize once" (unnormalised sums, clamp 1e-37, lse = c + log sum).
 *  - "DCP (Decode Context Parallelism)", sections "Decode Compute Pattern"
 *    (partial attention + LSE, weight_i = exp(local_lse - global_lse)),
 *    "local_filled Computation", "Active Token Handling and dcp_active_mask",
 *    "Slot Mapping and KV Cache" (block b of I tokens lives on rank b mod W)
 *    and "Segmented Attention CP" (local slot s -> global (s//I)*(W*I)+R*I+s%I;
 *    chunked prefill against prior + current local KV, causal by global
 *    position, then the LSE merge).
 *  - "Sharding the Input" (striped layout: token t on device t mod cp;
 *    causal masking: a later token never influences an earlier one; Ring
 *    Pass-Q decode: the query visits the shards of the cache, partials are
 *    merged).
 *  - "Context Parallelism in vLLM Omni Neuron", section "Self-Attention with
 *    Context Parallelism" (q/k norm over the whole hidden, head split,
 *    rotary embedding at each token's position).
 *
 * Parity pins: every function here is pinned by the not-gpu tests in
 * tests/test_oracle_pins.py and tests/test_index_maps.py (closed forms,
 * invariants, brute force on tiny inputs, the pages' worked examples), and
 * its independent routes are cross-checked on random shapes in
 * tests/test_oracle_fuzz.py.  No function is left "parity unpinned".
 *
 * Row conventions.  q is [B, Hq, S, D], k and v are [B, Hkv, S, D], all
 * row-major.  The S rows of a head are stored shard-major: row rho = r*Ls + a
 * is local token a of virtual shard r (Ls = S / cp).  Its global token
 * position is rho for the contiguous layout and a*cp + r for the striped one.
 * Query head h reads key/value head h / (Hq/Hkv).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORA_LAYOUT_CONTIGUOUS 0
#define ORA_LAYOUT_STRIPED 1

/* Zero-filled allocation that stops the process with a message when memory
 * runs out, so that a failed allocation can never pass for a result. */
static void *ora_alloc(size_t count, size_t size) {
  void *p = calloc(count ? count : 1, size);
  if (!p) {
    fprintf(stderr, "oracle: out of memory (%zu x %zu bytes)\n", count, size);
    abort();
  }
  return p;
}

/* Global token position of stored row rho (see the row conventions above).
 * Contiguous: shard r holds tokens [r*Ls, (r+1)*Ls) in order.
 * Striped: token t is dealt to shard t mod cp as its (t div cp)-th token. */
static int64_t global_pos(int layout, int cp, int64_t Ls, int64_t rho) {
  int64_t r = rho / Ls, a = rho % Ls;
  if (layout == ORA_LAYOUT_STRIPED) return a * cp + r;
  return r * Ls + a;
}

/* Exported form of global_pos, for the index-map pins. */
int64_t ora_global_pos(int layout, int cp, int64_t Ls, int64_t rho) {
  return global_pos(layout, cp, Ls, rho);
}

/* One query row against the keys with stored index in [k_begin, k_end) that
 * the causal rule allows.  Writes the normalised output and the natural-log
 * LSE (scale included).  Empty allowed set: o = 0, lse = -inf. */
static void attend_row(const float *qrow, const float *kh, const float *vh,
                       int64_t S, int D, double scale, int causal, int layout,
                       int cp, int64_t qrho, int64_t k_begin, int64_t k_end,
                       double *orow, double *lse_out) {
  int64_t Ls = S / cp;
  int64_t qpos = global_pos(layout, cp, Ls, qrho);
  double *s = (double *)ora_alloc((size_t)(k_end - k_begin + 1), sizeof(double));
  double m = -INFINITY;
  for (int64_t j = k_begin; j < k_end; ++j) {
    int allowed = 1;
    if (causal) allowed = global_pos(layout, cp, Ls, j) <= qpos;
    if (!allowed) {
      s[j - k_begin] = -INFINITY;
      continue;
    }
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += (double)qrow[d] * (double)kh[j * D + d];
    s[j - k_begin] = scale * dot;
    if (s[j - k_begin] > m) m = s[j - k_begin];
  }
  for (int d = 0; d < D; ++d) orow[d] = 0.0;
  if (m == -INFINITY) {
    *lse_out = -INFINITY;
    free(s);
    return;
  }
  double l = 0.0;
  for (int64_t j = k_begin; j < k_end; ++j) {
    double sj = s[j - k_begin];
    if (sj == -INFINITY) continue;
    double p = exp(sj - m);
    l += p;
    for (int d = 0; d < D; ++d) orow[d] += p * (double)vh[j * D + d];
  }
  for (int d = 0; d < D; ++d) orow[d] /= l;
  *lse_out = m + log(l);
  free(s);
}

/* Full softmax attention for selected rows.  rows[i] is the flat row id
 * (b*Hq + h)*S + rho.  o is [nrows, D], lse is [nrows]. */
void ora_attention_rows(const float *q, const float *k, const float *v, int B,
                        int Hq, int Hkv, int64_t S, int D, double scale,
                        int causal, int layout, int cp, const int64_t *rows,
                        int64_t nrows, double *o, double *lse) {
  int G = Hq / Hkv;
  (void)B;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t id = rows[i];
    int64_t rho = id % S;
    int64_t bh = id / S;
    int64_t b = bh / Hq, h = bh % Hq;
    int64_t bk = b * Hkv + h / G;
    attend_row(q + id * D, k + bk * S * D, v + bk * S * D, S, D, scale, causal,
               layout, cp, rho, 0, S, o + i * D, lse + i);
  }
}

/* Partial attention of selected rows against the keys of one virtual shard
 * (stored rows [s*Ls, (s+1)*Ls)), with the same causal rule.  This is one ring
 * step's partial result (o_s normalised over the shard, lse_s). */
void ora_shard_partial_rows(const float *q, const float *k, const float *v,
                            int B, int Hq, int Hkv, int64_t S, int D,
                            double scale, int causal, int layout, int cp,
                            int kv_shard, const int64_t *rows, int64_t nrows,
                            double *o, double *lse) {
  int G = Hq / Hkv;
  int64_t Ls = S / cp;
  (void)B;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t id = rows[i];
    int64_t rho = id % S;
    int64_t bh = id / S;
    int64_t b = bh / Hq, h = bh % Hq;
    int64_t bk = b * Hkv + h / G;
    attend_row(q + id * D, k + bk * S * D, v + bk * S * D, S, D, scale, causal,
               layout, cp, rho, (int64_t)kv_shard * Ls,
               (int64_t)(kv_shard + 1) * Ls, o + i * D, lse + i);
  }
}

/* LSE merge of n partials (DCP page, decode steps 5-7):
 *   M = max_i lse_i (partials with lse = -inf are skipped),
 *   L = M + ln sum_i exp(lse_i - M),
 *   o = sum_i exp(lse_i - L) * o_i.
 * All partials empty: o = 0, L = -inf.
 * o_parts is [n, nrows, D], lse_parts is [n, nrows]. */
void ora_lse_merge(const double *o_parts, const double *lse_parts, int n,
                   int64_t nrows, int D, double *o, double *lse) {
#pragma omp parallel for
  for (int64_t r = 0; r < nrows; ++r) {
    double M = -INFINITY;
    for (int i = 0; i < n; ++i)
      if (lse_parts[(int64_t)i * nrows + r] > M) M = lse_parts[(int64_t)i * nrows + r];
    for (int d = 0; d < D; ++d) o[r * D + d] = 0.0;
    if (M == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double acc = 0.0;
    for (int i = 0; i < n; ++i) {
      double li = lse_parts[(int64_t)i * nrows + r];
      if (li == -INFINITY) continue;
      acc += exp(li - M);
    }
    double L = M + log(acc);
    for (int i = 0; i < n; ++i) {
      double li = lse_parts[(int64_t)i * nrows + r];
      if (li == -INFINITY) continue;
      double w = exp(li - L);
      for (int d = 0; d < D; ++d)
        o[r * D + d] += w * o_parts[((int64_t)i * nrows + r) * D + d];
    }
    lse[r] = L;
  }
}

/* Const-max bound (const-max page, "Picking a max ..." and "Assembling the
 * bound"): kmax2[b, hk] = max over ALL S keys of the head of |k_j|^2, and
 * c[b, h, rho] = scale * |q_rho| * sqrt(kmax2[b, h / G]).
 * c is [B, Hq, S], kmax2 is [B, Hkv]. */
void ora_const_max_bound(const float *q, const float *k, int B, int Hq, int Hkv,
                         int64_t S, int D, double scale, double *c,
                         double *kmax2) {
  int G = Hq / Hkv;
  for (int64_t bk = 0; bk < (int64_t)B * Hkv; ++bk) {
    double mx = 0.0;
    for (int64_t j = 0; j < S; ++j) {
      double n2 = 0.0;
      for (int d = 0; d < D; ++d) {
        double x = (double)k[(bk * S + j) * D + d];
        n2 += x * x;
      }
      if (n2 > mx) mx = n2;
    }
    kmax2[bk] = mx;
  }
#pragma omp parallel for
  for (int64_t id = 0; id < (int64_t)B * Hq * S; ++id) {
    int64_t bh = id / S;
    int64_t b = bh / Hq, h = bh % Hq;
    double n2 = 0.0;
    for (int d = 0; d < D; ++d) {
      double x = (double)q[id * D + d];
      n2 += x * x;
    }
    c[id] = scale * sqrt(n2) * sqrt(kmax2[b * Hkv + h / G]);
  }
}

/* Ring attention for selected rows, step by step as the const-max page's
 * "Overview" draws it: query row rho lives on shard r = rho / Ls and, at ring
 * step t = 0..cp-1, meets the keys of shard (r - t) mod cp.
 *
 * mode 0 (online max): each step gives a normalised partial (o_t, lse_t) and
 *   the partials are LSE-merged in ring order (the merge above).
 * mode 1 (const max): with the bound c (array [B,Hq,S] from
 *   ora_const_max_bound), every step adds its unnormalised sums
 *   acc_o += sum_j exp(s_j - c) v_j and acc_l += sum_j exp(s_j - c); at the
 *   end o = acc_o / max(acc_l, 1e-37) and lse = c + ln(acc_l).
 *
 * overshoot (nullable, [nrows]) receives c - max_j s_j in const mode (the
 * number of nats by which the bound exceeds the row's true maximum); the
 * page says rows whose overshoot passes ~85 nats underflow in fp32. */
void ora_ring_rows(const float *q, const float *k, const float *v, int B,
                   int Hq, int Hkv, int64_t S, int D, double scale, int causal,
                   int layout, int cp, int mode, const double *c,
                   const int64_t *rows, int64_t nrows, double *o, double *lse,
                   double *overshoot) {
  int G = Hq / Hkv;
  int64_t Ls = S / cp;
  (void)B;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t id = rows[i];
    int64_t rho = id % S;
    int64_t bh = id / S;
    int64_t b = bh / Hq, h = bh % Hq;
    int64_t bk = b * Hkv + h / G;
    const float *qrow = q + id * D;
    const float *kh = k + bk * S * D;
    const float *vh = v + bk * S * D;
    int r = (int)(rho / Ls);
    int64_t qpos = global_pos(layout, cp, Ls, rho);
    double *orow = o + i * D;
    if (mode == 0) {
      double *op = (double *)ora_alloc((size_t)cp * D, sizeof(double));
      double *lp = (double *)ora_alloc((size_t)cp, sizeof(double));
      for (int t = 0; t < cp; ++t) {
        int s = ((r - t) % cp + cp) % cp;
        attend_row(qrow, kh, vh, S, D, scale, causal, layout, cp, rho,
                   (int64_t)s * Ls, (int64_t)(s + 1) * Ls, op + (int64_t)t * D,
                   lp + t);
      }
      /* merge of cp partials for this one row */
      double M = -INFINITY;
      for (int t = 0; t < cp; ++t)
        if (lp[t] > M) M = lp[t];
      for (int d = 0; d < D; ++d) orow[d] = 0.0;
      if (M == -INFINITY) {
        lse[i] = -INFINITY;
      } else {
        double acc = 0.0;
        for (int t = 0; t < cp; ++t)
          if (lp[t] != -INFINITY) acc += exp(lp[t] - M);
        double L = M + log(acc);
        for (int t = 0; t < cp; ++t) {
          if (lp[t] == -INFINITY) continue;
          double w = exp(lp[t] - L);
          for (int d = 0; d < D; ++d) orow[d] += w * op[(int64_t)t * D + d];
        }
        lse[i] = L;
      }
      if (overshoot) overshoot[i] = NAN;
      free(op);
      free(lp);
    } else {
      double ci = c[id];
      double acc_l = 0.0, smax = -INFINITY;
      for (int d = 0; d < D; ++d) orow[d] = 0.0;
      for (int t = 0; t < cp; ++t) {
        int s = ((r - t) % cp + cp) % cp;
        for (int64_t j = (int64_t)s * Ls; j < (int64_t)(s + 1) * Ls; ++j) {
          if (causal && global_pos(layout, cp, Ls, j) > qpos) continue;
          double dot = 0.0;
          for (int d = 0; d < D; ++d) dot += (double)qrow[d] * (double)kh[j * D + d];
          double sj = scale * dot;
          if (sj > smax) smax = sj;
          double p = exp(sj - ci);
          acc_l += p;
          for (int d = 0; d < D; ++d) orow[d] += p * (double)vh[j * D + d];
        }
      }
      double denom = acc_l > 1e-37 ? acc_l : 1e-37;
      for (int d = 0; d < D; ++d) orow[d] /= denom;
      lse[i] = ci + log(acc_l);
      if (overshoot) overshoot[i] = ci - smax;
    }
  }
}

/* ---------------------------------------------------------------------------
 * DCP index maps, by enumeration.  The DCP page's "Slot Mapping and KV Cache"
 * deals blocks of I consecutive tokens to the W ranks round robin (block 0 to
 * rank 0, block 1 to rank 1, ..., block W to rank 0 again).  The functions
 * below simulate that dealing token by token; they never evaluate the closed
 * forms that the CUDA library uses.
 * ------------------------------------------------------------------------- */

/* For global positions 0..n-1: owner rank and local index on that rank. */
void ora_dcp_deal(int64_t n, int W, int I, int32_t *owner, int64_t *local) {
  int rank = 0, in_block = 0;
  int64_t *count = (int64_t *)ora_alloc((size_t)W, sizeof(int64_t));
  for (int64_t p = 0; p < n; ++p) {
    owner[p] = rank;
    local[p] = count[rank]++;
    if (++in_block == I) {
      in_block = 0;
      rank = (rank + 1) % W;
    }
  }
  free(count);
}

/* Number of tokens among positions 0..N-1 that rank R holds. */
int64_t ora_dcp_local_filled(int64_t N, int W, int I, int R) {
  int32_t *own = (int32_t *)ora_alloc((size_t)(N > 0 ? N : 1), sizeof(int32_t));
  int64_t *loc = (int64_t *)ora_alloc((size_t)(N > 0 ? N : 1), sizeof(int64_t));
  ora_dcp_deal(N, W, I, own, loc);
  int64_t cnt = 0;
  for (int64_t p = 0; p < N; ++p) cnt += own[p] == R;
  free(own);
  free(loc);
  return cnt;
}

/* DCP decode for one query token per sequence (DCP page, "Decode Compute
 * Pattern").  q [N, Hq, D]; k_shards, v_shards [W, N, Hkv, Lloc, D], where
 * shard r holds its dealt tokens in local order.  Sequence n attends to global
 * positions [0, seq_lens[n]) (all of them are visible: the decoded token's own
 * K/V is already in the cache, held by its owner only).  Each rank computes a
 * partial (o_r, lse_r) over the local slots it holds, then the partials are
 * LSE-merged.  o [N, Hq, D], lse [N, Hq]. */
void ora_dcp_decode(const float *q, const float *k_shards,
                    const float *v_shards, int N, int Hq, int Hkv,
                    int64_t Lloc, int D, int W, int I, const int64_t *seq_lens,
                    double scale, double *o, double *lse) {
  int G = Hq / Hkv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t nh = 0; nh < (int64_t)N * Hq; ++nh) {
    int64_t n = nh / Hq, h = nh % Hq, hk = h / G;
    int64_t L = seq_lens[n];
    const float *qrow = q + nh * D;
    /* which local slots of each rank are valid: deal positions 0..L-1 */
    int32_t *own = (int32_t *)ora_alloc((size_t)(L > 0 ? L : 1), sizeof(int32_t));
    int64_t *loc = (int64_t *)ora_alloc((size_t)(L > 0 ? L : 1), sizeof(int64_t));
    ora_dcp_deal(L, W, I, own, loc);
    double *op = (double *)ora_alloc((size_t)W * D, sizeof(double));
    double *lp = (double *)ora_alloc((size_t)W, sizeof(double));
    for (int r = 0; r < W; ++r) {
      const float *kh = k_shards + (((int64_t)r * N + n) * Hkv + hk) * Lloc * D;
      const float *vh = v_shards + (((int64_t)r * N + n) * Hkv + hk) * Lloc * D;
      double m = -INFINITY;
      for (int64_t p = 0; p < L; ++p) {
        if (own[p] != r) continue;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (double)qrow[d] * (double)kh[loc[p] * D + d];
        if (scale * dot > m) m = scale * dot;
      }
      if (m == -INFINITY) {
        lp[r] = -INFINITY;
        continue;
      }
      double l = 0.0;
      for (int64_t p = 0; p < L; ++p) {
        if (own[p] != r) continue;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (double)qrow[d] * (double)kh[loc[p] * D + d];
        double w = exp(scale * dot - m);
        l += w;
        for (int d = 0; d < D; ++d) op[(int64_t)r * D + d] += w * (double)vh[loc[p] * D + d];
      }
      for (int d = 0; d < D; ++d) op[(int64_t)r * D + d] /= l;
      lp[r] = m + log(l);
    }
    ora_lse_merge(op, lp, W, 1, D, o + nh * D, lse + nh);
    free(own);
    free(loc);
    free(op);
    free(lp);
  }
}

/* Ring Pass-Q decode ("Sharding the Input", its paragraph on the decode
 * phase): the KV cache stays where the sharded prefill left it and the single
 * query token of each sequence visits every shard, which computes a partial
 * attention over its own part of the cache; the partials are merged by their
 * log-sum-exp.  The cache is the ring layout: k, v [B, Hkv, S, D], each head's
 * S rows shard-major (row rho = r*Ls + a is local token a of shard r, at the
 * global position global_pos gives).  Sequence b's query attends to the
 * global positions [0, seq_lens[b]), all visible (it is the next token).
 * Shard r's partial covers its rows whose global position is below
 * seq_lens[b] (none: lse_r = -inf); the cp partials are LSE-merged.
 * q [B, Hq, D]; o [B, Hq, D], lse [B, Hq]. */
void ora_ring_decode(const float *q, const float *k, const float *v, int B, int Hq, int Hkv,
                     int64_t S, int D, int cp, int layout, const int64_t *seq_lens,
                     double scale, double *o, double *lse) {
  int G = Hq / Hkv;
  int64_t Ls = S / cp;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
    int64_t b = bh / Hq, h = bh % Hq, hk = h / G;
    int64_t L = seq_lens[b];
    const float *qrow = q + bh * D;
    const float *kh = k + ((int64_t)b * Hkv + hk) * S * D;
    const float *vh = v + ((int64_t)b * Hkv + hk) * S * D;
    double *op = (double *)ora_alloc((size_t)cp * D, sizeof(double));
    double *lp = (double *)ora_alloc((size_t)cp, sizeof(double));
    for (int r = 0; r < cp; ++r) {
      double m = -INFINITY;
      for (int64_t rho = r * Ls; rho < (r + 1) * Ls; ++rho) {
        if (global_pos(layout, cp, Ls, rho) >= L) continue;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (double)qrow[d] * (double)kh[rho * D + d];
        if (scale * dot > m) m = scale * dot;
      }
      if (m == -INFINITY) {
        lp[r] = -INFINITY;
        continue;
      }
      double l = 0.0;
      for (int64_t rho = r * Ls; rho < (r + 1) * Ls; ++rho) {
        if (global_pos(layout, cp, Ls, rho) >= L) continue;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (double)qrow[d] * (double)kh[rho * D + d];
        double w = exp(scale * dot - m);
        l += w;
        for (int d = 0; d < D; ++d) op[(int64_t)r * D + d] += w * (double)vh[rho * D + d];
      }
      for (int d = 0; d < D; ++d) op[(int64_t)r * D + d] /= l;
      lp[r] = m + log(l);
    }
    ora_lse_merge(op, lp, cp, 1, D, o + bh * D, lse + bh);
    free(op);
    free(lp);
  }
}

/* DCP prefill of one chunk ("DCP (Decode Context Parallelism)", section
 * "Segmented Attention CP"): every rank R holds, locally, the prior tokens
 * dealt to it (prior slots) and its share of the current chunk (current
 * tokens).  The gathered queries of the chunk attend to each rank's local
 * prior + current KV with a causal mask on global positions, giving a
 * partial (o_R, lse_R); the partials are LSE-merged.
 *
 * Global positions, as the page's algorithm step 3 defines them: prior
 * tokens are the positions [0, P) dealt from position 0; current chunk
 * token j of rank R sits at P + (chunk position of j), the chunk's own
 * positions dealt from the chunk start; query i of the chunk sits at P + i.
 * Both deals are simulated token by token (ora_dcp_deal).
 *
 * q [Hq, Sc, D]; k_prior, v_prior [W, Hkv, Lcap, D] (slot s of rank R in
 * row s); k_cur, v_cur [W, Hkv, Lc, D] (current token j of rank R in row j).
 * rows: flat query ids h*Sc + i to compute (nrows of them); o [nrows, D],
 * lse [nrows].  If part_rank >= 0 only that rank's partial is computed (no
 * merge). */
void ora_dcp_prefill(const float *q, const float *k_prior, const float *v_prior,
                     const float *k_cur, const float *v_cur, int Hq, int Hkv,
                     int64_t Sc, int D, int W, int I, int64_t P, int64_t Lcap,
                     int64_t Lc, double scale, int part_rank, const int64_t *rows,
                     int64_t nrows, double *o, double *lse) {
  int G = Hq / Hkv;
  int32_t *own_p = (int32_t *)ora_alloc((size_t)(P > 0 ? P : 1), sizeof(int32_t));
  int64_t *loc_p = (int64_t *)ora_alloc((size_t)(P > 0 ? P : 1), sizeof(int64_t));
  int32_t *own_c = (int32_t *)ora_alloc((size_t)(Sc > 0 ? Sc : 1), sizeof(int32_t));
  int64_t *loc_c = (int64_t *)ora_alloc((size_t)(Sc > 0 ? Sc : 1), sizeof(int64_t));
  ora_dcp_deal(P, W, I, own_p, loc_p);
  ora_dcp_deal(Sc, W, I, own_c, loc_c);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t ri = 0; ri < nrows; ++ri) {
    const int64_t hi = rows[ri];
    int64_t h = hi / Sc, i = hi % Sc, hk = h / G;
    const float *qrow = q + hi * D;
    double *op = (double *)ora_alloc((size_t)W * D, sizeof(double));
    double *lp = (double *)ora_alloc((size_t)W, sizeof(double));
    for (int r = 0; r < W; ++r) {
      lp[r] = -INFINITY;
      if (part_rank >= 0 && r != part_rank) continue;
      const float *kp = k_prior + ((int64_t)r * Hkv + hk) * Lcap * D;
      const float *vp = v_prior + ((int64_t)r * Hkv + hk) * Lcap * D;
      const float *kc = k_cur + ((int64_t)r * Hkv + hk) * Lc * D;
      const float *vc = v_cur + ((int64_t)r * Hkv + hk) * Lc * D;
      /* visible keys of rank r: its prior tokens (all before the chunk) and
       * its current tokens at chunk positions <= i */
      double m = -INFINITY;
      for (int pass = 0; pass < 2; ++pass) {
        double l = 0.0;
        for (int64_t p = 0; p < P + i + 1; ++p) {
          const float *kr, *vr;
          if (p < P) {
            if (own_p[p] != r) continue;
            kr = kp + loc_p[p] * D;
            vr = vp + loc_p[p] * D;
          } else {
            if (own_c[p - P] != r) continue;
            kr = kc + loc_c[p - P] * D;
            vr = vc + loc_c[p - P] * D;
          }
          double dot = 0.0;
          for (int d = 0; d < D; ++d) dot += (double)qrow[d] * (double)kr[d];
          double sj = scale * dot;
          if (pass == 0) {
            if (sj > m) m = sj;
          } else {
            double w = exp(sj - m);
            l += w;
            for (int d = 0; d < D; ++d) op[(int64_t)r * D + d] += w * (double)vr[d];
          }
        }
        if (pass == 0 && m == -INFINITY) break;
        if (pass == 1) {
          for (int d = 0; d < D; ++d) op[(int64_t)r * D + d] /= l;
          lp[r] = m + log(l);
        }
      }
    }
    if (part_rank >= 0) {
      for (int d = 0; d < D; ++d) o[ri * D + d] = op[(int64_t)part_rank * D + d];
      lse[ri] = lp[part_rank];
    } else {
      ora_lse_merge(op, lp, W, 1, D, o + ri * D, lse + ri);
    }
    free(op);
    free(lp);
  }
  free(own_p);
  free(loc_p);
  free(own_c);
  free(loc_c);
}

/* DCP decode over a paged KV cache ("DCP (Decode Context Parallelism)",
 * sections "Slot Mapping and KV Cache" and "Segmented Attention CP", step 1:
 * the prior KV is read from the cache through the block table).  Rank r's
 * cache holds blocks of `bs` slots per KV head: k_cache[r][blk][hk][t][d]
 * ([W, nblk, Hkv, bs, D]).  Local slot s of sequence n on rank r lives in
 * block block_tables[r][n][s / bs] at offset s % bs.  The decode itself is
 * ora_dcp_decode's: gather each rank's local slots in order, then the same
 * per-rank partials and LSE merge.  block_tables is [W, N, max_blocks]. */
void ora_dcp_decode_paged(const float *q, const float *k_cache, const float *v_cache,
                          const int32_t *block_tables, int N, int Hq, int Hkv, int64_t nblk,
                          int bs, int64_t max_blocks, int D, int W, int I,
                          const int64_t *seq_lens, double scale, double *o, double *lse) {
  int64_t Lloc = max_blocks * bs;
  float *ks = (float *)ora_alloc((size_t)W * N * Hkv * Lloc * D, sizeof(float));
  float *vs = (float *)ora_alloc((size_t)W * N * Hkv * Lloc * D, sizeof(float));
  for (int r = 0; r < W; ++r)
    for (int n = 0; n < N; ++n) {
      /* only the slots the sequence actually has on this rank are gathered */
      int32_t *own = (int32_t *)ora_alloc((size_t)(seq_lens[n] > 0 ? seq_lens[n] : 1), sizeof(int32_t));
      int64_t *loc = (int64_t *)ora_alloc((size_t)(seq_lens[n] > 0 ? seq_lens[n] : 1), sizeof(int64_t));
      ora_dcp_deal(seq_lens[n], W, I, own, loc);
      for (int64_t p = 0; p < seq_lens[n]; ++p) {
        if (own[p] != r) continue;
        int64_t s = loc[p];
        int64_t blk = block_tables[((int64_t)r * N + n) * max_blocks + s / bs];
        for (int hk = 0; hk < Hkv; ++hk)
          for (int d = 0; d < D; ++d) {
            int64_t src = (((int64_t)r * nblk + blk) * Hkv + hk) * bs * D + (s % bs) * D + d;
            int64_t dst = ((((int64_t)r * N + n) * Hkv + hk) * Lloc + s) * D + d;
            ks[dst] = k_cache[src];
            vs[dst] = v_cache[src];
          }
      }
      free(own);
      free(loc);
    }
  ora_dcp_decode(q, ks, vs, N, Hq, Hkv, Lloc, D, W, I, seq_lens, scale, o, lse);
  free(ks);
  free(vs);
}

/* Prologue of const-max attention on one projected tensor: from activations
 * x [B, S, H*D] in token order (token p at global position p) to the
 * attention input out [B, H, S, D] in the shard-major row order of `layout`
 * (stored row rho holds token global_pos(rho)).  "Context Parallelism in
 * vLLM Omni Neuron", section "Self-Attention with Context Parallelism": the
 * projected q and k are normalised over the whole hidden before the head
 * split, then rotary embeddings are applied to every head at the token's
 * position.
 *  - norm != 0: y_j = x_j / sqrt(mean over all H*D channels of x^2 + eps)
 *    * g_j (g == NULL: g_j = 1), the RMS norm of the whole hidden;
 *    norm == 0: y = x (the value tensor).
 *  - cs != NULL: every head's channel pairs (2i, 2i+1) turn by the angle of
 *    token p whose cosine and sine are cs[p*(D/2) + i], sn[p*(D/2) + i]:
 *      y'_2i = y_2i c - y_2i+1 s,   y'_2i+1 = y_2i s + y_2i+1 c.
 * All arithmetic in double from the stored (widened) inputs. */
void ora_qk_prologue(const float *x, const float *g, double eps, const float *cs,
                     const float *sn, int B, int64_t S, int H, int D, int cp,
                     int layout, int norm, double *out) {
  const int64_t Ls = S / cp;
  const int64_t HD = (int64_t)H * D;
#pragma omp parallel for collapse(2) schedule(static)
  for (int b = 0; b < B; ++b)
    for (int64_t rho = 0; rho < S; ++rho) {
      const int64_t p = global_pos(layout, cp, Ls, rho);
      const float *xr = x + ((int64_t)b * S + p) * HD;
      double scale = 1.0;
      if (norm) {
        double ss = 0.0;
        for (int64_t j = 0; j < HD; ++j) ss += (double)xr[j] * (double)xr[j];
        scale = 1.0 / sqrt(ss / (double)HD + eps);
      }
      for (int h = 0; h < H; ++h) {
        double *o = out + (((int64_t)b * H + h) * S + rho) * D;
        for (int d = 0; d < D; ++d) {
          const int64_t j = (int64_t)h * D + d;
          double y = (double)xr[j];
          if (norm) y = y * scale * (g ? (double)g[j] : 1.0);
          o[d] = y;
        }
        if (cs) {
          for (int i = 0; i < D / 2; ++i) {
            const double c = cs[p * (D / 2) + i], s = sn[p * (D / 2) + i];
            const double y0 = o[2 * i], y1 = o[2 * i + 1];
            o[2 * i] = y0 * c - y1 * s;
            o[2 * i + 1] = y0 * s + y1 * c;
          }
        }
      }
    }
}

/* Number of OpenMP threads a parallel region here would use. */
int ora_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
