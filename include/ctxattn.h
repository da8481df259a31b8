/*
 * ctxattn.h -- C ABI of libctxattn.so: the hot path of context-parallel
 * attention on one NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages on context parallelism):
 *   [CM]   "Kernel reference: ring_attention_const_max_fwd const-max ring
 *          attention" (Neuron docs, vllm-omni-neuron).
 *   [DCP]  "DCP (Decode Context Parallelism)" (Neuron docs, vllm-neuron).
 *   [CP]   "Context Parallelism in vLLM Omni Neuron" (Neuron docs).
 *   [SHI]  "Sharding the Input" (iop.systems blog).
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers marked "device" are CUDA device (or managed) addresses of the
 *   current device; pointers marked "host" are host addresses.  The caller
 *   owns and allocates every buffer, workspace included.  The library never
 *   allocates, frees or synchronises; device work is enqueued on `stream`
 *   (a cudaStream_t passed as void*, NULL = legacy default stream).
 * - Tensors are dense row-major, no strides.  Element types: CA_DTYPE_BF16
 *   (inputs and outputs bf16, all accumulation fp32) or CA_DTYPE_F32 (fp32
 *   end to end).  LSE values are fp32, natural log, softmax scale included:
 *   lse_i = ln sum_j exp(scale * q_i . k_j).
 * - Attention tensors: q is [B, Hq, S, D]; k and v are [B, Hkv, S, D]; query
 *   head h reads key/value head h / (Hq / Hkv) (consecutive groups).
 * - Virtual shards: the S rows of a head are `cp_size` shards of Ls = S /
 *   cp_size rows, stored shard-major: row r*Ls + a is local token a of shard
 *   r.  Its global position is r*Ls + a (CA_LAYOUT_CONTIGUOUS, [CP] "Model
 *   Implementation": start = cp_rank * local_S) or a*cp_size + r
 *   (CA_LAYOUT_STRIPED, [SHI]: token t on shard t mod cp).  Outputs use the
 *   same row order as q.
 * - Causal: key j is visible to query i iff global(j) <= global(i).
 * - Sizes (batch, heads, rows, head dimension, sequences, shards) must be
 *   positive: an empty problem is CA_ERR_INVALID_ARG.  The one exception is
 *   ca_paged_kv_write with T = 0 new tokens, a valid no-op.
 * - Errors: every call validates its arguments on the host first and returns
 *   a ca_status; on a host-side error nothing is enqueued and nothing is
 *   written.  There is no fallback path: an unsupported case is an error.
 *   CA_ERR_CUDA reports a failed launch (cudaGetLastError after the launch).
 *   Device-side faults of the bounded waits are reported by
 *   ca_device_status().
 * - Supported: bf16 with D = 128; fp32 with 1 <= D <= 128.  Device: compute
 *   capability 10.3 (GB300) for the bf16 kernels; the fp32 and
 *   data-movement kernels run on the same build (sm_103a).
 */
#ifndef CTXATTN_H
#define CTXATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CA_OK = 0,
  CA_ERR_INVALID_ARG = 1, /* null pointer, bad enum, non-positive size */
  CA_ERR_SHAPE = 2,       /* S % cp_size != 0, Hq % Hkv != 0, bad shard sizes */
  CA_ERR_UNSUPPORTED = 3, /* dtype/D combination or device not supported */
  CA_ERR_ALIGNMENT = 4,   /* a device pointer is not 16-byte aligned */
  CA_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required */
  CA_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed */
  CA_ERR_TIMEOUT = 7      /* a bounded device-side wait gave up */
} ca_status;

typedef enum { CA_DTYPE_F32 = 0, CA_DTYPE_BF16 = 1 } ca_dtype;
typedef enum { CA_MODE_ONLINE_MAX = 0, CA_MODE_CONST_MAX = 1 } ca_mode;
typedef enum { CA_LAYOUT_CONTIGUOUS = 0, CA_LAYOUT_STRIPED = 1 } ca_layout;

/* Human-readable name of a status code (static string, never NULL). */
const char *ca_status_string(ca_status status);

/* Library ABI version (major*100 + minor). */
int ca_version(void);

/* ------------------------------------------------------------------------
 * Ring attention forward ([CM] "Overview", "Design", "Interface").
 *
 * Q stays resident; the K/V of the cp_size virtual shards are visited one
 * ring step at a time: the query rows of shard r meet, at step t = 0 ..
 * cp_size-1, the keys of shard (r - t) mod cp_size.  Every step's partial
 * result is folded into an fp32 accumulator that never leaves the SM.
 *   mode CA_MODE_ONLINE_MAX: flash-style running row maximum; folding a step
 *     is the LSE merge w_i = exp(lse_i - lse_global) ([DCP] "Decode Compute
 *     Pattern", steps 4-7) applied tile by tile.
 *   mode CA_MODE_CONST_MAX: the per-row Cauchy-Schwarz bound
 *     c_i = scale * |q_i| * max_j |k_j| (max over all S keys of the key/value
 *     head, [CM] "Picking a max that is safe without measuring it") replaces
 *     the running max; steps merge by pure addition of unnormalised sums and
 *     the row is normalised once, o = acc_o / max(acc_l, 1e-37), lse =
 *     c + ln(acc_l) ([CM] "A static bound makes the ring reduction pure
 *     addition", "Accumulate, then normalize once").  Rows whose bound
 *     overshoots the true row maximum by more than ~87 nats underflow to the
 *     clamp, exactly as the page warns ("Common issues").
 *
 * q, k, v     device, [B,Hq,S,D] / [B,Hkv,S,D], dtype, 16-byte aligned.
 * o           device, [B,Hq,S,D], dtype (same row order as q).
 * lse         device, [B,Hq,S] fp32, or NULL.
 * softmax_scale  <= 0 selects 1/sqrt(D).
 * workspace   device, at least ca_ring_attn_fwd_workspace_size() bytes
 *             (may be NULL when that size is 0).  Const max uses it for
 *             kmax2 [B,Hkv]: one streaming pass over k (ca_key_max2), after
 *             which the attention kernel forms each row's bound from the q
 *             row it has loaded anyway ([CM] "Best practices": side
 *             quantities inside a pass already paid for).
 * Errors: CA_ERR_SHAPE if S % cp_size != 0 ([CP] "Sequence Length
 * Constraints": S=3645 with cp_size=8 is rejected) or Hq % Hkv != 0;
 * CA_ERR_UNSUPPORTED for bf16 with D != 128 or B*Hq*S >= 2^31 (the kernel
 * addresses rows with 32-bit indices), and for fp32 with D > 128.
 * ---------------------------------------------------------------------- */
size_t ca_ring_attn_fwd_workspace_size(int B, int Hq, int Hkv, int64_t S, int D,
                                       int cp_size, ca_mode mode);
ca_status ca_ring_attn_fwd(const void *q, const void *k, const void *v, void *o,
                           float *lse, ca_dtype dtype, int B, int Hq, int Hkv,
                           int64_t S, int D, int cp_size, ca_mode mode,
                           int causal, ca_layout layout, float softmax_scale,
                           void *workspace, size_t workspace_bytes,
                           void *stream);

/* Ring attention in const-max mode with a caller-provided bound
 * ([CM] "Picking a max that is safe without measuring it")
 * c [B,Hq,S] fp32 (device; e.g. from ca_const_max_bound): the same
 * computation as ca_ring_attn_fwd(mode = CA_MODE_CONST_MAX) without the bound
 * pass, for callers that compute or reuse the bound themselves.  Needs no
 * workspace. */
ca_status ca_ring_attn_fwd_bounded(const void *q, const void *k, const void *v,
                                   const float *c, void *o, float *lse,
                                   ca_dtype dtype, int B, int Hq, int Hkv,
                                   int64_t S, int D, int cp_size, int causal,
                                   ca_layout layout, float softmax_scale,
                                   void *stream);

/* Ring attention in const-max mode with a caller-provided key maximum
 * kmax2 [B,Hkv] fp32 (device): max over all keys of the head of |k_j|^2, as
 * ca_key_max2 gives it for local keys; a caller whose keys span several
 * processes takes the elementwise max of their kmax2 first ([CM] "Global
 * key max": one all-reduce(max) of one value per head).  The kernel forms
 * c_i = sqrt(scale^2 * kmax2 * |q_i|^2) from each q row it loads.  Same
 * output as ca_ring_attn_fwd(mode = CA_MODE_CONST_MAX); no workspace. */
ca_status ca_ring_attn_fwd_kmax(const void *q, const void *k, const void *v,
                                const float *kmax2, void *o, float *lse,
                                ca_dtype dtype, int B, int Hq, int Hkv,
                                int64_t S, int D, int cp_size, int causal,
                                ca_layout layout, float softmax_scale,
                                void *stream);

/* ------------------------------------------------------------------------
 * One ring step ([CM] "Overview", step t: acc_r += attn(Q_r, K_{r-t},
 * V_{r-t})): the queries of shard q_rank against the keys of shard kv_rank
 * only, with the causal rule evaluated on global positions of the given
 * layout.
 *
 * q_shard     device [B,Hq,Ls,D]; k_shard, v_shard device [B,Hkv,Ls,D].
 * c           CA_MODE_CONST_MAX: device [B,Hq,Ls] fp32 bound rows of this
 *             shard (from ca_const_max_bound); CA_MODE_ONLINE_MAX: NULL.
 * o_part      device [B,Hq,Ls,D] fp32.  Online max: the normalised partial
 *             o_i.  Const max: the unnormalised sum acc_o = sum_j
 *             exp(s_ij - c_i) v_j.
 * lse_part    device [B,Hq,Ls] fp32: the partial's log-sum-exp (both modes;
 *             in const max it is c_i + ln acc_l).  A row with no visible key
 *             gets o_part = 0 and lse_part = -inf.
 * ---------------------------------------------------------------------- */
ca_status ca_attn_partial_step(const void *q_shard, const void *k_shard,
                               const void *v_shard, ca_dtype dtype, int B,
                               int Hq, int Hkv, int64_t Ls, int D, int q_rank,
                               int kv_rank, int cp_size, ca_mode mode,
                               int causal, ca_layout layout,
                               float softmax_scale, const float *c,
                               float *o_part, float *lse_part, void *stream);

/* ------------------------------------------------------------------------
 * LSE merge of n partial results ([DCP] "Decode Compute Pattern" steps 5-7
 * and "Segmented Attention CP" step 6; [CM] "Accumulate, then normalize
 * once").
 *
 * o_parts     device [n, R, D] fp32; lse_parts device [n, R] fp32.
 * c == NULL:  partials are normalised; L = ln sum_i exp(lse_i),
 *             o = sum_i exp(lse_i - L) o_i.  Partials with lse = -inf get
 *             weight 0; if all are -inf the row gets o = 0, lse = -inf.
 * c != NULL:  device [R] fp32 bound; partials are the unnormalised const-max
 *             sums of ca_attn_partial_step; acc_l_i = exp(lse_i - c),
 *             o = sum_i o_i / max(sum_i acc_l_i, 1e-37), lse = c + ln sum_i
 *             acc_l_i (pure addition).
 * A partial of zero weight (lse_i = -inf in either mode, or, with c ==
 * NULL, a weight that underflows to 0) adds nothing: its o row is not used
 * and may hold any bits, NaN included.
 * o           device [R, D] of out_dtype; lse device [R] fp32 or NULL.
 * ---------------------------------------------------------------------- */
ca_status ca_lse_merge(const float *o_parts, const float *lse_parts, int n,
                       int64_t R, int D, const float *c, void *o,
                       ca_dtype out_dtype, float *lse, void *stream);

/* ------------------------------------------------------------------------
 * QKV prologue of const-max attention ([CP] "Self-Attention with Context
 * Parallelism": the projected q and k are normalised over the whole hidden
 * before the head split and rotary embeddings are applied per head at each
 * token's position; [CM] "Best practices", "Transpose prologue with fused
 * norms": the per-head key maximum is reduced in the same pass).  One read
 * of the activations, one write of the attention inputs:
 *   q, k:  y_j = x_j / sqrt(mean over the H*D channels of x^2 + eps) * g_j,
 *          then every head's channel pairs (2i, 2i+1) turn by the token's
 *          angle: y'_2i = y_2i c - y_2i+1 s, y'_2i+1 = y_2i s + y_2i+1 c with
 *          c = rope_cos[p*D/2 + i], s = rope_sin[p*D/2 + i]; rounded to bf16;
 *   v:     split into heads unchanged.
 * Token p (its global position) lands on row layout-shard-row(p) of every
 * head of the [B,H,S,D] outputs (contiguous: p; striped: (p mod cp)*S/cp +
 * p div cp), the row order ca_ring_attn_fwd takes.  kmax2[b,h] = max over the
 * rows of |k_row|^2 summed in fp32 from the rounded bf16 outputs, ready for
 * ca_ring_attn_fwd_kmax.
 *
 * x_q         device [B,S,Hq*D] bf16 (token order); x_k, x_v [B,S,Hkv*D];
 *             x_v may be NULL (then v is not written).
 * g_q, g_k    device [Hq*D] / [Hkv*D] fp32 gains, or NULL (gain 1).
 * eps         >= 0, added to the mean square.
 * rope_cos, rope_sin  device [S, D/2] fp32, both or neither (no rotation).
 * q, k, v     device [B,Hq,S,D] / [B,Hkv,S,D] bf16 outputs.
 * kmax2       device [B,Hkv] fp32 output (zeroed, then reduced into), or NULL.
 * All tensor pointers 16-byte aligned (kmax2 4-byte); B*S*3 < 2^31.
 * Errors: CA_ERR_SHAPE if Hq % Hkv or S % cp_size; CA_ERR_UNSUPPORTED unless
 * bf16 with D in {64, 128} and Hq*D <= 8192.
 * ---------------------------------------------------------------------- */
ca_status ca_qkv_prologue(const void *x_q, const void *x_k, const void *x_v,
                          const float *g_q, const float *g_k, float eps,
                          const float *rope_cos, const float *rope_sin,
                          ca_dtype dtype, int B, int64_t S, int Hq, int Hkv,
                          int D, int cp_size, ca_layout layout, void *q,
                          void *k, void *v, float *kmax2, void *stream);

/* ------------------------------------------------------------------------
 * Key maximum of the const-max bound ([CM] "Global key max", "Transpose
 * prologue with fused norms": per head, the running max of |k_j|^2):
 * kmax2[b,hk] = max over the S rows of k[b,hk] of |k_j|^2, squares summed in
 * fp32.  kmax2 is zeroed first, then reduced into (an fp32 max of
 * non-negative values, exact whatever the order).
 *
 * k           device [B,Hkv,S,D], dtype, 16-byte aligned.
 * kmax2       device [B,Hkv] fp32 (output), 4-byte aligned.
 * ---------------------------------------------------------------------- */
ca_status ca_key_max2(const void *k, ca_dtype dtype, int B, int Hkv, int64_t S,
                      int D, float *kmax2, void *stream);

/* ------------------------------------------------------------------------
 * Const-max bound ([CM] "Picking a max ...", "Global key max", "Assembling
 * the bound"): kmax2[b,hk] = max_j |k_j|^2 over all S rows of the head, then
 * c[b,h,i] = sqrt(scale^2 * kmax2[b,h/G] * |q_i|^2) (one square root per row).
 *
 * q, k        device, [B,Hq,S,D] / [B,Hkv,S,D], dtype.
 * c           device [B,Hq,S] fp32 (output).
 * kmax2       device [B,Hkv] fp32 (output; also the reduction target).
 * ---------------------------------------------------------------------- */
ca_status ca_const_max_bound(const void *q, const void *k, ca_dtype dtype,
                             int B, int Hq, int Hkv, int64_t S, int D,
                             float softmax_scale, float *c, float *kmax2,
                             void *stream);

/* ------------------------------------------------------------------------
 * DCP decode ([DCP] "DCP Decode", "Decode Compute Pattern", "local_filled
 * Computation"): one query token per sequence against K/V shards whose
 * blocks of `interleave` tokens are dealt round robin to dcp ranks (block b
 * on rank b mod dcp, [DCP] "Slot Mapping and KV Cache").  Each rank's local
 * slots [0, local_filled(seq_len, rank)) are valid; every rank computes a
 * partial (o_r, lse_r) and the partials are LSE-merged.
 *
 * q           device [N, Hq, D], dtype.
 * k_shards, v_shards  device [dcp, N, Hkv, Lloc, D], dtype.
 * seq_lens    device int32 [N] (tokens in the cache, 0..dcp*Lloc), or NULL
 *             for dcp*Lloc everywhere.
 * o           device [N, Hq, D], dtype; lse device [N, Hq] fp32 (or NULL).
 * workspace   device, ca_dcp_decode_workspace_size() bytes (partials).
 * Errors: CA_ERR_SHAPE if Hq % Hkv != 0 or Lloc % interleave != 0;
 * CA_ERR_UNSUPPORTED unless bf16 with D = 128 and Hq/Hkv <= 8.
 * ---------------------------------------------------------------------- */
size_t ca_dcp_decode_workspace_size(int N, int Hq, int Hkv, int64_t Lloc,
                                    int D, int dcp, int interleave);
ca_status ca_dcp_decode(const void *q, const void *k_shards,
                        const void *v_shards, ca_dtype dtype, int N, int Hq,
                        int Hkv, int64_t Lloc, int D, int dcp, int interleave,
                        const int32_t *seq_lens, float softmax_scale, void *o,
                        float *lse, void *workspace, size_t workspace_bytes,
                        void *stream);

/* DCP decode without a workspace, for callers that cannot allocate device
 * memory at call time: code running inside a framework whose allocator
 * already owns all device memory, or plugin-style enqueue paths that must
 * not allocate.  The pages have no counterpart of this call; it exists for
 * such callers only.
 *
 * Same arguments and results as ca_dcp_decode, minus the workspace, and the
 * same argument checks in the same order (null pointers and sizes, shape,
 * unsupported dtype or head layout, alignment); where ca_dcp_decode then
 * checks its workspace, this call checks its scratch.  The split-KV partials
 * live in a scratch array built into the library's device image: 16 MiB,
 * held on every GPU that loads the library until the process exits.  A
 * problem whose partials need more than that
 * (ca_dcp_decode_workspace_size() > 16 MiB) is rejected with
 * CA_ERR_WORKSPACE before anything is enqueued; on a device other than a
 * GB300 the call returns CA_ERR_UNSUPPORTED.  The call allocates nothing.
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress, once per device, cached for the process: calls
 * after cudaDeviceReset are unsupported); make that first call before any
 * stream capture.  All calls on a device share the one scratch array, so
 * calls whose kernels overlap on the GPU race on it and must be serialised
 * by the caller.  Nothing in it needs to start at zero: the same call writes
 * the log-sum-exp of every partial slot, and the o row of every slot that
 * holds tokens (the merge does not use the others). */
ca_status ca_dcp_decode_noalloc(const void *q, const void *k_shards,
                                const void *v_shards, ca_dtype dtype, int N,
                                int Hq, int Hkv, int64_t Lloc, int D, int dcp,
                                int interleave, const int32_t *seq_lens,
                                float softmax_scale, void *o, float *lse,
                                void *stream);

/* ------------------------------------------------------------------------
 * Ring Pass-Q decode ([SHI], its paragraph on the decode phase): the KV
 * cache stays in the ring layout the sharded prefill left it in and the one
 * query token of each sequence visits every shard; shard r computes a
 * partial (o_r, lse_r) over its slots that hold one of the global positions
 * [0, seq_len) -- all of them visible, the query being the next token -- and
 * the cp partials are LSE-merged ([DCP] "Decode Compute Pattern").  On one
 * GPU the query's "visits" are work items of one kernel; no data moves.
 *
 * q           device [B, Hq, D], dtype (one query token per sequence).
 * k, v        device [B, Hkv, S, D], dtype, each head's rows shard-major as
 *             in ca_ring_attn_fwd: row r*Ls + a is local token a of shard r,
 *             at global position r*Ls + a (CA_LAYOUT_CONTIGUOUS) or a*cp + r
 *             (CA_LAYOUT_STRIPED).  Slots at global positions >= seq_len are
 *             never read.
 * seq_lens    device int32 [B] (tokens in the cache, 0..S), or NULL for S.
 * o           device [B, Hq, D], dtype; lse device [B, Hq] fp32 (or NULL).
 *             A sequence with seq_len 0 gets o = 0, lse = -inf.
 * workspace   device, ca_ring_decode_workspace_size() bytes (partials).
 * Errors: CA_ERR_SHAPE if Hq % Hkv != 0 or S % cp_size != 0;
 * CA_ERR_UNSUPPORTED unless bf16 with D = 128, Hq/Hkv <= 8 and
 * B*Hkv*S < 2^31.
 * ---------------------------------------------------------------------- */
size_t ca_ring_decode_workspace_size(int B, int Hq, int Hkv, int64_t S, int D,
                                     int cp_size);
ca_status ca_ring_decode(const void *q, const void *k, const void *v,
                         ca_dtype dtype, int B, int Hq, int Hkv, int64_t S,
                         int D, int cp_size, ca_layout layout,
                         const int32_t *seq_lens, float softmax_scale, void *o,
                         float *lse, void *workspace, size_t workspace_bytes,
                         void *stream);

/* ------------------------------------------------------------------------
 * DCP decode over paged KV caches ([DCP] "Slot Mapping and KV Cache",
 * "Segmented Attention CP" step 1: KV read from the cache through the block
 * table).  Same computation as ca_dcp_decode; rank r's local slot s of
 * sequence n lives in block block_tables[r][n][s / block_size] of rank r's
 * cache at offset s % block_size.
 *
 * k_cache, v_cache  device [dcp, nblk, Hkv, block_size, D] bf16 (one cache
 *             per rank; blocks hold block_size consecutive slots per head).
 * block_tables device int32 [dcp, N, max_blocks]; only the entries covering
 *             a sequence's valid slots on a rank are read.
 * seq_lens    device int32 [N] (required; at most dcp*max_blocks*block_size).
 * workspace   ca_dcp_decode_workspace_size(N, Hq, Hkv,
 *             max_blocks*block_size, D, dcp, interleave) bytes.
 * Errors: CA_ERR_UNSUPPORTED unless bf16, D = 128, Hq/Hkv <= 8,
 * block_size in {8, 16, 32, 64, 128}, and both dcp*nblk*Hkv*block_size (the
 * caches' rows) and dcp*N*Hkv*max_blocks*block_size (the slots the block
 * tables address) below 2^31.
 * ---------------------------------------------------------------------- */
ca_status ca_dcp_decode_paged(const void *q, const void *k_cache,
                              const void *v_cache, const int32_t *block_tables,
                              ca_dtype dtype, int N, int Hq, int Hkv,
                              int64_t nblk, int block_size, int64_t max_blocks,
                              int D, int dcp, int interleave,
                              const int32_t *seq_lens, float softmax_scale,
                              void *o, float *lse, void *workspace,
                              size_t workspace_bytes, void *stream);

/* Write new tokens' K/V into the paged caches by slot mapping ([DCP] "Active
 * Token Handling and dcp_active_mask", "Slot Mapping and KV Cache"): token t
 * goes to rank r's slot slots[r*T + t] (block slot / block_size, offset
 * slot % block_size); -1 means rank r does not own the token and nothing is
 * written.  Slots can come from ca_dcp_slot_mapping.  Bit-exact copies.
 * k_new, v_new device [T, Hkv, D]; slots device int64 [dcp, T];
 * k_cache, v_cache device [dcp, nblk, Hkv, block_size, D]; D*elem % 16 == 0.
 * Slots whose block is >= nblk are skipped. */
ca_status ca_paged_kv_write(const void *k_new, const void *v_new,
                            const int64_t *slots, void *k_cache, void *v_cache,
                            ca_dtype dtype, int T, int Hkv, int D, int dcp,
                            int64_t nblk, int block_size, void *stream);

/* ------------------------------------------------------------------------
 * DCP prefill of one chunk ([DCP] "Segmented Attention CP", "DCP Prefill"
 * compute pattern): the chunk's Sc gathered queries (global positions
 * P .. P+Sc-1, P = prior_tokens) attend, on every rank R, to R's local KV --
 * its prior cache slots (the positions [0, P) it was dealt, slot s at global
 * (s/I)*(dcp*I) + R*I + s%I) and its share of the chunk (chunk position p
 * dealt from the chunk start, global P + p) -- with a causal mask on global
 * positions; the per-rank partials (o_R, lse_R) are LSE-merged.  On one GPU
 * the merge happens in the accumulator; ca_dcp_prefill_partial returns one
 * rank's partial for an explicit ca_lse_merge.  Online max only.
 *
 * q           device [Hq, Sc, D] bf16.
 * k_prior, v_prior  device [dcp, Hkv, Lcap, D] bf16; rank R's prior slot s
 *             in row s; slots >= local_filled(P, R) are never read (any
 *             values, NaN included).
 * k_cur, v_cur device [dcp, Hkv, Lc, D] bf16; rank R's chunk token j in row
 *             j; rows >= local_filled(Sc, R) are never read.
 * o           device [Hq, Sc, D] bf16 (ca_dcp_prefill) or fp32
 *             (ca_dcp_prefill_partial: the normalised partial of `rank`).
 * lse         device [Hq, Sc] fp32 (nullable for ca_dcp_prefill).
 * Errors: CA_ERR_SHAPE if Hq % Hkv != 0, Lcap < local_filled(P, 0) or
 * Lc < local_filled(Sc, 0); CA_ERR_UNSUPPORTED unless bf16 with D = 128 and
 * 1 <= dcp <= 8.
 * ---------------------------------------------------------------------- */
ca_status ca_dcp_prefill(const void *q, const void *k_prior, const void *v_prior,
                         const void *k_cur, const void *v_cur, ca_dtype dtype,
                         int Hq, int Hkv, int64_t Sc, int D, int dcp,
                         int interleave, int64_t prior_tokens, int64_t Lcap,
                         int64_t Lc, float softmax_scale, void *o, float *lse,
                         void *stream);
ca_status ca_dcp_prefill_partial(const void *q, const void *k_prior,
                                 const void *v_prior, const void *k_cur,
                                 const void *v_cur, ca_dtype dtype, int Hq,
                                 int Hkv, int64_t Sc, int D, int dcp,
                                 int interleave, int64_t prior_tokens,
                                 int64_t Lcap, int64_t Lc, int rank,
                                 float softmax_scale, float *o_part,
                                 float *lse_part, void *stream);

/* ------------------------------------------------------------------------
 * Device layout permutations (bit-exact copies of rows of row_bytes bytes).
 *
 * ca_layout_to_shards: x holds BH heads of S rows in global token order;
 *   y receives them shard-major for `layout` (y row r*Ls + a = x row
 *   global(r, a)).  ca_layout_from_shards is the inverse.
 * ca_dcp_shard_kv: kv holds NH heads of L rows in global token order; shards
 *   receives [dcp, NH, L/dcp] rows, global position p going to rank
 *   (p / interleave) mod dcp at its local slot ([DCP] "Slot Mapping and KV
 *   Cache", "Segmented Attention CP": slot s of rank R is global
 *   (s / I)*(dcp*I) + R*I + s % I).  Requires L % (dcp*interleave) == 0.
 * row_bytes must be a multiple of 16; pointers 16-byte aligned.
 * ---------------------------------------------------------------------- */
ca_status ca_layout_to_shards(const void *x, void *y, int64_t BH, int64_t S,
                              int64_t row_bytes, int cp_size, ca_layout layout,
                              void *stream);
ca_status ca_layout_from_shards(const void *y, void *x, int64_t BH, int64_t S,
                                int64_t row_bytes, int cp_size,
                                ca_layout layout, void *stream);
ca_status ca_dcp_shard_kv(const void *kv, void *shards, int64_t NH, int64_t L,
                          int64_t row_bytes, int dcp, int interleave,
                          void *stream);

/* ------------------------------------------------------------------------
 * Host index helpers (pure functions, no CUDA calls).  The kernels use the
 * same closed forms on the device.
 * ---------------------------------------------------------------------- */

/* Global token position of stored row `row` (= r*Ls + a) for `layout`
 * (contiguous: r*Ls + a, [CP] "Model Implementation"; striped: a*cp + r,
 * [SHI]); -1 on bad arguments. */
int64_t ca_layout_global_index(ca_layout layout, int cp_size, int64_t Ls,
                               int64_t row);
/* Inverse: stored row of global token `token`; -1 on bad arguments. */
int64_t ca_layout_shard_row(ca_layout layout, int cp_size, int64_t Ls,
                            int64_t token);
/* Ring schedule ([CM] "Overview"): K/V shard met by shard `rank` at `step`,
 * (rank - step) mod cp_size; -1 on bad arguments. */
int ca_ring_kv_shard(int rank, int step, int cp_size);

/* Owner rank of global position pos ([DCP] "Active Token Handling and
 * dcp_active_mask", "Slot Mapping and KV Cache"): (pos / interleave) mod
 * dcp. */
int ca_dcp_owner(int64_t pos, int dcp, int interleave);
/* Local slot of pos on its owner, the inverse of ca_dcp_local_to_global
 * ([DCP] "Segmented Attention CP"): (pos / (dcp*I))*I + pos % I. */
int64_t ca_dcp_local_index(int64_t pos, int dcp, int interleave);
/* Global position of local slot s on rank R ([DCP] "Segmented Attention
 * CP"): (s / I)*(dcp*I) + R*I + s % I. */
int64_t ca_dcp_local_to_global(int64_t local, int rank, int dcp,
                               int interleave);
/* Tokens among positions [0, N) held by rank R: the [DCP] "local_filled
 * Computation" formula, evaluated as printed (block_size = the KV block size;
 * the pages require it to equal interleave). -1 on bad arguments. */
int64_t ca_dcp_local_filled(int64_t N, int dcp, int interleave, int block_size,
                            int rank);
/* [DCP] "Active Token Handling": 1 if rank owns the token at position N
 * (the decoded token), else 0; -1 on bad arguments. */
int ca_dcp_active_mask(int64_t N, int dcp, int interleave, int block_size,
                       int rank);
/* [DCP] "Slot Mapping and KV Cache": for each position, -1 unless `rank`
 * owns it, else block_table[p / (block_size*dcp)] * block_size + the
 * position's offset among the rank's tokens of that virtual block.
 * positions, block_table, slots: host arrays. */
ca_status ca_dcp_slot_mapping(const int64_t *positions, int64_t n,
                              const int32_t *block_table, int64_t n_blocks,
                              int block_size, int dcp, int rank,
                              int interleave, int64_t *slots);

/* ------------------------------------------------------------------------
 * Diagnostic of the failure path: launches one warp on `stream` that waits on
 * an mbarrier nothing ever completes.  Its bounded wait gives up after
 * `limit_cycles` SM clock cycles and raises the device error word, as a
 * stalled pipeline's waits would, without any fault.  ca_device_status then
 * reports CA_ERR_TIMEOUT, and the context stays usable.
 * Errors: CA_ERR_INVALID_ARG unless 0 < limit_cycles <= the kernels' own
 * wait limit (4e9 cycles, ~2 s).
 * ---------------------------------------------------------------------- */
ca_status ca_selftest_wait_timeout(long long limit_cycles, void *stream);

/* ------------------------------------------------------------------------
 * Device status: reads (synchronously, on the current device) the error word
 * that bounded waits set when they give up, and clears it if `reset`.
 * Returns CA_OK, CA_ERR_TIMEOUT, or CA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
ca_status ca_device_status(int reset);

#ifdef __cplusplus
}
#endif

#endif /* CTXATTN_H */
