// internal.h -- launcher interfaces between the C ABI layer (capi.cu) and the
// kernel translation units.  Every launcher enqueues on `stream`, performs no
// host synchronisation and returns the launch's cudaError_t.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ctxattn.h"

namespace ca {

// Geometry and options of one ring-attention launch (fused ring or one
// partial step).
struct RingArgs {
  const void* q;  // [B, Hq, Sq, D]
  const void* k;  // [B, Hkv, Sk, D]
  const void* v;
  int B, Hq, Hkv, D;
  int64_t Sq, Sk;     // rows per head in the q / k,v tensors
  int64_t Ls;         // rows per virtual shard
  int cp;             // ring size (schedule and causal positions)
  int q_shards;       // shards stored in q (cp for the fused ring, 1 for a step)
  int q_rank_fixed;   // logical rank of the stored q shard (-1: row r*Ls.. is rank r)
  int kv_rank_fixed;  // step: logical rank of the stored kv shard; -1: ring over cp
  int causal, layout, mode;
  float scale;        // softmax scale
  const float* c;     // const-max bound [B, Hq, Sq] (natural units) or null
  // const max with c == null: per (batch, kv head) max |k|^2 [B, Hkv]; the
  // kernel forms each row's bound from the q tile it already holds
  const float* kmax2 = nullptr;
  void* o;            // output
  int out_f32;        // 1: fp32 output rows, 0: input dtype (bf16)
  int unnormalized;   // const-max step: write acc_o instead of acc_o / acc_l
  float* lse;         // [B, Hq, Sq] or null
  unsigned* err;      // device error word
};

cudaError_t launch_ring_tc_bf16(const RingArgs& a, cudaStream_t stream);

// DCP prefill of one chunk on the tensor-core kernel's segmented schedule.
struct DcpPrefillArgs {
  const void* q;        // [Hq, Sc, D]
  const void* k_prior;  // [W, Hkv, Lcap, D]
  const void* v_prior;
  const void* k_cur;    // [W, Hkv, Lc, D]
  const void* v_cur;
  int Hq, Hkv, D, W, I;
  int64_t Sc, P, Lcap, Lc;
  float scale;
  int part_rank;        // -1: all ranks merged; else one rank's partial
  void* o;              // [Hq, Sc, D]: bf16 (merged) or fp32 (partial)
  int out_f32;
  float* lse;           // [Hq, Sc] or null
  unsigned* err;
};
constexpr int kDcpPrefillMaxRanks = 8;
cudaError_t launch_dcp_prefill_tc(const DcpPrefillArgs& d, cudaStream_t stream);
cudaError_t launch_ring_simt_f32(const RingArgs& a, cudaStream_t stream);

// kmax2[b, hk] = max over the S keys of |k|^2 (zeroes kmax2 first).
cudaError_t launch_key_max2(const void* k, int is_bf16, int B, int Hkv, int64_t S, int D,
                            float* kmax2, cudaStream_t stream);
cudaError_t launch_const_max_bound(const void* q, const void* k, int is_bf16, int B,
                                   int Hq, int Hkv, int64_t S, int D, float scale,
                                   float* c, float* kmax2, cudaStream_t stream);

// The LSE merge kernels wait on the grid dependency before they read a
// partial and are launched with programmatic stream serialization, so the
// kernel ahead of them (the decode partials, which release them early) and
// the merge overlap their launch; after any other kernel the wait is the
// ordinary stream order.  Once past the wait they release the kernel after
// them, so a following decode, launched the same way, sets up while the
// merge runs and waits before it touches global memory.
cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int n,
                             int64_t R, int D, const float* c, void* o, int out_bf16,
                             float* lse, cudaStream_t stream);

struct DecodeArgs {
  const void* q;          // [N, Hq, D] bf16
  const void* k;          // [W, N, Hkv, Lloc, D] bf16
  const void* v;
  int N, Hq, Hkv, D, W, I;
  int64_t Lloc;
  const int32_t* seq_lens;  // [N] or null
  float scale;
  int64_t stages;         // 128-token stages per (shard, sequence, KV head) pair
  int ctas;               // CTAs of the partial kernel
  int slots;              // partial slots per pair: W * slots partials per query row
  int dealt;              // 1: pairs' splits dealt round robin; 0: contiguous ranges
  int64_t split_stages;   // stages per split when dealt
  float* o_parts;         // [W*slots, N*Hq, D]
  float* lse_parts;       // [W*slots, N*Hq]
  unsigned* err;
  // paged cache (k, v are [W, nblk, Hkv, bs, D]; Lloc = max_blocks * bs)
  int paged;
  const int32_t* block_tables;  // [W, N, max_blocks]
  int64_t nblk, max_blocks;
  int bs;
  // -1: DCP shards [W, N, Hkv, Lloc, D] (interleave I); kLayoutContiguous or
  // kLayoutStriped: the ring layout [N, Hkv, W*Lloc, D], shard-major rows
  int ring_layout = -1;
};
cudaError_t launch_dcp_decode_partials(const DecodeArgs& a, cudaStream_t stream);
// Decode work geometry shared by the workspace query and the launch.  With
// many (shard, sequence, KV head) pairs (kDecodeDealPairs or more) each
// pair's 128-token stages form splits of up to 32 stages that are dealt to
// the CTAs round robin, one partial per split: the CTAs then stream
// neighbouring parts of the cache at any moment.  With fewer pairs the
// stages, pair after pair, are cut into `ctas` contiguous ranges whose
// lengths differ by at most one stage; a CTA writes one partial for each
// pair its range meets, into the pair's slot numbered by its CTA index minus
// that of the pair's first CTA, and `slots` bounds how many ranges one pair
// can meet.  The workspace query takes max_ctas = kDecodeMaxCtas, an upper
// bound of every launch's count, so it never sizes for fewer slots than a
// launch uses.
constexpr int kDecodeMaxCtas = 256;
constexpr int64_t kDecodeDealPairs = 256;
struct DecodeGeometry {
  int64_t stages;        // stages per pair
  int64_t units;         // pairs * stages (contiguous) or pairs * splits (dealt)
  int ctas;
  int slots;
  int dealt;
  int64_t split_stages;  // dealt: stages per split
};
DecodeGeometry dcp_decode_geometry(int64_t pairs, int64_t Lloc, int max_ctas);

cudaError_t launch_paged_kv_write(const void* k_new, const void* v_new, const int64_t* slots,
                                  void* k_cache, void* v_cache, int T, int Hkv, int D, int W,
                                  int64_t nblk, int bs, int elem_bytes, cudaStream_t stream);

cudaError_t launch_permute_rows(const void* src, void* dst, int64_t BH, int64_t S,
                                int64_t row_bytes, int cp, int layout, int to_shards,
                                cudaStream_t stream);
cudaError_t launch_dcp_shard_rows(const void* src, void* dst, int64_t NH, int64_t L,
                                  int64_t row_bytes, int W, int I, cudaStream_t stream);

// QK(V) prologue of const-max attention: whole-hidden RMS norm + gain +
// rotary turn for q and k, head split / transpose into the shard layout for
// q, k, v, and kmax2 of the rounded k.
struct QkvPrologueArgs {
  const void* x_q;   // [B, S, Hq*D] bf16
  const void* x_k;   // [B, S, Hkv*D]
  const void* x_v;   // [B, S, Hkv*D] or null
  const float* g_q;  // [Hq*D] or null
  const float* g_k;  // [Hkv*D] or null
  float eps;
  const float* cos;  // [S, D/2] or null
  const float* sin;
  int B, Hq, Hkv, D;
  int64_t S;
  int cp, layout;
  void* q;           // [B, Hq, S, D] bf16
  void* k;           // [B, Hkv, S, D]
  void* v;           // [B, Hkv, S, D] or null
  float* kmax2;      // [B, Hkv] or null
  unsigned* err;     // device error word
};
cudaError_t launch_qkv_prologue(const QkvPrologueArgs& a, cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// CA_OK when the current device is a GB300 (compute capability 10.3),
// CA_ERR_UNSUPPORTED for any other device, CA_ERR_CUDA if it cannot be read.
ca_status device_is_gb300();

// Host checks of a DCP decode call, everything but its workspace (capi.cu).
ca_status check_dcp_decode(const void* q, const void* k_shards, const void* v_shards,
                           ca_dtype dtype, int N, int Hq, int Hkv, int64_t Lloc, int D, int dcp,
                           int interleave, const int32_t* seq_lens, const void* o,
                           const float* lse);

}  // namespace ca
