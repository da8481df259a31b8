// capi.cu -- the C ABI of libctxattn.so (declared in include/ctxattn.h):
// argument validation, workspace carving and kernel dispatch.  Every entry
// point validates on the host before it touches the device; on a host-side
// error nothing is enqueued.  There is no CPU or fallback path: a case no
// kernel supports returns CA_ERR_UNSUPPORTED.
#include <atomic>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "../../include/ctxattn.h"
#include "index_maps.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ca {

// The per-device caches below (and the kernels' shared-memory attribute
// flags) may be filled by concurrent first calls from several host threads:
// they are atomic, and every writer stores the same value.

// Device error word raised by bounded waits (see ptx.cuh).  Kernels get its
// device address from device_error_word().
static __device__ unsigned g_error_word;

static unsigned* device_error_word() {
  static std::atomic<unsigned*> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
      cudaGetLastError();  // the failed lookup must not surface in a later, unrelated launch check
      return nullptr;
    }
    cache[dev] = static_cast<unsigned*>(p);
  }
  return cache[dev];
}

// Diagnostic: one warp waits on an mbarrier that nothing ever completes.
// The bounded wait gives up after `limit` cycles and raises the device
// error word, exactly as a stalled pipeline's waits would, without a fault.
__global__ void wait_timeout_kernel(unsigned* err, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_cycles(smem_u32(&bar), 0, &abort_flag, err, limit);
}

int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

static bool trace_enabled() {
  static std::atomic<int> t{-1};
  if (t < 0) {
    const char* e = getenv("CTXATTN_TRACE");
    t = (e && e[0] && e[0] != '0') ? 1 : 0;
  }
  return t == 1;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ca_status device_is_gb300() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CA_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return CA_ERR_CUDA;
  return (major == 10 && minor == 3) ? CA_OK : CA_ERR_UNSUPPORTED;
}

static ca_status launched(cudaError_t e) {
  if (e == cudaSuccess) return CA_OK;
  if (trace_enabled()) fprintf(stderr, "[ctxattn] launch failed: %s\n", cudaGetErrorString(e));
  return CA_ERR_CUDA;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static bool valid_dtype(ca_dtype d) { return d == CA_DTYPE_F32 || d == CA_DTYPE_BF16; }
static bool valid_mode(ca_mode m) { return m == CA_MODE_ONLINE_MAX || m == CA_MODE_CONST_MAX; }
static bool valid_layout(ca_layout l) {
  return l == CA_LAYOUT_CONTIGUOUS || l == CA_LAYOUT_STRIPED;
}

// Shape rules common to the attention calls.
static ca_status check_attn_shape(ca_dtype dtype, int B, int Hq, int Hkv, int64_t S, int D) {
  if (!valid_dtype(dtype)) return CA_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || D <= 0) return CA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return CA_ERR_SHAPE;
  if ((int64_t)B * Hq > 65535 && dtype == CA_DTYPE_F32) return CA_ERR_UNSUPPORTED;
  if (dtype == CA_DTYPE_BF16 && D != 128) return CA_ERR_UNSUPPORTED;
  if (dtype == CA_DTYPE_F32 && D > 128) return CA_ERR_UNSUPPORTED;
  // TMA coordinates are 32-bit
  if (dtype == CA_DTYPE_BF16 && (int64_t)B * Hq * S >= ((int64_t)1 << 31)) return CA_ERR_UNSUPPORTED;
  return CA_OK;
}

// Host checks of a DCP decode call, everything but its workspace, in the
// order ca_dcp_decode applies them (ca_dcp_decode_noalloc runs the same ones
// before it looks at its scratch).
ca_status check_dcp_decode(const void* q, const void* k_shards, const void* v_shards,
                           ca_dtype dtype, int N, int Hq, int Hkv, int64_t Lloc, int D, int dcp,
                           int interleave, const int32_t* seq_lens, const void* o,
                           const float* lse) {
  if (!q || !k_shards || !v_shards || !o) return CA_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || N <= 0 || Hq <= 0 || Hkv <= 0 || Lloc <= 0 || D <= 0 || dcp <= 0 ||
      interleave <= 0)
    return CA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || Lloc % interleave != 0) return CA_ERR_SHAPE;
  if (dtype != CA_DTYPE_BF16 || D != 128 || Hq / Hkv > 8) return CA_ERR_UNSUPPORTED;
  if ((int64_t)dcp * N * Hkv * Lloc >= ((int64_t)1 << 31)) return CA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_shards) || !aligned16(v_shards) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
      (seq_lens && (reinterpret_cast<uintptr_t>(seq_lens) & 3u)))
    return CA_ERR_ALIGNMENT;
  return CA_OK;
}

}  // namespace ca

using namespace ca;

extern "C" {

const char* ca_status_string(ca_status s) {
  switch (s) {
    case CA_OK: return "CA_OK";
    case CA_ERR_INVALID_ARG: return "CA_ERR_INVALID_ARG";
    case CA_ERR_SHAPE: return "CA_ERR_SHAPE";
    case CA_ERR_UNSUPPORTED: return "CA_ERR_UNSUPPORTED";
    case CA_ERR_ALIGNMENT: return "CA_ERR_ALIGNMENT";
    case CA_ERR_WORKSPACE: return "CA_ERR_WORKSPACE";
    case CA_ERR_CUDA: return "CA_ERR_CUDA";
    case CA_ERR_TIMEOUT: return "CA_ERR_TIMEOUT";
  }
  return "CA_ERR_UNKNOWN";
}

int ca_version(void) { return 100; }

// ------------------------------------------------------------------ ring
size_t ca_ring_attn_fwd_workspace_size(int B, int Hq, int Hkv, int64_t S, int D, int cp_size,
                                       ca_mode mode) {
  (void)D;
  (void)cp_size;
  if (mode != CA_MODE_CONST_MAX || B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0) return 0;
  return align256(sizeof(float) * (size_t)B * Hkv);  // kmax2
}

static ca_status ring_common(const void* q, const void* k, const void* v, const float* c,
                             const float* kmax2, void* o,
                             float* lse, ca_dtype dtype, int B, int Hq, int Hkv, int64_t S, int D,
                             int cp_size, ca_mode mode, int causal, ca_layout layout,
                             float softmax_scale, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!q || !k || !v || !o) return CA_ERR_INVALID_ARG;
  if (!valid_mode(mode) || !valid_layout(layout) || cp_size <= 0) return CA_ERR_INVALID_ARG;
  ca_status st = check_attn_shape(dtype, B, Hq, Hkv, S, D);
  if (st != CA_OK) return st;
  if (S % cp_size != 0) return CA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) || (c && (reinterpret_cast<uintptr_t>(c) & 3u)) ||
      (kmax2 && (reinterpret_cast<uintptr_t>(kmax2) & 3u)))
    return CA_ERR_ALIGNMENT;
  const bool own_bound = mode == CA_MODE_CONST_MAX && c == nullptr && kmax2 == nullptr;
  const size_t need = own_bound ? ca_ring_attn_fwd_workspace_size(B, Hq, Hkv, S, D, cp_size, mode) : 0;
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return CA_ERR_WORKSPACE;
  if (dtype == CA_DTYPE_BF16 && (st = device_is_gb300()) != CA_OK) return st;
  unsigned* err = device_error_word();
  if (!err) return CA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);

  RingArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.Sq = S;
  a.Sk = S;
  a.Ls = S / cp_size;
  a.cp = cp_size;
  a.q_shards = cp_size;
  a.q_rank_fixed = -1;
  a.kv_rank_fixed = -1;
  a.causal = causal ? 1 : 0;
  a.layout = (int)layout;
  a.mode = (int)mode;
  a.scale = scale;
  a.c = c;
  a.kmax2 = kmax2;
  a.o = o;
  a.out_f32 = dtype == CA_DTYPE_F32;
  a.unnormalized = 0;
  a.lse = lse;
  a.err = err;
  if (own_bound) {
    // the key pass only: both kernels form each row's bound from the q rows
    // they load anyway
    float* kw = static_cast<float*>(workspace);
    cudaError_t e = launch_key_max2(k, dtype == CA_DTYPE_BF16, B, Hkv, S, D, kw, s);
    if (e != cudaSuccess) return launched(e);
    a.kmax2 = kw;
  }
  if (trace_enabled())
    fprintf(stderr, "[ctxattn] ring_attn_fwd dtype=%d B=%d Hq=%d Hkv=%d S=%lld D=%d cp=%d mode=%d causal=%d layout=%d\n",
            (int)dtype, B, Hq, Hkv, (long long)S, D, cp_size, (int)mode, a.causal, a.layout);
  return launched(dtype == CA_DTYPE_BF16 ? launch_ring_tc_bf16(a, s) : launch_ring_simt_f32(a, s));
}

ca_status ca_ring_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                           ca_dtype dtype, int B, int Hq, int Hkv, int64_t S, int D, int cp_size,
                           ca_mode mode, int causal, ca_layout layout, float softmax_scale,
                           void* workspace, size_t workspace_bytes, void* stream) {
  return ring_common(q, k, v, nullptr, nullptr, o, lse, dtype, B, Hq, Hkv, S, D, cp_size, mode,
                     causal, layout, softmax_scale, workspace, workspace_bytes, stream);
}

ca_status ca_ring_attn_fwd_bounded(const void* q, const void* k, const void* v, const float* c,
                                   void* o, float* lse, ca_dtype dtype, int B, int Hq, int Hkv,
                                   int64_t S, int D, int cp_size, int causal, ca_layout layout,
                                   float softmax_scale, void* stream) {
  if (!c) return CA_ERR_INVALID_ARG;
  return ring_common(q, k, v, c, nullptr, o, lse, dtype, B, Hq, Hkv, S, D, cp_size,
                     CA_MODE_CONST_MAX, causal, layout, softmax_scale, nullptr, 0, stream);
}

ca_status ca_ring_attn_fwd_kmax(const void* q, const void* k, const void* v, const float* kmax2,
                                void* o, float* lse, ca_dtype dtype, int B, int Hq, int Hkv,
                                int64_t S, int D, int cp_size, int causal, ca_layout layout,
                                float softmax_scale, void* stream) {
  if (!kmax2) return CA_ERR_INVALID_ARG;
  return ring_common(q, k, v, nullptr, kmax2, o, lse, dtype, B, Hq, Hkv, S, D, cp_size,
                     CA_MODE_CONST_MAX, causal, layout, softmax_scale, nullptr, 0, stream);
}

ca_status ca_attn_partial_step(const void* q_shard, const void* k_shard, const void* v_shard,
                               ca_dtype dtype, int B, int Hq, int Hkv, int64_t Ls, int D,
                               int q_rank, int kv_rank, int cp_size, ca_mode mode, int causal,
                               ca_layout layout, float softmax_scale, const float* c,
                               float* o_part, float* lse_part, void* stream) {
  if (!q_shard || !k_shard || !v_shard || !o_part || !lse_part) return CA_ERR_INVALID_ARG;
  if (!valid_mode(mode) || !valid_layout(layout) || cp_size <= 0) return CA_ERR_INVALID_ARG;
  if (q_rank < 0 || q_rank >= cp_size || kv_rank < 0 || kv_rank >= cp_size) return CA_ERR_INVALID_ARG;
  if ((mode == CA_MODE_CONST_MAX) != (c != nullptr)) return CA_ERR_INVALID_ARG;
  ca_status st = check_attn_shape(dtype, B, Hq, Hkv, Ls, D);
  if (st != CA_OK) return st;
  if (!aligned16(q_shard) || !aligned16(k_shard) || !aligned16(v_shard) || !aligned16(o_part) ||
      (reinterpret_cast<uintptr_t>(lse_part) & 3u) || (c && (reinterpret_cast<uintptr_t>(c) & 3u)))
    return CA_ERR_ALIGNMENT;
  if (dtype == CA_DTYPE_BF16 && (st = device_is_gb300()) != CA_OK) return st;
  unsigned* err = device_error_word();
  if (!err) return CA_ERR_CUDA;
  RingArgs a;
  a.q = q_shard;
  a.k = k_shard;
  a.v = v_shard;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.Sq = Ls;
  a.Sk = Ls;
  a.Ls = Ls;
  a.cp = cp_size;
  a.q_shards = 1;
  a.q_rank_fixed = q_rank;
  a.kv_rank_fixed = kv_rank;
  a.causal = causal ? 1 : 0;
  a.layout = (int)layout;
  a.mode = (int)mode;
  a.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
  a.c = c;
  a.o = o_part;
  a.out_f32 = 1;
  a.unnormalized = mode == CA_MODE_CONST_MAX;
  a.lse = lse_part;
  a.err = err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return launched(dtype == CA_DTYPE_BF16 ? launch_ring_tc_bf16(a, s) : launch_ring_simt_f32(a, s));
}

// ------------------------------------------------------------------ merge
ca_status ca_lse_merge(const float* o_parts, const float* lse_parts, int n, int64_t R, int D,
                       const float* c, void* o, ca_dtype out_dtype, float* lse, void* stream) {
  if (!o_parts || !lse_parts || !o || n <= 0 || R <= 0 || D <= 0) return CA_ERR_INVALID_ARG;
  if (!valid_dtype(out_dtype)) return CA_ERR_INVALID_ARG;
  if (D % 4 != 0 || D > 512) return CA_ERR_UNSUPPORTED;
  if (!aligned16(o_parts) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) || (c && (reinterpret_cast<uintptr_t>(c) & 3u)))
    return CA_ERR_ALIGNMENT;
  return launched(launch_lse_merge(o_parts, lse_parts, n, R, D, c, o, out_dtype == CA_DTYPE_BF16,
                                   lse, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ bound
ca_status ca_const_max_bound(const void* q, const void* k, ca_dtype dtype, int B, int Hq, int Hkv,
                             int64_t S, int D, float softmax_scale, float* c, float* kmax2,
                             void* stream) {
  if (!q || !k || !c || !kmax2) return CA_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || D <= 0)
    return CA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return CA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || (reinterpret_cast<uintptr_t>(c) & 3u) ||
      (reinterpret_cast<uintptr_t>(kmax2) & 3u))
    return CA_ERR_ALIGNMENT;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
  return launched(launch_const_max_bound(q, k, dtype == CA_DTYPE_BF16, B, Hq, Hkv, S, D, scale, c,
                                         kmax2, static_cast<cudaStream_t>(stream)));
}

ca_status ca_key_max2(const void* k, ca_dtype dtype, int B, int Hkv, int64_t S, int D, float* kmax2,
                      void* stream) {
  if (!k || !kmax2) return CA_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || B <= 0 || Hkv <= 0 || S <= 0 || D <= 0) return CA_ERR_INVALID_ARG;
  if (!aligned16(k) || (reinterpret_cast<uintptr_t>(kmax2) & 3u)) return CA_ERR_ALIGNMENT;
  return launched(launch_key_max2(k, dtype == CA_DTYPE_BF16, B, Hkv, S, D, kmax2,
                                  static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ prologue
ca_status ca_qkv_prologue(const void* x_q, const void* x_k, const void* x_v, const float* g_q,
                          const float* g_k, float eps, const float* rope_cos,
                          const float* rope_sin, ca_dtype dtype, int B, int64_t S, int Hq,
                          int Hkv, int D, int cp_size, ca_layout layout, void* q, void* k,
                          void* v, float* kmax2, void* stream) {
  if (!x_q || !x_k || !q || !k || (x_v && !v) || (!rope_cos != !rope_sin)) return CA_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || !valid_layout(layout) || B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 ||
      cp_size <= 0 || !(eps >= 0.f))
    return CA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || S % cp_size != 0) return CA_ERR_SHAPE;
  if (dtype != CA_DTYPE_BF16 || (D != 64 && D != 128) || (int64_t)Hq * D > 8192) return CA_ERR_UNSUPPORTED;
  if ((int64_t)B * S * 3 >= ((int64_t)1 << 31)) return CA_ERR_UNSUPPORTED;  // 32-bit row indices
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!aligned16(x_q) || !aligned16(x_k) || (x_v && !aligned16(x_v)) || !aligned16(q) ||
      !aligned16(k) || (v && !aligned16(v)) || (g_q && !aligned16(g_q)) || (g_k && !aligned16(g_k)) ||
      (rope_cos && (!aligned16(rope_cos) || !aligned16(rope_sin))) || (kmax2 && !a4(kmax2)))
    return CA_ERR_ALIGNMENT;
  QkvPrologueArgs a;
  a.x_q = x_q;
  a.x_k = x_k;
  a.x_v = x_v;
  a.g_q = g_q;
  a.g_k = g_k;
  a.eps = eps;
  a.cos = rope_cos;
  a.sin = rope_sin;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.S = S;
  a.cp = cp_size;
  a.layout = (int)layout;
  a.q = q;
  a.k = k;
  a.v = x_v ? v : nullptr;
  a.kmax2 = kmax2;
  a.err = device_error_word();
  if (!a.err) return CA_ERR_CUDA;
  return launched(launch_qkv_prologue(a, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ decode
size_t ca_dcp_decode_workspace_size(int N, int Hq, int Hkv, int64_t Lloc, int D, int dcp,
                                    int interleave) {
  (void)interleave;
  if (N <= 0 || Hq <= 0 || Hkv <= 0 || Lloc <= 0 || D <= 0 || dcp <= 0) return 0;
  const DecodeGeometry g = dcp_decode_geometry((int64_t)dcp * N * Hkv, Lloc, kDecodeMaxCtas);
  const size_t parts = (size_t)dcp * g.slots;
  return align256(sizeof(float) * parts * N * Hq * D) + align256(sizeof(float) * parts * N * Hq);
}

// The decode entry points share one kernel pair: these fill the arguments
// they have in common, then place the split-KV partials in the workspace and
// launch the partial kernel and the LSE merge on the caller's stream.
static DecodeArgs decode_args(const void* q, const void* k, const void* v, int N, int Hq, int Hkv,
                              int D, int W, int I, int64_t Lloc, const int32_t* seq_lens,
                              float softmax_scale) {
  DecodeArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.N = N;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.D = D;
  a.W = W;
  a.I = I;
  a.Lloc = Lloc;
  a.seq_lens = seq_lens;
  a.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
  a.paged = 0;
  a.block_tables = nullptr;
  a.nblk = a.max_blocks = 0;
  a.bs = 0;
  return a;
}

static ca_status decode_run(DecodeArgs& a, void* workspace, void* o, float* lse, void* stream) {
  ca_status st = device_is_gb300();
  if (st != CA_OK) return st;
  unsigned* err = device_error_word();
  if (!err) return CA_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return CA_ERR_CUDA;
  const DecodeGeometry g = dcp_decode_geometry((int64_t)a.W * a.N * a.Hkv, a.Lloc,
                                               sms < kDecodeMaxCtas ? sms : kDecodeMaxCtas);
  a.stages = g.stages;
  a.ctas = g.ctas;
  a.slots = g.slots;
  a.dealt = g.dealt;
  a.split_stages = g.split_stages;
  const size_t parts = (size_t)a.W * a.slots;
  a.o_parts = static_cast<float*>(workspace);
  a.lse_parts = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         align256(sizeof(float) * parts * a.N * a.Hq * a.D));
  a.err = err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_dcp_decode_partials(a, s);
  if (e != cudaSuccess) return launched(e);
  return launched(launch_lse_merge(a.o_parts, a.lse_parts, (int)parts, (int64_t)a.N * a.Hq, a.D, nullptr,
                                   o, 1, lse, s));
}

ca_status ca_dcp_decode(const void* q, const void* k_shards, const void* v_shards, ca_dtype dtype,
                        int N, int Hq, int Hkv, int64_t Lloc, int D, int dcp, int interleave,
                        const int32_t* seq_lens, float softmax_scale, void* o, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream) {
  const ca_status chk = check_dcp_decode(q, k_shards, v_shards, dtype, N, Hq, Hkv, Lloc, D, dcp,
                                         interleave, seq_lens, o, lse);
  if (chk != CA_OK) return chk;
  const size_t need = ca_dcp_decode_workspace_size(N, Hq, Hkv, Lloc, D, dcp, interleave);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return CA_ERR_WORKSPACE;
  DecodeArgs a = decode_args(q, k_shards, v_shards, N, Hq, Hkv, D, dcp, interleave, Lloc, seq_lens,
                             softmax_scale);
  return decode_run(a, workspace, o, lse, stream);
}

size_t ca_ring_decode_workspace_size(int B, int Hq, int Hkv, int64_t S, int D, int cp_size) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || D <= 0 || cp_size <= 0 || S % cp_size != 0) return 0;
  const DecodeGeometry g =
      dcp_decode_geometry((int64_t)cp_size * B * Hkv, S / cp_size, kDecodeMaxCtas);
  const size_t parts = (size_t)cp_size * g.slots;
  return align256(sizeof(float) * parts * B * Hq * D) + align256(sizeof(float) * parts * B * Hq);
}

ca_status ca_ring_decode(const void* q, const void* k, const void* v, ca_dtype dtype, int B, int Hq,
                         int Hkv, int64_t S, int D, int cp_size, ca_layout layout,
                         const int32_t* seq_lens, float softmax_scale, void* o, float* lse,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o) return CA_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || !valid_layout(layout) || B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 ||
      D <= 0 || cp_size <= 0)
    return CA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || S % cp_size != 0) return CA_ERR_SHAPE;
  if (dtype != CA_DTYPE_BF16 || D != 128 || Hq / Hkv > 8) return CA_ERR_UNSUPPORTED;
  if ((int64_t)B * Hkv * S >= ((int64_t)1 << 31)) return CA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
      (seq_lens && (reinterpret_cast<uintptr_t>(seq_lens) & 3u)))
    return CA_ERR_ALIGNMENT;
  const size_t need = ca_ring_decode_workspace_size(B, Hq, Hkv, S, D, cp_size);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return CA_ERR_WORKSPACE;
  // the decode kernel over the ring layout: sequence n = batch element b,
  // W = cp shards of Lloc = S/cp rows each
  DecodeArgs a = decode_args(q, k, v, B, Hq, Hkv, D, cp_size, 1, S / cp_size, seq_lens, softmax_scale);
  a.ring_layout = (int)layout;
  return decode_run(a, workspace, o, lse, stream);
}

ca_status ca_dcp_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, ca_dtype dtype, int N, int Hq, int Hkv,
                              int64_t nblk, int block_size, int64_t max_blocks, int D, int dcp,
                              int interleave, const int32_t* seq_lens, float softmax_scale, void* o,
                              float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !o) return CA_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || N <= 0 || Hq <= 0 || Hkv <= 0 || nblk <= 0 || block_size <= 0 ||
      max_blocks <= 0 || D <= 0 || dcp <= 0 || interleave <= 0)
    return CA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return CA_ERR_SHAPE;
  if (dtype != CA_DTYPE_BF16 || D != 128 || Hq / Hkv > 8) return CA_ERR_UNSUPPORTED;
  if (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64 &&
      block_size != 128)
    return CA_ERR_UNSUPPORTED;
  if ((int64_t)dcp * nblk * Hkv * block_size >= ((int64_t)1 << 31)) return CA_ERR_UNSUPPORTED;
  // the slots the block tables address, as the kernel's 32-bit work walk counts them
  if ((int64_t)dcp * N * Hkv * max_blocks * block_size >= ((int64_t)1 << 31)) return CA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return CA_ERR_ALIGNMENT;
  const int64_t Lloc = max_blocks * block_size;
  const size_t need = ca_dcp_decode_workspace_size(N, Hq, Hkv, Lloc, D, dcp, interleave);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return CA_ERR_WORKSPACE;
  DecodeArgs a = decode_args(q, k_cache, v_cache, N, Hq, Hkv, D, dcp, interleave, Lloc, seq_lens,
                             softmax_scale);
  a.paged = 1;
  a.block_tables = block_tables;
  a.nblk = nblk;
  a.max_blocks = max_blocks;
  a.bs = block_size;
  return decode_run(a, workspace, o, lse, stream);
}

ca_status ca_paged_kv_write(const void* k_new, const void* v_new, const int64_t* slots,
                            void* k_cache, void* v_cache, ca_dtype dtype, int T, int Hkv, int D,
                            int dcp, int64_t nblk, int block_size, void* stream) {
  if (!k_new || !v_new || !slots || !k_cache || !v_cache) return CA_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || T < 0 || Hkv <= 0 || D <= 0 || dcp <= 0 || nblk <= 0 ||
      block_size <= 0)
    return CA_ERR_INVALID_ARG;
  const int elem = dtype == CA_DTYPE_BF16 ? 2 : 4;
  if ((D * elem) % 16 != 0) return CA_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slots) & 7u))
    return CA_ERR_ALIGNMENT;
  return launched(launch_paged_kv_write(k_new, v_new, slots, k_cache, v_cache, T, Hkv, D, dcp, nblk,
                                        block_size, elem, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ DCP prefill
static ca_status dcp_prefill_common(const void* q, const void* k_prior, const void* v_prior,
                                    const void* k_cur, const void* v_cur, ca_dtype dtype, int Hq,
                                    int Hkv, int64_t Sc, int D, int dcp, int interleave,
                                    int64_t prior_tokens, int64_t Lcap, int64_t Lc, int rank,
                                    float softmax_scale, void* o, int out_f32, float* lse,
                                    void* stream) {
  if (!q || !k_prior || !v_prior || !k_cur || !v_cur || !o) return CA_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || Hq <= 0 || Hkv <= 0 || Sc <= 0 || D <= 0 || dcp <= 0 ||
      interleave <= 0 || prior_tokens < 0 || Lcap <= 0 || Lc <= 0)
    return CA_ERR_INVALID_ARG;
  if (rank >= dcp) return CA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return CA_ERR_SHAPE;
  if (dtype != CA_DTYPE_BF16 || D != 128 || dcp > kDcpPrefillMaxRanks) return CA_ERR_UNSUPPORTED;
  if (Lcap < dcp_local_filled(prior_tokens, dcp, interleave, interleave, 0) ||
      Lc < dcp_local_filled(Sc, dcp, interleave, interleave, 0))
    return CA_ERR_SHAPE;
  if ((int64_t)Hq * Sc >= ((int64_t)1 << 31) || Lcap >= ((int64_t)1 << 31)) return CA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_prior) || !aligned16(v_prior) || !aligned16(k_cur) ||
      !aligned16(v_cur) || !aligned16(o) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return CA_ERR_ALIGNMENT;
  ca_status st = device_is_gb300();
  if (st != CA_OK) return st;
  unsigned* err = device_error_word();
  if (!err) return CA_ERR_CUDA;
  DcpPrefillArgs d;
  d.q = q;
  d.k_prior = k_prior;
  d.v_prior = v_prior;
  d.k_cur = k_cur;
  d.v_cur = v_cur;
  d.Hq = Hq;
  d.Hkv = Hkv;
  d.D = D;
  d.W = dcp;
  d.I = interleave;
  d.Sc = Sc;
  d.P = prior_tokens;
  d.Lcap = Lcap;
  d.Lc = Lc;
  d.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)D);
  d.part_rank = rank;
  d.o = o;
  d.out_f32 = out_f32;
  d.lse = lse;
  d.err = err;
  return launched(launch_dcp_prefill_tc(d, static_cast<cudaStream_t>(stream)));
}

ca_status ca_dcp_prefill(const void* q, const void* k_prior, const void* v_prior, const void* k_cur,
                         const void* v_cur, ca_dtype dtype, int Hq, int Hkv, int64_t Sc, int D,
                         int dcp, int interleave, int64_t prior_tokens, int64_t Lcap, int64_t Lc,
                         float softmax_scale, void* o, float* lse, void* stream) {
  return dcp_prefill_common(q, k_prior, v_prior, k_cur, v_cur, dtype, Hq, Hkv, Sc, D, dcp,
                            interleave, prior_tokens, Lcap, Lc, -1, softmax_scale, o, 0, lse,
                            stream);
}

ca_status ca_dcp_prefill_partial(const void* q, const void* k_prior, const void* v_prior,
                                 const void* k_cur, const void* v_cur, ca_dtype dtype, int Hq,
                                 int Hkv, int64_t Sc, int D, int dcp, int interleave,
                                 int64_t prior_tokens, int64_t Lcap, int64_t Lc, int rank,
                                 float softmax_scale, float* o_part, float* lse_part,
                                 void* stream) {
  if (rank < 0 || !lse_part) return CA_ERR_INVALID_ARG;
  return dcp_prefill_common(q, k_prior, v_prior, k_cur, v_cur, dtype, Hq, Hkv, Sc, D, dcp,
                            interleave, prior_tokens, Lcap, Lc, rank, softmax_scale, o_part, 1,
                            lse_part, stream);
}

// ------------------------------------------------------------------ layouts
static ca_status check_rows(const void* a, const void* b, int64_t BH, int64_t S, int64_t row_bytes) {
  if (!a || !b || BH <= 0 || S <= 0 || row_bytes <= 0) return CA_ERR_INVALID_ARG;
  if (row_bytes % 16 != 0) return CA_ERR_UNSUPPORTED;
  if (!aligned16(a) || !aligned16(b)) return CA_ERR_ALIGNMENT;
  return CA_OK;
}

ca_status ca_layout_to_shards(const void* x, void* y, int64_t BH, int64_t S, int64_t row_bytes,
                              int cp_size, ca_layout layout, void* stream) {
  ca_status st = check_rows(x, y, BH, S, row_bytes);
  if (st != CA_OK) return st;
  if (cp_size <= 0 || !valid_layout(layout)) return CA_ERR_INVALID_ARG;
  if (S % cp_size != 0) return CA_ERR_SHAPE;
  return launched(launch_permute_rows(x, y, BH, S, row_bytes, cp_size, (int)layout, 1,
                                      static_cast<cudaStream_t>(stream)));
}

ca_status ca_layout_from_shards(const void* y, void* x, int64_t BH, int64_t S, int64_t row_bytes,
                                int cp_size, ca_layout layout, void* stream) {
  ca_status st = check_rows(y, x, BH, S, row_bytes);
  if (st != CA_OK) return st;
  if (cp_size <= 0 || !valid_layout(layout)) return CA_ERR_INVALID_ARG;
  if (S % cp_size != 0) return CA_ERR_SHAPE;
  return launched(launch_permute_rows(y, x, BH, S, row_bytes, cp_size, (int)layout, 0,
                                      static_cast<cudaStream_t>(stream)));
}

ca_status ca_dcp_shard_kv(const void* kv, void* shards, int64_t NH, int64_t L, int64_t row_bytes,
                          int dcp, int interleave, void* stream) {
  ca_status st = check_rows(kv, shards, NH, L, row_bytes);
  if (st != CA_OK) return st;
  if (dcp <= 0 || interleave <= 0) return CA_ERR_INVALID_ARG;
  if (L % ((int64_t)dcp * interleave) != 0) return CA_ERR_SHAPE;
  return launched(launch_dcp_shard_rows(kv, shards, NH, L, row_bytes, dcp, interleave,
                                        static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ host index helpers
int64_t ca_layout_global_index(ca_layout layout, int cp_size, int64_t Ls, int64_t row) {
  if (!valid_layout(layout) || cp_size <= 0 || Ls <= 0 || row < 0 || row >= Ls * cp_size) return -1;
  return layout_global((int)layout, cp_size, Ls, (int)(row / Ls), row % Ls);
}

int64_t ca_layout_shard_row(ca_layout layout, int cp_size, int64_t Ls, int64_t token) {
  if (!valid_layout(layout) || cp_size <= 0 || Ls <= 0 || token < 0 || token >= Ls * cp_size)
    return -1;
  int r;
  int64_t a;
  layout_locate((int)layout, cp_size, Ls, token, &r, &a);
  return (int64_t)r * Ls + a;
}

int ca_ring_kv_shard(int rank, int step, int cp_size) {
  if (cp_size <= 0 || rank < 0 || rank >= cp_size || step < 0) return -1;
  return ring_kv_shard(rank, step, cp_size);
}

int ca_dcp_owner(int64_t pos, int dcp, int interleave) {
  if (pos < 0 || dcp <= 0 || interleave <= 0) return -1;
  return dcp_owner(pos, dcp, interleave);
}

int64_t ca_dcp_local_index(int64_t pos, int dcp, int interleave) {
  if (pos < 0 || dcp <= 0 || interleave <= 0) return -1;
  return dcp_local_index(pos, dcp, interleave);
}

int64_t ca_dcp_local_to_global(int64_t local, int rank, int dcp, int interleave) {
  if (local < 0 || dcp <= 0 || interleave <= 0 || rank < 0 || rank >= dcp) return -1;
  return dcp_local_to_global(local, rank, dcp, interleave);
}

int64_t ca_dcp_local_filled(int64_t N, int dcp, int interleave, int block_size, int rank) {
  if (N < 0 || dcp <= 0 || interleave <= 0 || block_size <= 0 || rank < 0 || rank >= dcp) return -1;
  return dcp_local_filled(N, dcp, interleave, block_size, rank);
}

int ca_dcp_active_mask(int64_t N, int dcp, int interleave, int block_size, int rank) {
  if (N < 0 || dcp <= 0 || interleave <= 0 || block_size <= 0 || rank < 0 || rank >= dcp) return -1;
  return dcp_active_mask(N, dcp, interleave, block_size, rank);
}

ca_status ca_dcp_slot_mapping(const int64_t* positions, int64_t n, const int32_t* block_table,
                              int64_t n_blocks, int block_size, int dcp, int rank, int interleave,
                              int64_t* slots) {
  if (!positions || !block_table || !slots || n < 0 || n_blocks <= 0 || block_size <= 0 ||
      dcp <= 0 || interleave <= 0 || rank < 0 || rank >= dcp)
    return CA_ERR_INVALID_ARG;
  if (block_size % interleave != 0) return CA_ERR_SHAPE;
  const int64_t vblock = (int64_t)block_size * dcp;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t p = positions[i];
    if (p < 0 || p / vblock >= n_blocks) return CA_ERR_INVALID_ARG;
  }
  for (int64_t i = 0; i < n; ++i) {
    const int64_t p = positions[i];
    const int64_t off = p % vblock;  // position inside its virtual block
    if (dcp_owner(off, dcp, interleave) != rank) {
      slots[i] = -1;
      continue;
    }
    slots[i] = (int64_t)block_table[p / vblock] * block_size + dcp_local_index(off, dcp, interleave);
  }
  return CA_OK;
}

// ------------------------------------------------------------------ status
ca_status ca_selftest_wait_timeout(long long limit_cycles, void* stream) {
  if (limit_cycles <= 0 || limit_cycles > kWaitLimitCycles) return CA_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return CA_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, limit_cycles);
  return launched(cudaGetLastError());
}

ca_status ca_device_status(int reset) {
  unsigned* p = device_error_word();
  if (!p) return CA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return CA_ERR_CUDA;
  if (reset && v) {
    const unsigned z = 0;
    if (cudaMemcpy(p, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return CA_ERR_CUDA;
  }
  return v ? CA_ERR_TIMEOUT : CA_OK;
}

}  // extern "C"
