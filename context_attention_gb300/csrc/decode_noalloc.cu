// decode_noalloc.cu -- DCP decode for callers that cannot allocate device
// memory.
//
// ca_dcp_decode() needs a caller-provided workspace for its split-KV partial
// results.  Some callers cannot provide one: code that runs inside a host
// framework whose allocator already owns all device memory (so a cudaMalloc
// of its own would fail or fragment the pool), or plugin-style enqueue paths
// that are not allowed to allocate at call time.  ca_dcp_decode_noalloc()
// serves them: it runs the same decode and merge kernels, but keeps the
// partials in a fixed scratch array that is part of this library's device
// image, so it never allocates anything itself.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes.  Every
// GPU that loads the library holds it until the process exits.  All calls on a
// device share it, so calls whose kernels overlap on the GPU (for example on
// two streams without ordering between them) race on it; callers must
// serialise them.  The decode kernel writes every partial slot it later reads
// (empty splits write o = 0 and lse = -inf), so nothing in the scratch has to
// start at zero and the previous call's leftovers are never read.
#include <cuda_runtime.h>
#include <math.h>
#include <mutex>
#include <stdint.h>

#include "../../include/ctxattn.h"
#include "internal.h"

namespace ca {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array for the current device.  In host code
// the array's name only stands for the host-side shadow symbol, so its device
// address has to be looked up once per device (with that device current).
// The cache is per device ordinal: it assumes the device's primary context
// lives as long as the process (calls after cudaDeviceReset are unsupported).
void* scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();  // the failed lookup must not surface in a later, unrelated launch check
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace ca

using namespace ca;

extern "C" ca_status ca_dcp_decode_noalloc(const void* q, const void* k_shards,
                                           const void* v_shards, ca_dtype dtype, int N, int Hq,
                                           int Hkv, int64_t Lloc, int D, int dcp, int interleave,
                                           const int32_t* seq_lens, float softmax_scale, void* o,
                                           float* lse, void* stream) {
  // the same argument checks, in the same order, as ca_dcp_decode ...
  ca_status st = check_dcp_decode(q, k_shards, v_shards, dtype, N, Hq, Hkv, Lloc, D, dcp,
                                  interleave, seq_lens, o, lse);
  if (st != CA_OK) return st;
  // ... then, in place of its workspace check, the partials must fit in the
  // built-in scratch: larger problems are rejected
  const size_t need = ca_dcp_decode_workspace_size(N, Hq, Hkv, Lloc, D, dcp, interleave);
  if (need == 0 || need > kNoAllocScratchBytes) return CA_ERR_WORKSPACE;
  // on any other GPU the library's device code (and so the scratch array)
  // does not exist: say so before looking the array up
  if ((st = device_is_gb300()) != CA_OK) return st;
  void* scratch = scratch_address();
  if (!scratch) return CA_ERR_CUDA;
  // ca_dcp_decode runs the decode and merge kernels on the partials it is
  // given; handing it the scratch array keeps this call free of any
  // allocation.
  return ca_dcp_decode(q, k_shards, v_shards, dtype, N, Hq, Hkv, Lloc, D, dcp, interleave,
                       seq_lens, softmax_scale, o, lse, scratch, kNoAllocScratchBytes, stream);
}
