// noalloc.cu -- kvq_attend_noalloc: decode + combine whose split-partial
// scratch lives in a fixed, library-owned device array instead of a
// caller-allocated workspace.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocator) at the
// point where they run attention -- for example a plugin hosted by a runtime
// that owns all device memory and offers no scratch allocator, or a
// latency-critical loop that must not pay cudaMalloc's implicit device
// synchronization.  They still pass their own inputs and outputs; only the
// scratch moves into this file.
//
// The scratch is one file-scope __device__ array of kNoAllocScratchBytes
// (16 MiB); every GPU that loads the library holds it until the process
// exits.  Host code must not use the array's name as a device address (on
// the host it is only a stand-in); the device address is looked up once per
// device with cudaGetSymbolAddress and passed to the kernels.
#include <mutex>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDev] = {};

// Device address of the scratch array on the current device, looked up on the
// first call made with that device current.
kvq_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return KVQ_OK;
}

}  // namespace
}  // namespace kvq

extern "C" KVQ_API kvq_status kvq_attend_noalloc(const kvq_cache* cache, const kvq_decode_params* params,
                                                 const void* q, const int32_t* block_table,
                                                 const int32_t* seq_lens, const float* head_sink, void* out,
                                                 float* lse_out, kvq_stream_t stream) {
  size_t need = 0;
  if (kvq_status s = kvq_decode_workspace_size(cache, params, &need)) return s;
  if (need > kvq::kNoAllocScratchBytes) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (kvq_status s = kvq::noalloc_scratch(&scratch)) return s;
  // Nothing in the scratch has to start at zero: kvq_decode writes the split
  // plan and every partial that kvq_combine then reads, on the same stream.
  if (kvq_status s = kvq_decode(cache, params, q, block_table, seq_lens, scratch, kvq::kNoAllocScratchBytes, stream))
    return s;
  return kvq_combine(cache, params, scratch, kvq::kNoAllocScratchBytes, head_sink, out, lse_out, stream);
}
