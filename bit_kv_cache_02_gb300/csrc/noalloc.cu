// Decode attention without a caller-provided workspace.
//
// kv_decode_attn needs device scratch for the per-split partial results.
// Some callers have no way to provide it: code embedded in a host program
// whose device memory is owned and pre-planned by another runtime (a plugin
// inside an inference server or game engine with a fixed memory budget), and
// callers on a path where a cudaMalloc would be disallowed because it can
// synchronize the device.  This entry point serves them with scratch that
// lives in the library itself: a file-scope __device__ array of fixed size,
// which every GPU that loads this library keeps until the process exits.
#include <mutex>

#include "kvq_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per device

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of g_decode_scratch for each device ordinal, looked up once
// per device (with that device current) and reused afterwards.
std::mutex g_mu;
void *g_scratch_ptr[64] = {};

int scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev < 0 || dev >= 64) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" int kv_decode_attn_noalloc(const kvq_cache *cache, int32_t num_q_heads, const uint16_t *q,
                                      float softmax_scale, uint16_t *out, int32_t max_len, void *stream) {
  const int64_t need = kv_decode_workspace_bytes(cache, num_q_heads, max_len);
  if (need < 0) {
    // same argument errors as kv_decode_attn reports
    return kv_decode_attn(cache, num_q_heads, q, softmax_scale, out, nullptr, 0, max_len, stream);
  }
  if (static_cast<uint64_t>(need) > kScratchBytes) return KVQ_ERR_WORKSPACE;
  void *scratch = nullptr;
  const int e = scratch_for_current_device(&scratch);
  if (e != KVQ_OK) return e;
  // the array is shared by calls of every geometry, so each call clears its
  // own merge counters instead of relying on the previous call to leave them zero
  return kvq::decode_attn_clearing(cache, num_q_heads, q, softmax_scale, out, scratch, kScratchBytes, max_len,
                                   stream);
}
