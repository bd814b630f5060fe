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
#include "kvq_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per device

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of g_decode_scratch in the current device's context.  The
// host-side name of the array is only a stand-in and must never reach a
// kernel.  Looked up on every call rather than cached: a cached address
// would go stale after cudaDeviceReset or under another context of the same
// device.  The first lookup on a device loads this module there (which is
// why the first call must not happen inside a stream capture); later ones
// are a table lookup.
int scratch_for_current_device(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
  *out = p;
  return KVQ_OK;
}

}  // namespace

extern "C" int kv_decode_attn_noalloc(const kvq_cache *cache, int32_t num_q_heads, const uint16_t *q,
                                      float softmax_scale, uint16_t *out, int32_t max_len, void *stream) {
  void *scratch = nullptr;
  const int e = scratch_for_current_device(&scratch);
  if (e != KVQ_OK) return e;
  // Arguments are checked exactly as kv_decode_attn checks them, then a
  // geometry whose workspace exceeds the array gets KVQ_ERR_WORKSPACE; either
  // way nothing is enqueued.  The array is shared by calls of every
  // geometry, so each call clears its own merge counters instead of relying
  // on the previous call to leave them zero.
  return kvq::decode_attn_clearing(cache, num_q_heads, q, softmax_scale, out, scratch, kScratchBytes, max_len,
                                   stream);
}
