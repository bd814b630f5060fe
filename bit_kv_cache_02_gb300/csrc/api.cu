// C ABI of the low-bit KV-cache library: argument validation, sizing and
// dispatch.  Every entry point checks its arguments before anything is
// enqueued and returns a KVQ_ERR_* code instead of throwing or aborting.
#include <cuda_runtime.h>
#include <math.h>

#include <atomic>

#include "kvq_internal.cuh"

namespace {

std::atomic<uint64_t> g_launches{0};

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Geometry checks shared by every entry point.
int check_geometry(const kvq_cache *c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->num_seqs < 1 || c->num_kv_heads < 1 || c->capacity < 1) return KVQ_ERR_INVALID_ARG;
  if (c->head_dim != kvq::kD || (c->bits != 2 && c->bits != 4) || c->group != kvq::kG) return KVQ_ERR_UNSUPPORTED;
  if (c->residual < kvq::kG || c->residual > 128 || c->residual % kvq::kG != 0) return KVQ_ERR_UNSUPPORTED;
  if (c->num_sink != 0 && c->num_sink != 1) return KVQ_ERR_UNSUPPORTED;
  if (c->pre_rope != 0 && c->pre_rope != 1) return KVQ_ERR_INVALID_ARG;
  if (c->pre_rope && !(c->rope_theta > 1.f && isfinite(c->rope_theta))) return KVQ_ERR_INVALID_ARG;
  if (c->key_per_token != 0 && c->key_per_token != 1) return KVQ_ERR_INVALID_ARG;
  if (c->key_per_token && c->pre_rope) return KVQ_ERR_UNSUPPORTED;
  if (c->hadamard != 0 && c->hadamard != 1) return KVQ_ERR_INVALID_ARG;
  if (c->hadamard && c->pre_rope) return KVQ_ERR_UNSUPPORTED;
  if (c->outliers != 0 && c->outliers != 1) return KVQ_ERR_INVALID_ARG;
  if (c->outliers && (c->pre_rope || c->hadamard)) return KVQ_ERR_UNSUPPORTED;
  if (c->block_table && c->num_blocks < 0) return KVQ_ERR_INVALID_ARG;
  if (c->num_seqs > 65535 || c->num_kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

int max_groups_of(const kvq_cache *c) {
  const int stream_cap = c->capacity > c->num_sink ? c->capacity - c->num_sink : 0;
  return (stream_cap / c->residual) * c->residual / kvq::kG;
}

// Geometry plus the buffers every kernel touches.
int check_buffers(const kvq_cache *c) {
  int e = check_geometry(c);
  if (e) return e;
  const bool need_pool = c->block_table ? c->num_blocks > 0 : max_groups_of(c) > 0;
  if ((!c->blocks && need_pool) || !c->k_res || !c->v_res || !c->seq_len) return KVQ_ERR_INVALID_ARG;
  // a paged cache that can hold groups needs at least one pool block (reads
  // through a bad table entry fall back to block 0)
  if (c->block_table && max_groups_of(c) > 0 && c->num_blocks < 1) return KVQ_ERR_INVALID_ARG;
  if (c->block_table && !aligned(c->block_table, 4)) return KVQ_ERR_ALIGNMENT;
  if (c->num_sink && (!c->k_sink || !c->v_sink)) return KVQ_ERR_INVALID_ARG;
  if (!aligned(c->blocks, 128) || !aligned(c->k_res, 16) || !aligned(c->v_res, 16) || !aligned(c->seq_len, 4))
    return KVQ_ERR_ALIGNMENT;
  if (c->num_sink && (!aligned(c->k_sink, 16) || !aligned(c->v_sink, 16))) return KVQ_ERR_ALIGNMENT;
  if (c->status && !aligned(c->status, 4)) return KVQ_ERR_ALIGNMENT;
  return KVQ_OK;
}

kvq::Geo make_geo(const kvq_cache *c) {
  kvq::Geo g;
  g.S = c->num_seqs;
  g.H = c->num_kv_heads;
  g.R = c->residual;
  g.ns = c->num_sink;
  g.bits = c->bits;
  g.pre_rope = c->pre_rope;
  g.kpt = c->key_per_token;
  g.rot = c->hadamard;
  g.sparse = c->outliers;
  g.theta = c->rope_theta;
  g.capacity = c->capacity;
  g.max_groups = max_groups_of(c);
  g.blocks = c->blocks;
  g.k_res = reinterpret_cast<__half *>(c->k_res);
  g.v_res = reinterpret_cast<__half *>(c->v_res);
  g.k_sink = reinterpret_cast<__half *>(c->k_sink);
  g.v_sink = reinterpret_cast<__half *>(c->v_sink);
  g.seq_len = c->seq_len;
  g.status = c->status;
  g.table = c->block_table;
  g.num_blocks = c->block_table ? c->num_blocks : 0;
  return g;
}

int from_cuda(cudaError_t e, uint64_t launched) {
  g_launches.fetch_add(launched);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace

extern "C" {

int32_t kvq_block_bytes(int32_t bits, int32_t head_dim, int32_t key_per_token, int32_t outliers) {
  if (head_dim != kvq::kD || (bits != 2 && bits != 4) || (key_per_token != 0 && key_per_token != 1) ||
      (outliers != 0 && outliers != 1))
    return 0;
  return kvq::block_bytes(bits, key_per_token != 0, outliers != 0);
}

int32_t kvq_max_groups(const kvq_cache *cache) {
  if (check_geometry(cache)) return -1;
  return max_groups_of(cache);
}

int64_t kvq_buffer_bytes(const kvq_cache *c, int32_t which) {
  if (check_geometry(c)) return -1;
  const int64_t sh = static_cast<int64_t>(c->num_seqs) * c->num_kv_heads;
  switch (which) {
    case KVQ_BUF_BLOCKS:
      return (c->block_table ? static_cast<int64_t>(c->num_blocks) : sh * max_groups_of(c)) *
             kvq::block_bytes(c->bits, c->key_per_token != 0, c->outliers != 0);
    case KVQ_BUF_BLOCK_TABLE: return c->block_table ? sh * max_groups_of(c) * 4 : 0;
    case KVQ_BUF_K_RES:
    case KVQ_BUF_V_RES: return sh * c->residual * kvq::kD * 2;
    case KVQ_BUF_K_SINK:
    case KVQ_BUF_V_SINK: return sh * c->num_sink * kvq::kD * 2;
    case KVQ_BUF_SEQ_LEN: return static_cast<int64_t>(c->num_seqs) * 4;
    default: return -1;
  }
}

int kv_quant_append(const kvq_cache *cache, const uint16_t *k_new, const uint16_t *v_new, const int32_t *new_len,
                    int32_t max_new, void *stream) {
  int e = check_buffers(cache);
  if (e) return e;
  if (!new_len || max_new < 0) return KVQ_ERR_INVALID_ARG;
  if (max_new > cache->capacity) return KVQ_ERR_CAPACITY;
  if (max_new > 0 && (!k_new || !v_new)) return KVQ_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(new_len, 4)) return KVQ_ERR_ALIGNMENT;
  const kvq::Geo geo = make_geo(cache);
  // grid.x of the flush kernel is bounded by the groups one append can fill
  if (static_cast<int64_t>(cache->residual - 1 + max_new) / cache->residual * (cache->residual / kvq::kG) >
      2147483647LL)
    return KVQ_ERR_UNSUPPORTED;
  uint64_t n = 0;
  cudaError_t ce = kvq::launch_quant_append(geo, reinterpret_cast<const __half *>(k_new),
                                            reinterpret_cast<const __half *>(v_new), new_len, max_new,
                                            static_cast<cudaStream_t>(stream), &n);
  return from_cuda(ce, n);
}

int64_t kv_decode_workspace_bytes(const kvq_cache *cache, int32_t num_q_heads, int32_t max_len) {
  if (check_geometry(cache)) return -1;
  if (num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0) return -1;
  const int gq = num_q_heads / cache->num_kv_heads;
  if (gq != 1 && gq != 2 && gq != 4) return -1;
  if (max_len < 1 || max_len > cache->capacity) return -1;
  return static_cast<int64_t>(kvq::plan_decode(make_geo(cache), num_q_heads, max_len).bytes);
}

static int decode_attn(const kvq_cache *cache, int32_t num_q_heads, const uint16_t *q, float softmax_scale,
                       uint16_t *out, void *workspace, size_t workspace_bytes, int32_t max_len, void *stream,
                       bool zero_counters) {
  int e = check_buffers(cache);
  if (e) return e;
  if (!q || !out || num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  const int gq = num_q_heads / cache->num_kv_heads;
  if (gq != 1 && gq != 2 && gq != 4) return KVQ_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(cache->num_seqs) * num_q_heads > 2147483647LL) return KVQ_ERR_UNSUPPORTED;
  if (max_len < 1) return KVQ_ERR_INVALID_ARG;
  if (max_len > cache->capacity) return KVQ_ERR_CAPACITY;
  if (!aligned(q, 16) || !aligned(out, 16)) return KVQ_ERR_ALIGNMENT;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) softmax_scale = 1.f / sqrtf(static_cast<float>(kvq::kD));
  const kvq::Geo geo = make_geo(cache);
  const kvq::DecodePlan plan = kvq::plan_decode(geo, num_q_heads, max_len);
  if (!workspace || workspace_bytes < plan.bytes) return KVQ_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KVQ_ERR_ALIGNMENT;
  uint64_t n = 0;
  cudaError_t ce = kvq::launch_decode(geo, num_q_heads, reinterpret_cast<const __half *>(q), softmax_scale,
                                      reinterpret_cast<__half *>(out), workspace, plan, max_len, zero_counters,
                                      static_cast<cudaStream_t>(stream), &n);
  return from_cuda(ce, n);
}

int kv_decode_attn(const kvq_cache *cache, int32_t num_q_heads, const uint16_t *q, float softmax_scale,
                   uint16_t *out, void *workspace, size_t workspace_bytes, int32_t max_len, void *stream) {
  return decode_attn(cache, num_q_heads, q, softmax_scale, out, workspace, workspace_bytes, max_len, stream, false);
}


int kv_dequant(const kvq_cache *cache, float *k_out, float *v_out, void *stream) {
  int e = check_buffers(cache);
  if (e) return e;
  if (!k_out || !v_out) return KVQ_ERR_INVALID_ARG;
  if (!aligned(k_out, 4) || !aligned(v_out, 4)) return KVQ_ERR_ALIGNMENT;
  uint64_t n = 0;
  cudaError_t ce = kvq::launch_dequant(make_geo(cache), k_out, v_out, static_cast<cudaStream_t>(stream), &n);
  return from_cuda(ce, n);
}

const char *kvq_strerror(int err) {
  switch (err) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CAPACITY: return "length exceeds cache capacity";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KVQ_ERR_ALIGNMENT: return "buffer misaligned";
    case KVQ_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown error";
  }
}

uint64_t kvq_launch_count(void) { return g_launches.load(); }

int kvq_set_decode_warps(int32_t warps) { return kvq::set_decode_warps(warps) ? KVQ_ERR_INVALID_ARG : KVQ_OK; }

int kvq_set_wait_test(int64_t limit_cycles, int32_t wait_before_fetch) {
  return kvq::set_wait_test(limit_cycles, wait_before_fetch) ? KVQ_ERR_INVALID_ARG : KVQ_OK;
}

}  // extern "C"

namespace kvq {

int decode_attn_clearing(const kvq_cache *cache, int32_t num_q_heads, const uint16_t *q, float softmax_scale,
                         uint16_t *out, void *workspace, size_t workspace_bytes, int32_t max_len, void *stream) {
  return ::decode_attn(cache, num_q_heads, q, softmax_scale, out, workspace, workspace_bytes, max_len, stream, true);
}

}  // namespace kvq
