// C ABI of the kvq library: argument validation on the host, then launches.
// Every check happens before any CUDA call, so a rejected call touches
// neither the GPU nor the stream.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_type(int t) { return t >= KVQ_TYPE_Q4_0 && t <= KVQ_TYPE_Q5_1; }
bool has_qh(int t) { return t == KVQ_TYPE_Q5_0 || t == KVQ_TYPE_Q5_1; }
bool has_min(int t) { return t == KVQ_TYPE_Q4_1 || t == KVQ_TYPE_Q5_1; }
bool valid_dtype(int t) { return t == KVQ_F32 || t == KVQ_BF16 || t == KVQ_F16; }

// sizes and types only (no pointers)
bool shape_ok(const kvq_cache* c) {
  if (!c) return false;
  if (c->batch <= 0 || c->batch > 65535 || c->n_kv_heads <= 0 || c->n_kv_heads > 4096) return false;
  if (c->head_dim < 32 || c->head_dim > 512 || c->head_dim % 32) return false;
  // positions, chunk ends and seq_len + n_new stay below 2^31 in the kernels' int arithmetic
  if (c->max_ctx <= 0 || c->max_ctx % 64 || c->max_ctx > (1 << 30)) return false;
  if (c->tail_len < 0 || c->tail_len > (1 << 24)) return false;
  if (!valid_type(c->k_type) || !valid_type(c->v_type)) return false;
  if (c->flags & ~(KVQ_ROT_AUTO | KVQ_ROT_K_OFF | KVQ_ROT_V_OFF)) return false;
  // paged layout: pages of a multiple of 64 tokens that divide the capacity
  if (c->page_tokens < 0 || c->n_pages < 0) return false;
  if (c->page_tokens && (c->page_tokens % 64 || c->max_ctx % c->page_tokens || c->n_pages == 0)) return false;
  if (!c->page_tokens && c->n_pages) return false;
  // outlier channels: 32 per KV head, below head_dim
  if (c->n_outlier != 0 && (c->n_outlier != 32 || c->head_dim < 64)) return false;
  // every plane offset must stay below 2^62 bytes
  const double rows = double(c->batch) * c->n_kv_heads * c->max_ctx;
  const double prow = double(c->n_pages) * c->n_kv_heads * c->page_tokens;
  if (rows * c->head_dim * 2 > 4.0e18 || prow * c->head_dim * 2 > 4.0e18) return false;
  return true;
}

size_t plane_bytes(const kvq_cache* c, int plane) {
  const size_t rows = c->page_tokens ? size_t(c->n_pages) * c->n_kv_heads * c->page_tokens
                                     : size_t(c->batch) * c->n_kv_heads * c->max_ctx;
  const size_t nb = size_t(c->head_dim) / 32;
  const size_t d = size_t(c->head_dim);
  switch (plane) {
    case KVQ_PLANE_K_QS: return rows * kvq::qs_row_bytes_host(c->k_type, c->head_dim);
    case KVQ_PLANE_V_QS: return rows * kvq::qs_row_bytes_host(c->v_type, c->head_dim);
    case KVQ_PLANE_K_QH: return has_qh(c->k_type) ? rows * nb * 4 : 0;
    case KVQ_PLANE_V_QH: return has_qh(c->v_type) ? rows * nb * 4 : 0;
    case KVQ_PLANE_K_D: return rows * nb * (has_min(c->k_type) ? 4 : 2);
    case KVQ_PLANE_V_D: return rows * nb * (has_min(c->v_type) ? 4 : 2);
    case KVQ_PLANE_K_TAIL:
    case KVQ_PLANE_V_TAIL: return size_t(c->batch) * c->n_kv_heads * size_t(c->tail_len) * d * 2;
    case KVQ_PLANE_SEQ_LEN: return size_t(c->batch) * 4;
    case KVQ_PLANE_STATUS: return 16;
    case KVQ_PLANE_OUTLIER: return c->n_outlier ? rows / 16 * 1088 : 0;  // rows is a multiple of 64
    case KVQ_PLANE_OUTLIER_IDX: return size_t(c->n_kv_heads) * size_t(c->n_outlier) * 4;
    default: return 0;
  }
}

kvq_status check_cache(const kvq_cache* c) {
  if (!shape_ok(c)) return KVQ_ERR_INVALID_ARG;
  const void* must[] = {c->k_qs, c->k_d, c->v_qs, c->v_d, c->seq_len, c->status};
  for (const void* p : must)
    if (!p || !aligned16(p)) return KVQ_ERR_INVALID_ARG;
  if (c->page_tokens && (!c->page_table || (reinterpret_cast<uintptr_t>(c->page_table) & 3u))) return KVQ_ERR_INVALID_ARG;
  if (!c->page_tokens && c->page_table) return KVQ_ERR_INVALID_ARG;
  if (has_qh(c->k_type) != (c->k_qh != nullptr)) return KVQ_ERR_INVALID_ARG;
  if (has_qh(c->v_type) != (c->v_qh != nullptr)) return KVQ_ERR_INVALID_ARG;
  if (c->k_qh && !aligned16(c->k_qh)) return KVQ_ERR_INVALID_ARG;
  if (c->v_qh && !aligned16(c->v_qh)) return KVQ_ERR_INVALID_ARG;
  const bool has_tail = c->tail_len > 0;
  if (has_tail != (c->k_tail != nullptr) || has_tail != (c->v_tail != nullptr)) return KVQ_ERR_INVALID_ARG;
  if (has_tail && (!aligned16(c->k_tail) || !aligned16(c->v_tail))) return KVQ_ERR_INVALID_ARG;
  const void* outl[] = {c->outlier_idx, c->outl};
  for (const void* p : outl) {
    if (c->n_outlier && (!p || !aligned16(p))) return KVQ_ERR_INVALID_ARG;
    if (!c->n_outlier && p) return KVQ_ERR_INVALID_ARG;
  }
  return KVQ_OK;
}

kvq_status resolve(const kvq_cache* c, kvq::Rot* r) {
  const int d = c->head_dim;
  const bool eligible = d >= 64 && d % 64 == 0;
  const bool want_k = !(c->flags & KVQ_ROT_K_OFF);
  const bool want_v = !(c->flags & KVQ_ROT_V_OFF);
  if (c->flags & KVQ_ROT_AUTO) {
    r->k = eligible && want_k;
    r->v = eligible && want_v;
    return KVQ_OK;
  }
  if ((want_k || want_v) && !eligible) return KVQ_ERR_UNSUPPORTED;
  r->k = want_k;
  r->v = want_v;
  return KVQ_OK;
}

kvq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

int sm_count() { return kvq::device_sm_count(); }

}  // namespace

namespace kvq {
size_t qs_row_bytes_host(int qt, int d) { return qt == KVQ_TYPE_Q8_0 ? size_t(d) : size_t(d) / 2; }

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}
}  // namespace kvq

extern "C" {

int32_t kvq_version(void) { return KVQ_VERSION; }

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_TIMEOUT: return "on-device wait timed out";
    case KVQ_ERR_DEVICE_RANGE: return "device-side range check failed";
    default: return "unknown status";
  }
}

size_t kvq_plane_bytes(const kvq_cache* c, int32_t plane) {
  if (!shape_ok(c)) return 0;
  return plane_bytes(c, plane);
}

kvq_status kvq_cache_check(const kvq_cache* c) { return check_cache(c); }

kvq_status kvq_resolve_rotation(const kvq_cache* c, int32_t* rot_k, int32_t* rot_v) {
  if (!shape_ok(c) || !rot_k || !rot_v) return KVQ_ERR_INVALID_ARG;
  kvq::Rot r{};
  const kvq_status s = resolve(c, &r);
  if (s != KVQ_OK) return s;
  *rot_k = r.k;
  *rot_v = r.v;
  return KVQ_OK;
}

kvq_status kvq_rotate_quantize_append(const kvq_cache* c, const void* k, const void* v, int32_t in_dtype,
                                      int32_t n_new, const int32_t* n_new_per_seq, uint32_t append_flags,
                                      void* stream) {
  kvq_status s = check_cache(c);
  if (s != KVQ_OK) return s;
  kvq::Rot r{};
  if ((s = resolve(c, &r)) != KVQ_OK) return s;
  if (!valid_dtype(in_dtype) || n_new < 0 || (append_flags & ~KVQ_INPUT_PREROTATED)) return KVQ_ERR_INVALID_ARG;
  if (c->n_outlier && (append_flags & KVQ_INPUT_PREROTATED)) return KVQ_ERR_INVALID_ARG;  // outliers: original basis
  if (n_new == 0) return KVQ_OK;
  if (!k || !v || !aligned16(k) || !aligned16(v)) return KVQ_ERR_INVALID_ARG;
  if ((long long)c->batch * n_new * c->n_kv_heads * 2 > 0x7fffffffLL) return KVQ_ERR_INVALID_ARG;  // vectors < 2^31
  return from_cuda(kvq::launch_append(*c, r, k, v, in_dtype, n_new, n_new_per_seq, append_flags,
                                      static_cast<cudaStream_t>(stream)));
}

size_t kvq_decode_workspace_bytes(const kvq_cache* c, int32_t n_q_heads) {
  if (!shape_ok(c) || n_q_heads <= 0 || n_q_heads % c->n_kv_heads) return 0;
  return kvq::plan_decode(*c, n_q_heads, sm_count()).ws_bytes;
}

kvq_status kvq_decode_attention(const kvq_cache* c, const void* q, int32_t q_dtype, int32_t n_q_heads, float scale,
                                void* out, int32_t out_dtype, void* workspace, size_t ws_bytes, void* stream) {
  kvq_status s = check_cache(c);
  if (s != KVQ_OK) return s;
  kvq::Rot r{};
  if ((s = resolve(c, &r)) != KVQ_OK) return s;
  if (!valid_dtype(q_dtype) || !valid_dtype(out_dtype)) return KVQ_ERR_INVALID_ARG;
  if (n_q_heads <= 0 || n_q_heads % c->n_kv_heads || n_q_heads / c->n_kv_heads > 4096) return KVQ_ERR_INVALID_ARG;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  if (!(scale >= 0.0f) || scale > 1e30f) return KVQ_ERR_INVALID_ARG;
  if (!kvq::decode_supported(c->head_dim, c->k_type, c->v_type, c->n_outlier)) return KVQ_ERR_UNSUPPORTED;
  const kvq::DecodePlan plan = kvq::plan_decode(*c, n_q_heads, sm_count());
  if (!workspace || !aligned16(workspace) || ws_bytes < plan.ws_bytes) return KVQ_ERR_WORKSPACE;
  if (!kvq::decode_grid_ok(*c, plan)) return KVQ_ERR_UNSUPPORTED;
  const float sc = scale == 0.0f ? 1.0f / sqrtf(float(c->head_dim)) : scale;
  return from_cuda(kvq::launch_decode(*c, r, plan, q, q_dtype, n_q_heads, sc, out, out_dtype, workspace,
                                      static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_append_decode(const kvq_cache* c, const void* k, const void* v, int32_t in_dtype, int32_t n_new,
                             const int32_t* n_new_per_seq, uint32_t append_flags, const void* q, int32_t q_dtype,
                             int32_t n_q_heads, float scale, void* out, int32_t out_dtype, void* workspace,
                             size_t ws_bytes, void* stream) {
  kvq_status s = check_cache(c);
  if (s != KVQ_OK) return s;
  kvq::Rot r{};
  if ((s = resolve(c, &r)) != KVQ_OK) return s;
  // the append's arguments
  if (!valid_dtype(in_dtype) || n_new < 0 || (append_flags & ~KVQ_INPUT_PREROTATED)) return KVQ_ERR_INVALID_ARG;
  if (c->n_outlier && (append_flags & KVQ_INPUT_PREROTATED)) return KVQ_ERR_INVALID_ARG;
  if (n_new > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return KVQ_ERR_INVALID_ARG;
  if ((long long)c->batch * n_new * c->n_kv_heads * 2 > 0x7fffffffLL) return KVQ_ERR_INVALID_ARG;
  // the decode's arguments
  if (!valid_dtype(q_dtype) || !valid_dtype(out_dtype)) return KVQ_ERR_INVALID_ARG;
  if (n_q_heads <= 0 || n_q_heads % c->n_kv_heads || n_q_heads / c->n_kv_heads > 4096) return KVQ_ERR_INVALID_ARG;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  if (!(scale >= 0.0f) || scale > 1e30f) return KVQ_ERR_INVALID_ARG;
  if (!kvq::decode_supported(c->head_dim, c->k_type, c->v_type, c->n_outlier)) return KVQ_ERR_UNSUPPORTED;
  const kvq::DecodePlan plan = kvq::plan_decode(*c, n_q_heads, sm_count());
  if (!workspace || !aligned16(workspace) || ws_bytes < plan.ws_bytes) return KVQ_ERR_WORKSPACE;
  if (!kvq::decode_grid_ok(*c, plan)) return KVQ_ERR_UNSUPPORTED;
  const float sc = scale == 0.0f ? 1.0f / sqrtf(float(c->head_dim)) : scale;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (n_new > 0 && kvq::fused_step_ok(*c, plan, n_new)) {
    const kvq::FusedAppend fa{k, v, in_dtype, n_new, n_new_per_seq, (append_flags & KVQ_INPUT_PREROTATED) ? 1 : 0};
    return from_cuda(kvq::launch_decode(*c, r, plan, q, q_dtype, n_q_heads, sc, out, out_dtype, workspace, st, &fa));
  }
  // not fusable (or nothing to append): the two calls in sequence
  if (n_new > 0) {
    s = from_cuda(kvq::launch_append(*c, r, k, v, in_dtype, n_new, n_new_per_seq, append_flags, st));
    if (s != KVQ_OK) return s;
  }
  return from_cuda(kvq::launch_decode(*c, r, plan, q, q_dtype, n_q_heads, sc, out, out_dtype, workspace, st));
}

kvq_status kvq_decode_attention_noalloc(const kvq_cache* c, const void* q, int32_t q_dtype, int32_t n_q_heads,
                                        float scale, void* out, int32_t out_dtype, void* stream) {
  kvq_status s = check_cache(c);
  if (s != KVQ_OK) return s;
  kvq::Rot r{};
  if ((s = resolve(c, &r)) != KVQ_OK) return s;
  if (!valid_dtype(q_dtype) || !valid_dtype(out_dtype)) return KVQ_ERR_INVALID_ARG;
  if (n_q_heads <= 0 || n_q_heads % c->n_kv_heads || n_q_heads / c->n_kv_heads > 4096) return KVQ_ERR_INVALID_ARG;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  if (!(scale >= 0.0f) || scale > 1e30f) return KVQ_ERR_INVALID_ARG;
  if (!kvq::decode_supported(c->head_dim, c->k_type, c->v_type, c->n_outlier)) return KVQ_ERR_UNSUPPORTED;
  const kvq::DecodePlan plan = kvq::plan_decode(*c, n_q_heads, sm_count());
  if (plan.ws_bytes > KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;
  if (!kvq::decode_grid_ok(*c, plan)) return KVQ_ERR_UNSUPPORTED;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (kvq::decode_noalloc_scratch(&ws, &ws_bytes) != cudaSuccess || ws_bytes < plan.ws_bytes) return KVQ_ERR_CUDA;
  const float sc = scale == 0.0f ? 1.0f / sqrtf(float(c->head_dim)) : scale;
  return from_cuda(kvq::launch_decode(*c, r, plan, q, q_dtype, n_q_heads, sc, out, out_dtype, ws,
                                      static_cast<cudaStream_t>(stream)));
}

size_t kvq_prefill_workspace_bytes(const kvq_cache* c, int32_t n_q_heads, int32_t n_tokens) {
  if (!shape_ok(c) || n_tokens < 0 || n_q_heads <= 0 || n_q_heads % c->n_kv_heads) return 0;
  if (!kvq::prefill_supported(c->head_dim, n_q_heads / c->n_kv_heads)) return 0;
  return kvq::prefill_workspace_bytes(*c);
}

kvq_status kvq_prefill_attention(const kvq_cache* c, const void* q, int32_t q_dtype, int32_t n_q_heads,
                                 int32_t n_tokens, const int32_t* q_pos0, int32_t causal, int32_t chunk, float scale,
                                 void* out, int32_t out_dtype, void* workspace, size_t ws_bytes, void* stream) {
  kvq_status s = check_cache(c);
  if (s != KVQ_OK) return s;
  kvq::Rot r{};
  if ((s = resolve(c, &r)) != KVQ_OK) return s;
  if (!valid_dtype(q_dtype) || !valid_dtype(out_dtype)) return KVQ_ERR_INVALID_ARG;
  if (n_q_heads <= 0 || n_q_heads % c->n_kv_heads) return KVQ_ERR_INVALID_ARG;
  if (n_tokens < 0 || chunk < 0 || chunk % 64) return KVQ_ERR_INVALID_ARG;
  if (!(scale >= 0.0f) || scale > 1e30f) return KVQ_ERR_INVALID_ARG;
  if (n_tokens == 0) return KVQ_OK;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  if (!kvq::prefill_supported(c->head_dim, n_q_heads / c->n_kv_heads)) return KVQ_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) || ws_bytes < kvq::prefill_workspace_bytes(*c)) return KVQ_ERR_WORKSPACE;
  const float sc = scale == 0.0f ? 1.0f / sqrtf(float(c->head_dim)) : scale;
  return from_cuda(kvq::launch_prefill(*c, r, q, q_dtype, n_q_heads, n_tokens, q_pos0, causal, sc, out, out_dtype,
                                       workspace, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_dequant_debug(const kvq_cache* c, int32_t seq, int32_t kv_head, int32_t which, int32_t t0,
                             int32_t count, int32_t original_basis, float* out, void* blocks_ggml, void* stream) {
  kvq_status s = check_cache(c);
  if (s != KVQ_OK) return s;
  kvq::Rot r{};
  if ((s = resolve(c, &r)) != KVQ_OK) return s;
  if (seq < 0 || seq >= c->batch || kv_head < 0 || kv_head >= c->n_kv_heads) return KVQ_ERR_INVALID_ARG;
  if (which < 0 || which > 3 || t0 < 0 || count < 0) return KVQ_ERR_INVALID_ARG;
  if (which >= 2 && (c->tail_len == 0 || blocks_ggml)) return KVQ_ERR_INVALID_ARG;
  if (which < 2 && (long long)t0 + count > c->max_ctx) return KVQ_ERR_INVALID_ARG;
  if (count == 0) return KVQ_OK;
  if (!out && !blocks_ggml) return KVQ_ERR_INVALID_ARG;
  if (out && !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  return from_cuda(kvq::launch_debug(*c, r, seq, kv_head, which, t0, count, original_basis, out, blocks_ggml,
                                     static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_selftest_wait_timeout(const kvq_cache* c, int64_t limit_cycles, void* stream) {
  if (!c || !c->status || !aligned16(c->status)) return KVQ_ERR_INVALID_ARG;
  if (limit_cycles < 1 || limit_cycles > (int64_t(1) << 31)) return KVQ_ERR_INVALID_ARG;
  return from_cuda(kvq::launch_wait_timeout(c->status, limit_cycles, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_sync_status(const kvq_cache* c, void* stream, uint32_t* device_bits) {
  if (!c || !c->status) return KVQ_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return KVQ_ERR_CUDA;
  uint32_t bits = 0;
  if (cudaMemcpy(&bits, c->status, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ERR_CUDA;
  if (bits) {
    const uint32_t zero = 0;
    if (cudaMemcpy(c->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return KVQ_ERR_CUDA;
  }
  if (device_bits) *device_bits = bits;
  if (cudaGetLastError() != cudaSuccess) return KVQ_ERR_CUDA;
  if (bits & KVQ_DEV_ERR_TIMEOUT) return KVQ_ERR_TIMEOUT;
  if (bits) return KVQ_ERR_DEVICE_RANGE;
  return KVQ_OK;
}

}  // extern "C"
