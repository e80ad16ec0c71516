// Host-side declarations shared by the kvq translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>
#include <unordered_map>

#include "kvq.h"

namespace kvq {

struct Rot {
  int k;  // K (and query) rotation on
  int v;  // V rotation on (output rotated back)
};

// Hadamard group width used for a head: head_dim when it is a power of two,
// 64 for other multiples of 64, 32 when rotation is impossible (layout only).
inline int rotation_group(int d) {
  if (d >= 64 && d % 64 == 0) return (d & (d - 1)) == 0 ? d : 64;
  return 32;
}

size_t qs_row_bytes_host(int qt, int d);

// Raises a kernel's dynamic shared-memory limit once per device (again only for
// a larger size), so that steady-state calls make no attribute call and can be
// captured into a CUDA graph.
inline cudaError_t ensure_dynamic_smem(const void* kernel, int bytes) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static std::unordered_map<const void*, int[kMaxDevices]> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  std::lock_guard<std::mutex> lock(mu);
  int& have = done[kernel][dev];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

// Launchers (arguments already validated by the API layer).
// SMs of the current device (0 when the query fails).
int device_sm_count();

cudaError_t launch_append(const kvq_cache& c, Rot rot, const void* k, const void* v, int in_dtype,
                          int n_new, const int32_t* n_new_per_seq, uint32_t flags, cudaStream_t st);
cudaError_t launch_debug(const kvq_cache& c, Rot rot, int seq, int kv_head, int which, int t0,
                         int count, int original_basis, float* out, void* blocks, cudaStream_t st);

// One CTA waiting (bounded) on a barrier that never completes: the failure path.
cudaError_t launch_wait_timeout(uint32_t* status, long long limit_cycles, cudaStream_t st);

// Decode: split plan shared by the workspace query and the launch.  The work is cut
// on the device, from seq_len, by cost: per plane (KV head x head group) every
// sequence's tail and body form one stream of bytes to read, cut into `pieces`
// equal pieces, one CTA each (with a fused step every tail gets a CTA of its own,
// which also writes the new tokens, and the bodies form the stream).
struct DecodePlan {
  int heads_per_cta;   // query heads handled by one CTA (<= 8)
  int head_groups;     // CTAs along the head axis per KV head
  int planes;          // n_kv_heads * head_groups
  int pieces;          // stream pieces per plane (one wave of CTAs)
  int pieces_fused;    // stream pieces per plane beside the batch's tail CTAs (fused step)
  int slots;           // partial slots per plane (pieces plus the cuts at segment ends)
  long long cost_body; // bytes of one body token of one (sequence, KV head)
  long long cost_tail; // bytes of one tail token
  long long cost_min;  // smallest piece
  long long cost_gap;  // virtual bytes before each segment: a CTA's cost of switching segments
  int sms;             // SMs the plan fills
  // With one full wave of three CTAs per SM the pieces are weighted by dispatch slot
  // (an SM's first, second, third CTA), so that the SM's CTAs end together.
  int slot_weight[3];
  bool weighted, weighted_fused;
  size_t hdr_bytes;    // fused-step partition header at the start of the workspace
  size_t ws_bytes;     // header, then acc [planes][slots][heads_per_cta][D], (m, l) [..][2],
                       // with outlier channels their acc [..][32]
};
// n_outlier > 0: the q4_0 / q5_0 / q8_0 pairs at head_dim 64, 128 and 256.
bool decode_supported(int d, int kt, int vt, int n_outlier);
DecodePlan plan_decode(const kvq_cache& c, int n_q_heads, int sm_count);
// Address of the fixed decode scratch array on the current device (looked up
// once per device); size in *bytes.
cudaError_t decode_noalloc_scratch(void** ptr, size_t* bytes);
// New tokens appended by the decode launch itself (the fused step): the one
// tail CTA of each (sequence, KV head) writes them before its tail attention,
// and the merge kernel advances seq_len.  Requires n_new <= tail_len, one head
// group and one tail split (fused_step_ok).
struct FusedAppend {
  const void* k;
  const void* v;
  int in_dtype;
  int n_new;
  const int32_t* n_new_per_seq;  // device, may be NULL
  int prerotated;
};
bool fused_step_ok(const kvq_cache& c, const DecodePlan& plan, int n_new);
// grid dimensions within the launch limits
bool decode_grid_ok(const kvq_cache& c, const DecodePlan& plan);
cudaError_t launch_decode(const kvq_cache& c, Rot rot, const DecodePlan& plan, const void* q,
                          int q_dtype, int n_q_heads, float scale, void* out, int out_dtype,
                          void* ws, cudaStream_t st, const FusedAppend* fa = nullptr);
// per-head_dim launchers (one translation unit each)
#define KVQ_DECODE_LAUNCHER(NAME)                                                                     \
  cudaError_t NAME(const kvq_cache& c, Rot rot, const DecodePlan& plan, const void* q, int q_dtype,  \
                   int n_q_heads, float scale, void* out, int out_dtype, void* ws, cudaStream_t st,  \
                   const FusedAppend* fa);
KVQ_DECODE_LAUNCHER(launch_decode_d64)
KVQ_DECODE_LAUNCHER(launch_decode_d128)
KVQ_DECODE_LAUNCHER(launch_decode_d192)
KVQ_DECODE_LAUNCHER(launch_decode_d256)
KVQ_DECODE_LAUNCHER(launch_decode_d320)
#undef KVQ_DECODE_LAUNCHER

// Prefill (tcgen05): head_dim 64 or 128, GQA group up to 128.  The workspace
// holds every 64-key tile of every (sequence, KV head) up to max_ctx, staged
// once as fp16 hi / lo operand tiles (512 * head_dim bytes per tile).
bool prefill_supported(int d, int group);
size_t prefill_workspace_bytes(const kvq_cache& c);
cudaError_t launch_prefill(const kvq_cache& c, Rot rot, const void* q, int q_dtype, int n_q_heads, int n_tokens,
                           const int32_t* q_pos0, int causal, float scale, void* out, int out_dtype,
                           void* ws, cudaStream_t st);

}  // namespace kvq
