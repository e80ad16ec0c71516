// Decode attention: split planning, dispatch by head_dim, and the fixed scratch
// of the allocation-free entry point.  The kernels are in kvq_decode_impl.cuh
// (compiled once per head_dim in kvq_decode_d*.cu).

#include <mutex>

#include "kvq_decode_impl.cuh"

namespace kvq {
namespace {

// Scratch of kvq_decode_attention_noalloc: a fixed device array, so that
// callers who cannot allocate still get split partials somewhere.  Every GPU
// that loads the library holds it until exit.  Host code only sees a host-side
// stand-in for the name; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

}  // namespace

cudaError_t decode_noalloc_scratch(void** ptr, size_t* bytes) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {  // once per device, with that device current
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  *bytes = sizeof(g_decode_scratch);
  return cudaSuccess;
}

namespace {
// A fresh barrier expecting one arrival that never comes: the wait gives up
// after limit_cycles and reports it, as every kernel's bounded waits do.
__global__ void wait_timeout_kernel(uint32_t* status, long long limit_cycles) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, limit_cycles)) atomicOr(status, KVQ_DEV_ERR_TIMEOUT);
}
}  // namespace

cudaError_t launch_wait_timeout(uint32_t* status, long long limit_cycles, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status, limit_cycles);
  return cudaGetLastError();
}

bool decode_supported(int d, int kt, int vt, int n_outlier) {
  if (n_outlier)
    return (d == 64 || d == 128 || d == 256) && kt <= KVQ_TYPE_Q8_0 && vt <= KVQ_TYPE_Q8_0 && n_outlier == 32;
  if (d == 64 || d == 128 || d == 256) return true;  // every K / V format pair
  return d == 192 && kt == KVQ_TYPE_Q4_0 && vt == KVQ_TYPE_Q4_0;
}

DecodePlan plan_decode(const kvq_cache& c, int n_q_heads, int sm_count) {
  DecodePlan pl{};
  const int g = n_q_heads / c.n_kv_heads;
  pl.head_groups = (g + kMaxHeads - 1) / kMaxHeads;
  pl.heads_per_cta = (g + pl.head_groups - 1) / pl.head_groups;
  const long long pairs = (long long)c.batch * c.n_kv_heads * pl.head_groups;
  // tail: one CTA per (sequence, head group) for tails up to 4096 slots
  pl.tail_chunk = c.tail_len > 0 ? (c.tail_len < kTailChunkMax ? (c.tail_len + 63) / 64 * 64 : kTailChunkMax) : 64;
  pl.splits_tail = c.tail_len > 0 ? (c.tail_len + pl.tail_chunk - 1) / pl.tail_chunk : 0;
  // body: size the chunks so that all CTAs of a full cache fit in one wave of
  // kCtasPerSm CTAs per SM (shorter sequences leave their last splits empty)
  const long long slots = (long long)ctas_per_sm(c.head_dim, c.n_outlier != 0) * (sm_count > 0 ? sm_count : 148);
  long long per_pair = slots / pairs - pl.splits_tail;
  if (per_pair < 1) per_pair = 1;
  int chunk = int(((c.max_ctx + per_pair - 1) / per_pair + 63) / 64 * 64);
  if (chunk < 512) chunk = 512;
  pl.chunk = chunk;
  pl.splits_body = (c.max_ctx + chunk - 1) / chunk;
  pl.splits = pl.splits_body + pl.splits_tail;
  pl.cls_len[0] = chunk; pl.cls_len[1] = chunk; pl.cls_len[2] = chunk;
  pl.cls_cnt[0] = pl.splits_body; pl.cls_cnt[1] = 0; pl.cls_cnt[2] = 0;
  // One wave of three CTAs per SM: the CTAs are dispatched split by split (the kernel reads
  // its linear block index split-major), so the first sm_count take the first slot of every
  // SM, the next sm_count the second, the rest the third.  An SM's warp scheduler favours its
  // oldest warps: measured on the 64k workload, equal chunks end after 96, 105 and 113 us by
  // slot.  Chunks sized 1/96 : 1/105 : 1/113 by slot let the three end together.
  const int cps = ctas_per_sm(c.head_dim, c.n_outlier != 0);
  const long long sms = sm_count > 0 ? sm_count : 148;
  const long long ctas = (long long)pl.splits * pairs;
  if (cps == 3 && ctas <= 3 * sms && ctas > 2 * sms && pl.splits_body >= 3) {
    const double w[3] = {105.0 / 96.0, 1.0, 105.0 / 113.0};
    int cnt[3] = {0, 0, 0};
    for (int s = 0; s < pl.splits_body; ++s) {
      const long long mid = (long long)(s + pl.splits_tail) * pairs + pairs / 2;
      ++cnt[mid / sms >= 2 ? 2 : int(mid / sms)];
    }
    double tot = 0.0;
    for (int k = 0; k < 3; ++k) tot += cnt[k] * w[k];
    for (int k = 0; k < 3; ++k) {
      pl.cls_cnt[k] = cnt[k];
      pl.cls_len[k] = int(((long long)(c.max_ctx * w[k] / tot) + 64) / 64 * 64);
    }
  }
  pl.ws_bytes = (size_t)c.batch * n_q_heads * pl.splits * (c.head_dim + 2 + c.n_outlier) * sizeof(float);
  return pl;
}

bool fused_step_ok(const kvq_cache& c, const DecodePlan& plan, int n_new) {
  return c.tail_len > 0 && n_new >= 0 && n_new <= c.tail_len && plan.head_groups == 1 && plan.splits_tail == 1;
}

cudaError_t launch_decode(const kvq_cache& c, Rot rot, const DecodePlan& plan, const void* q, int q_dtype,
                          int n_q_heads, float scale, void* out, int out_dtype, void* ws, cudaStream_t st,
                          const FusedAppend* fa) {
  switch (c.head_dim) {
    case 64: return launch_decode_d64(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
    case 128: return launch_decode_d128(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
    case 256: return launch_decode_d256(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
    case 192: return launch_decode_d192(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
