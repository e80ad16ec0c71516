// Decode attention: split planning, dispatch by head_dim, and the fixed scratch
// of the allocation-free entry point.  The kernels are in kvq_decode_impl.cuh
// (compiled once per head_dim in kvq_decode_d*.cu).

#include <algorithm>

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
  // Looked up on every call with the caller's device current: a host-side lookup that
  // allocates nothing, and that follows the array if the device's context was reset and
  // the module reloaded at another address since an earlier call.
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess) return e;
  *ptr = p;
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
  return d == 64 || d == 128 || d == 192 || d == 256 || d == 320;  // every K / V format pair
}

DecodePlan plan_decode(const kvq_cache& c, int n_q_heads, int sm_count) {
  DecodePlan pl{};
  const int g = n_q_heads / c.n_kv_heads;
  pl.head_groups = (g + kMaxHeads - 1) / kMaxHeads;
  pl.heads_per_cta = (g + pl.head_groups - 1) / pl.head_groups;
  pl.planes = c.n_kv_heads * pl.head_groups;
  // one wave: as many pieces per plane as the SMs hold CTAs of this kernel
  const long long sms = sm_count > 0 ? sm_count : 148;
  const long long slots = (long long)ctas_per_sm(c.head_dim, c.n_outlier != 0) * sms;
  pl.pieces = int(std::max<long long>(1, slots / pl.planes));
  pl.pieces_fused = std::max(1, pl.pieces - c.batch);
  // a piece of the stream touches one more segment than it covers whole at each end:
  // slot = piece + segment index (or batch + piece + sequence with a fused step)
  pl.slots = std::max(pl.pieces, c.batch + pl.pieces_fused) + 2 * c.batch;
  // Costs in time, per token of one (sequence, KV head).  At head_dim 256 the 8-token tail
  // tiles make a tail token about 2.5 body tokens (the bytes ratio, 1024 : 416; a ratio of 2
  // measured 1.8% slower on the 64k workload).  Below it a tail token (16-token bf16 tiles)
  // costs 1.25 body tokens since body tiles hold 32 tokens (ragged 32-sequence batch at head_dim
  // 128: 16 : 16 took 108.5 us, 20 : 16 107.0 us, 24 : 16 109.0 us).
  pl.cost_body = 16;
  pl.cost_tail = c.head_dim >= 256 ? 40 : 20;
  pl.cost_min = 128 * pl.cost_body;          // 8 tiles: 2 per warp
  pl.cost_gap = 160 * pl.cost_body;          // ~4 us of a CTA's streaming time
  // Measured on the 64k-context workload: with equal pieces an SM's first, second and third
  // CTA ended after 94, 99 and 105 us; with pieces weighted 112 : 106 : 100 after 93, 95
  // and 98 us; with 118 : 109 : 100 after 92.6, 93.2 and 94.7 us.  The same weights serve
  // head_dim 128 with its 32-token body tiles (ragged 32-sequence batch 108.5 -> 107.0 us,
  // 4 x 64k at head_dim 128 155.8 -> 148.2 us against 118 : 102 : 83).
  pl.sms = int(sms);
  pl.slot_weight[0] = 118; pl.slot_weight[1] = 109; pl.slot_weight[2] = 98;
  const int cps = ctas_per_sm(c.head_dim, c.n_outlier != 0);
  auto one_wave = [&](long long ctas) { return cps == 3 && ctas > 2 * sms && ctas <= 3 * sms; };
  pl.weighted = one_wave((long long)pl.planes * pl.pieces);
  pl.weighted_fused = one_wave((long long)pl.planes * (c.batch + pl.pieces_fused));
  const size_t rows = (size_t)pl.planes * pl.slots * pl.heads_per_cta;
  pl.hdr_bytes = ((size_t)(1 + 2 * c.batch) * sizeof(long long) + 255) / 256 * 256;
  pl.ws_bytes = pl.hdr_bytes + rows * (c.head_dim + 2 + c.n_outlier) * sizeof(float);
  return pl;
}

bool fused_step_ok(const kvq_cache& c, const DecodePlan& plan, int n_new) {
  return c.tail_len > 0 && n_new >= 0 && n_new <= c.tail_len && c.tail_len <= kTailChunkMax &&
         plan.head_groups == 1;
}

bool decode_grid_ok(const kvq_cache& c, const DecodePlan& plan) {
  return (long long)c.batch + plan.pieces_fused <= 65535 && plan.pieces <= 65535 &&
         (long long)c.batch * c.n_kv_heads * plan.head_groups * kMaxHeads <= 0x7fffffffLL;
}

cudaError_t launch_decode(const kvq_cache& c, Rot rot, const DecodePlan& plan, const void* q, int q_dtype,
                          int n_q_heads, float scale, void* out, int out_dtype, void* ws, cudaStream_t st,
                          const FusedAppend* fa) {
  switch (c.head_dim) {
    case 64: return launch_decode_d64(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
    case 128: return launch_decode_d128(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
    case 256: return launch_decode_d256(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
    case 192: return launch_decode_d192(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
    case 320: return launch_decode_d320(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
