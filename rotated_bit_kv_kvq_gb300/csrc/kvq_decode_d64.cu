// Decode kernels for head_dim 64, every K / V format pair.
#include "kvq_decode_impl.cuh"

namespace kvq {

cudaError_t launch_decode_d64(const kvq_cache& c, Rot rot, const DecodePlan& plan, const void* q, int q_dtype,
                              int n_q_heads, float scale, void* out, int out_dtype, void* ws, cudaStream_t st,
                              const FusedAppend* fa) {
  return run_decode_d<64>(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
}

}  // namespace kvq
