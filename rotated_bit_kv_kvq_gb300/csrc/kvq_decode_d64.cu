// Decode kernels for head_dim 64, every K / V format pair (and head_dim 192, q4_0 / q4_0).
#include "kvq_decode_impl.cuh"

namespace kvq {

cudaError_t launch_decode_d64(const kvq_cache& c, Rot rot, const DecodePlan& plan, const void* q, int q_dtype,
                              int n_q_heads, float scale, void* out, int out_dtype, void* ws, cudaStream_t st,
                              const FusedAppend* fa) {
  return run_decode_d<64>(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype, ws, st, fa);
}

cudaError_t launch_decode_d192(const kvq_cache& c, Rot rot, const DecodePlan& plan, const void* q, int q_dtype,
                               int n_q_heads, float scale, void* out, int out_dtype, void* ws, cudaStream_t st,
                              const FusedAppend* fa) {
  if (c.k_type == KVQ_TYPE_Q4_0 && c.v_type == KVQ_TYPE_Q4_0)
    return run_decode<192, KVQ_TYPE_Q4_0, KVQ_TYPE_Q4_0, false>(c, rot, plan, q, q_dtype, n_q_heads, scale, out, out_dtype,
                                                         ws, st, fa);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
