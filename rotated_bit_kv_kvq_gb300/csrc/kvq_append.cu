// Write path: rotate -> block-quantize -> pack -> store, plus the bf16 tail
// (velog "fix-kv-cache-quantization-outliers", section 아다마르 회전: K and V
// are multiplied by the normalized Hadamard matrix and stored rotated in the
// unchanged GGUF block formats; aitrends.kr "KVarN과 Precision Tail", section
// 용어 해설: the most recent tokens are also kept in BF16).
//
// One warp per (sequence, new token, KV head, K-or-V) vector.  The vector is
// loaded with P = G/32 consecutive channels per lane per G-wide Hadamard
// group, transformed in registers with shuffles, and each 32-channel block is
// quantized by the 32/P lanes that hold it.  Quantizer arithmetic follows the
// block definition operation by operation (IEEE division, no fused
// multiply-add), so the codes equal the CPU definition bit for bit.
//
// Also here: the inspection kernel behind kvq_dequant_debug.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kAppendWarps = 8;

template <int P>
__device__ __forceinline__ void load_vals(const void* base, int in_dtype, size_t elem, float* out) {
  if (in_dtype == KVQ_F32) {
    const float* p = static_cast<const float*>(base) + elem;
    if constexpr (P % 4 == 0) {
#pragma unroll
      for (int i = 0; i < P; i += 4) {
        float4 t = *reinterpret_cast<const float4*>(p + i);
        out[i] = t.x; out[i + 1] = t.y; out[i + 2] = t.z; out[i + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < P; ++i) out[i] = p[i];
    }
  } else {
    const uint16_t* p = static_cast<const uint16_t*>(base) + elem;
    uint16_t raw[P];
    if constexpr (P % 8 == 0) {
#pragma unroll
      for (int i = 0; i < P; i += 8) *reinterpret_cast<uint4*>(raw + i) = *reinterpret_cast<const uint4*>(p + i);
    } else {
#pragma unroll
      for (int i = 0; i < P; ++i) raw[i] = p[i];
    }
#pragma unroll
    for (int i = 0; i < P; ++i)
      out[i] = in_dtype == KVQ_BF16 ? bf16_bits_to_f32(raw[i]) : __half2float(__ushort_as_half(raw[i]));
  }
}

template <int P>
__device__ __forceinline__ void store_bytes(uint8_t* dst, const uint8_t* src) {
  if constexpr (P == 8) {
    uint2 t; uint8_t* tb = reinterpret_cast<uint8_t*>(&t);
#pragma unroll
    for (int i = 0; i < 8; ++i) tb[i] = src[i];
    *reinterpret_cast<uint2*>(dst) = t;
  } else if constexpr (P == 4) {
    uint32_t t = src[0] | (src[1] << 8) | (src[2] << 16) | (uint32_t(src[3]) << 24);
    *reinterpret_cast<uint32_t*>(dst) = t;
  } else if constexpr (P == 2) {
    *reinterpret_cast<uint16_t*>(dst) = uint16_t(src[0] | (src[1] << 8));
  } else {
    dst[0] = src[0];
  }
}

template <int P>
__device__ __forceinline__ void store_bf16(uint16_t* dst, const float* v) {
  uint16_t t[P];
#pragma unroll
  for (int i = 0; i < P; ++i) t[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v[i]));
  if constexpr (P == 8) {
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<uint4*>(t);
  } else if constexpr (P == 4) {
    *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<uint2*>(t);
  } else if constexpr (P == 2) {
    *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<uint32_t*>(t);
  } else {
    dst[0] = t[0];
  }
}

// Quantize and store one 32-value block whose values are spread over L = 32/P
// lanes (lane r of the block holds channels r*P .. r*P+P-1 in y[0..P-1]).
// d_ptr: the block's fp16 scale, or for q4_1 / q5_1 its 32-bit (d, lo) word.
template <int P>
__device__ __forceinline__ void quantize_block(const float* y, int qt, int r, uint8_t* qs_blk,
                                               uint32_t* qh_word, void* d_ptr) {
  constexpr int L = 32 / P;
  uint8_t code[P];
  if (type_has_min(qt)) {
    // scale + minimum: smallest / largest value (first channel on ties), d = (hi - lo) / top,
    // code = min(top, trunc((x - lo) * (1/d) + 0.5)), one rounding per operation
    float lo = y[0], hi = y[0];
    int lc = r * P, hc = r * P;
#pragma unroll
    for (int j = 1; j < P; ++j) {
      if (y[j] < lo) { lo = y[j]; lc = r * P + j; }
      if (y[j] > hi) { hi = y[j]; hc = r * P + j; }
    }
#pragma unroll
    for (int m = 1; m < L; m <<= 1) {
      const float ol = __shfl_xor_sync(0xffffffffu, lo, m), oh = __shfl_xor_sync(0xffffffffu, hi, m);
      const int olc = __shfl_xor_sync(0xffffffffu, lc, m), ohc = __shfl_xor_sync(0xffffffffu, hc, m);
      if (ol < lo || (ol == lo && olc < lc)) { lo = ol; lc = olc; }
      if (oh > hi || (oh == hi && ohc < hc)) { hi = oh; hc = ohc; }
    }
    const int top = qt == KVQ_TYPE_Q5_1 ? 31 : 15;
    const float d = __fdiv_rn(__fsub_rn(hi, lo), float(top));
    const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
#pragma unroll
    for (int j = 0; j < P; ++j)
      code[j] = uint8_t(min(top, __float2int_rz(__fadd_rn(__fmul_rn(__fsub_rn(y[j], lo), id), 0.5f))));
    if (r == 0)
      *static_cast<uint32_t*>(d_ptr) = uint32_t(__half_as_ushort(__float2half_rn(d))) |
                                       (uint32_t(__half_as_ushort(__float2half_rn(lo))) << 16);
  } else {
    // signed value of largest magnitude, first channel on ties (strict '>' scan from +0)
    float best_a = 0.0f, best_m = 0.0f;
    int best_c = 1 << 30;
#pragma unroll
    for (int j = 0; j < P; ++j) {
      const float a = fabsf(y[j]);
      if (a > best_a) { best_a = a; best_m = y[j]; best_c = r * P + j; }
    }
#pragma unroll
    for (int m = 1; m < L; m <<= 1) {
      const float oa = __shfl_xor_sync(0xffffffffu, best_a, m);
      const float om = __shfl_xor_sync(0xffffffffu, best_m, m);
      const int oc = __shfl_xor_sync(0xffffffffu, best_c, m);
      if (oa > best_a || (oa == best_a && oc < best_c)) { best_a = oa; best_m = om; best_c = oc; }
    }
    float d;
    if (qt == KVQ_TYPE_Q8_0) {
      d = best_a / 127.0f;
      const float id = d != 0.0f ? 1.0f / d : 0.0f;
#pragma unroll
      for (int j = 0; j < P; ++j) code[j] = uint8_t(int8_t(int(roundf(__fmul_rn(y[j], id)))));
    } else {
      const bool q5 = qt == KVQ_TYPE_Q5_0;
      d = q5 ? best_m / -16.0f : best_m / -8.0f;
      const float id = d != 0.0f ? 1.0f / d : 0.0f;
      const float off = q5 ? 16.5f : 8.5f;
      const int top = q5 ? 31 : 15;
#pragma unroll
      for (int j = 0; j < P; ++j) code[j] = uint8_t(min(top, __float2int_rz(__fadd_rn(__fmul_rn(y[j], id), off))));
    }
    if (r == 0) *static_cast<__half*>(d_ptr) = __float2half_rn(d);
  }
  if (qt == KVQ_TYPE_Q8_0) {
    store_bytes<P>(qs_blk + r * P, code);
    return;
  }
  // nibble packing: byte k = code_k | code_{k+16} << 4
  uint8_t packed[P];
#pragma unroll
  for (int j = 0; j < P; ++j) {
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, uint32_t(code[j]), L / 2);
    packed[j] = uint8_t((code[j] & 0x0F) | ((hi & 0x0F) << 4));
  }
  if (r < L / 2) store_bytes<P>(qs_blk + r * P, packed);
  if (type_has_qh(qt)) {
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < P; ++j) w |= uint32_t((code[j] >> 4) & 1) << (r * P + j);
#pragma unroll
    for (int m = 1; m < L; m <<= 1) w |= __shfl_xor_sync(0xffffffffu, w, m);
    if (r == 0) *qh_word = w;
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kAppendWarps * 32)
append_kernel(kvq_cache c, int rot_k, int rot_v, const void* __restrict__ kin, const void* __restrict__ vin,
              int in_dtype, int n_new, const int32_t* __restrict__ n_new_per_seq, int prerotated) {
  constexpr int P = G / 32;
  constexpr int E = D / 32;
  constexpr int NB = D / kQK;
  const int lane = threadIdx.x & 31;
  const int warp = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  const int H = c.n_kv_heads;
  const long long tasks = (long long)c.batch * n_new * H * 2;

  if (warp < tasks) {
    // 32-bit index arithmetic (the host keeps the vector count below 2^31)
    const unsigned wu = unsigned(warp);
    const int which = int(wu & 1u);                   // 0 = K, 1 = V
    const unsigned vec = wu >> 1;                     // (b * n_new + i) * H + h
    const int h = int(vec % unsigned(H));
    const unsigned bi = vec / unsigned(H);
    const int i = int(bi % unsigned(n_new));
    const int b = int(bi / unsigned(n_new));
    const int n0 = c.seq_len[b];
    const int nb = n_new_per_seq ? n_new_per_seq[b] : n_new;
    const bool ok = nb >= 0 && nb <= n_new && n0 >= 0 && (long long)n0 + nb <= c.max_ctx;
    if (!ok) {
      if (i == 0 && h == 0 && which == 0 && lane == 0) atomicOr(&c.status[0], KVQ_DEV_ERR_APPEND_RANGE);
    } else if (i < nb) {
      const int pos = n0 + i;
      const void* src = which ? vin : kin;
      float v[E];
#pragma unroll
      for (int gi = 0; gi < D / G; ++gi)
        load_vals<P>(src, in_dtype, size_t(vec) * D + gi * G + lane * P, v + gi * P);
      const bool rot = (which ? rot_v : rot_k) && !prerotated;
      if (rot) {
        warp_fwht<D, G>(v, lane);
        const float s = inv_sqrt_group<G>();
#pragma unroll
        for (int j = 0; j < E; ++j) v[j] *= s;
      }
      const int qt = which ? c.v_type : c.k_type;
      const size_t row = ((size_t)b * H + h) * c.max_ctx + pos;
      uint8_t* qs = static_cast<uint8_t*>(which ? c.v_qs : c.k_qs) + row * qs_row_bytes(qt, D);
      uint32_t* qh = static_cast<uint32_t*>(which ? c.v_qh : c.k_qh);
      uint8_t* dp = static_cast<uint8_t*>(which ? c.v_d : c.k_d) + row * NB * (type_has_min(qt) ? 4 : 2);
      const int L = 32 / P;
      const int r = lane % L;
#pragma unroll
      for (int gi = 0; gi < D / G; ++gi) {
        const int blk = gi * P + lane / L;
        const int blk_bytes = qt == KVQ_TYPE_Q8_0 ? 32 : 16;
        quantize_block<P>(v + gi * P, qt, r, qs + blk * blk_bytes, qh ? qh + row * NB + blk : nullptr,
                          dp + blk * (type_has_min(qt) ? 4 : 2));
      }
      if (c.tail_len > 0 && i >= nb - c.tail_len) {
        uint16_t* tail = static_cast<uint16_t*>(which ? c.v_tail : c.k_tail) +
                         (((size_t)b * H + h) * c.tail_len + pos % c.tail_len) * D;
#pragma unroll
        for (int gi = 0; gi < D / G; ++gi) store_bf16<P>(tail + gi * G + lane * P, v + gi * P);
      }
    }
  }

  // The last CTA to finish advances seq_len: every CTA has read seq_len
  // before it counts itself in.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned done = atomicAdd(&c.status[1], 1u);
    if (done == gridDim.x - 1) {
      __threadfence();
      for (int b = 0; b < c.batch; ++b) {
        const int n0 = c.seq_len[b];
        const int nb = n_new_per_seq ? n_new_per_seq[b] : n_new;
        if (nb >= 0 && nb <= n_new && n0 >= 0 && (long long)n0 + nb <= c.max_ctx) c.seq_len[b] = n0 + nb;
      }
      c.status[1] = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// kvq_dequant_debug: one warp per position.
// ---------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(128)
debug_kernel(kvq_cache c, int rot_side, int seq, int kv_head, int which, int t0, int count,
             int original_basis, float* __restrict__ out, uint8_t* __restrict__ blocks) {
  constexpr int E = D / 32;
  constexpr int NB = D / kQK;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (t >= count) return;
  const int pos = t0 + t;
  const int H = c.n_kv_heads;
  const bool tail = which >= 2;
  const bool is_v = (which & 1) != 0;
  float v[E];
  if (tail) {
    const uint16_t* tp = static_cast<const uint16_t*>(is_v ? c.v_tail : c.k_tail) +
                         (((size_t)seq * H + kv_head) * c.tail_len + pos % c.tail_len) * D;
#pragma unroll
    for (int j = 0; j < E; ++j) v[j] = bf16_bits_to_f32(tp[fwht_channel<D, G>(lane, j)]);
  } else {
    const int qt = is_v ? c.v_type : c.k_type;
    const size_t row = ((size_t)seq * H + kv_head) * c.max_ctx + pos;
    const uint8_t* qs = static_cast<const uint8_t*>(is_v ? c.v_qs : c.k_qs) + row * qs_row_bytes(qt, D);
    const uint32_t* qh = static_cast<const uint32_t*>(is_v ? c.v_qh : c.k_qh);
    // block header: fp16 d, or for q4_1 / q5_1 the (d, lo) pair, as bytes
    const int hb = type_has_min(qt) ? 4 : 2;
    const uint8_t* dp = static_cast<const uint8_t*>(is_v ? c.v_d : c.k_d) + row * NB * hb;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const int ch = fwht_channel<D, G>(lane, j);
      const int blk = ch / kQK, k = ch % kQK;
      const float dv = __half2float(reinterpret_cast<const __half*>(dp + blk * hb)[0]);
      const float mv = type_has_min(qt) ? __half2float(reinterpret_cast<const __half*>(dp + blk * hb)[1]) : 0.0f;
      int code;
      if (qt == KVQ_TYPE_Q8_0) {
        code = int(int8_t(qs[blk * 32 + k]));
      } else {
        const uint8_t byte = qs[blk * 16 + (k & 15)];
        code = k < 16 ? (byte & 15) : (byte >> 4);
        if (type_has_qh(qt)) code |= int((qh[row * NB + blk] >> k) & 1u) << 4;
        code -= type_code_offset(qt);
      }
      v[j] = float(code) * dv + mv;
    }
    if (blocks) {
      // GGUF array-of-structs: [d:2][lo:2 (_1)][qh:4 (q5_x)][qs:16|32] per block
      const int bb = type_block_bytes(qt);
      uint8_t* ob = blocks + (size_t)t * NB * bb;
      const int qsb = qt == KVQ_TYPE_Q8_0 ? 32 : 16;
      const int qhb = type_has_qh(qt) ? 4 : 0;
      for (int idx = lane; idx < NB * bb; idx += 32) {
        const int blk = idx / bb, o = idx % bb;
        uint8_t val;
        if (o < hb) {
          val = dp[blk * hb + o];
        } else if (o < hb + qhb) {
          val = uint8_t(qh[row * NB + blk] >> (8 * (o - hb)));
        } else {
          val = qs[blk * qsb + (o - hb - qhb)];
        }
        ob[idx] = val;
      }
    }
  }
  if (original_basis && rot_side) {
    warp_fwht<D, G>(v, lane);
    const float s = inv_sqrt_group<G>();
#pragma unroll
    for (int j = 0; j < E; ++j) v[j] *= s;
  }
  if (out) {
#pragma unroll
    for (int j = 0; j < E; ++j) out[(size_t)t * D + fwht_channel<D, G>(lane, j)] = v[j];
  }
}

template <int D>
cudaError_t append_d(const kvq_cache& c, Rot rot, const void* k, const void* v, int in_dtype, int n_new,
                     const int32_t* nps, uint32_t flags, cudaStream_t st) {
  const long long warps = (long long)c.batch * n_new * c.n_kv_heads * 2;
  const long long blocks = (warps + kAppendWarps - 1) / kAppendWarps;
  if (warps > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int pre = (flags & KVQ_INPUT_PREROTATED) ? 1 : 0;
  constexpr int G = (D >= 64 && D % 64 == 0) ? (((D & (D - 1)) == 0) ? D : 64) : 32;
  append_kernel<D, G><<<unsigned(blocks), kAppendWarps * 32, 0, st>>>(c, rot.k, rot.v, k, v, in_dtype, n_new, nps, pre);
  return cudaGetLastError();
}

template <int D>
cudaError_t debug_d(const kvq_cache& c, Rot rot, int seq, int kv_head, int which, int t0, int count,
                    int original_basis, float* out, void* blocks, cudaStream_t st) {
  constexpr int G = (D >= 64 && D % 64 == 0) ? (((D & (D - 1)) == 0) ? D : 64) : 32;
  const int rot_side = (which & 1) ? rot.v : rot.k;
  debug_kernel<D, G><<<(count + 3) / 4, 128, 0, st>>>(c, rot_side, seq, kv_head, which, t0, count, original_basis,
                                                      out, static_cast<uint8_t*>(blocks));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const kvq_cache& c, Rot rot, const void* k, const void* v, int in_dtype, int n_new,
                          const int32_t* nps, uint32_t flags, cudaStream_t st) {
  switch (c.head_dim) {
    case 32: return append_d<32>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 64: return append_d<64>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 96: return append_d<96>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 128: return append_d<128>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 160: return append_d<160>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 192: return append_d<192>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 224: return append_d<224>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 256: return append_d<256>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_debug(const kvq_cache& c, Rot rot, int seq, int kv_head, int which, int t0, int count,
                         int original_basis, float* out, void* blocks, cudaStream_t st) {
  switch (c.head_dim) {
    case 32: return debug_d<32>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 64: return debug_d<64>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 96: return debug_d<96>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 128: return debug_d<128>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 160: return debug_d<160>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 192: return debug_d<192>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 224: return debug_d<224>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 256: return debug_d<256>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
