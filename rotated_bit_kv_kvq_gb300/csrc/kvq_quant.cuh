// Write-path device helpers shared by the append kernel and the fused
// append + decode step: loading a head vector's values, the block quantizers
// (GGUF q4_0 / q5_0 / q8_0 and q4_1 / q5_1, operation by operation as the block
// definitions state) and the packed / bf16 stores.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvq_device.cuh"

namespace kvq {
namespace {

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
  static_assert(P == 1 || P == 2 || P == 4 || P % 8 == 0, "lane width");
  if constexpr (P > 8) {  // 16-byte pieces (P = 16 at head_dim 512)
#pragma unroll
    for (int i = 0; i < P; i += 16) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        w[k] = src[i + 4 * k] | (src[i + 4 * k + 1] << 8) | (src[i + 4 * k + 2] << 16) |
               (uint32_t(src[i + 4 * k + 3]) << 24);
      *reinterpret_cast<uint4*>(dst + i) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else if constexpr (P == 8) {
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
  static_assert(P == 1 || P == 2 || P == 4 || P % 8 == 0, "lane width");
  if constexpr (P % 8 == 0) {
#pragma unroll
    for (int i = 0; i < P; i += 8) *reinterpret_cast<uint4*>(dst + i) = *reinterpret_cast<uint4*>(t + i);
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
// q8_0 codes go out as stored in the body planes, offset binary (code + 128,
// i.e. the GGUF byte XOR 0x80), unless `q8_signed` (the outlier plane keeps the
// GGUF bytes).
template <int P>
__device__ __forceinline__ void quantize_block(const float* y, int qt, int r, uint8_t* qs_blk, const QhDst& qh,
                                               void* d_ptr, bool q8_signed = false) {
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
      for (int j = 0; j < P; ++j)
        code[j] = uint8_t(int8_t(int(roundf(__fmul_rn(y[j], id))))) ^ (q8_signed ? 0u : 0x80u);
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
    if (r == 0) qh_put(qh, w);
  }
}

// Outlier channel of slot `lane` of KV head h (n_outlier = 32): the caller's
// list must be strictly increasing inside [0, D).  Returns the channel, or -1
// for an invalid slot (and sets KVQ_DEV_ERR_OUTLIER once per warp).
template <int D>
__device__ __forceinline__ int outlier_channel(const kvq_cache& c, int h, int lane) {
  const int ch = c.outlier_idx[(size_t)h * 32 + lane];
  const int prev = __shfl_up_sync(0xffffffffu, ch, 1);
  const bool ok = ch >= 0 && ch < D && (lane == 0 || prev < ch);
  const unsigned bad = __ballot_sync(0xffffffffu, !ok);
  if (bad && lane == 0) atomicOr(&c.status[0], KVQ_DEV_ERR_OUTLIER);
  return ok ? ch : -1;
}

// One warp: rotate (when `rot`), quantize and store one K (which = 0) or V
// (which = 1) vector of (sequence b, KV head h) at position pos, reading its
// head_dim values from src[elem0 ..]; also its bf16 tail row (slot pos % T)
// when `to_tail`.  Lane l holds channels l*P .. l*P+P-1 of every G-wide group.
// With outlier channels (c.n_outlier = 32) the body gets the vector with those
// channels zeroed (then rotated and quantized), slot l's value goes to a q8_0
// block of the outlier plane, unrotated, and the tail keeps the whole vector.
// OLW: whether that code is compiled in (callers without outlier channels leave
// it out).
template <int D, int G, bool OLW>
__device__ __forceinline__ void store_vector(const kvq_cache& c, int which, int b, int h, int pos, bool to_tail,
                                             const void* src, size_t elem0, int in_dtype, bool rot, int lane) {
  constexpr int P = G / 32;
  constexpr int E = D / 32;
  constexpr int NB = D / kQK;
  float v[E];
#pragma unroll
  for (int gi = 0; gi < D / G; ++gi) load_vals<P>(src, in_dtype, elem0 + gi * G + lane * P, v + gi * P);
  const bool outl = OLW && c.n_outlier != 0;
  float ov = 0.0f;      // outlier slot `lane`: its value (original basis)
  float vt[E];          // whole vector for the tail when the body's differs
  if (outl) {
    const int ch = outlier_channel<D>(c, h, lane);
    // slot value: channel ch lives in lane (ch % G) / P, register (ch / G) * P + ch % P
    const int src_lane = ch < 0 ? 0 : (ch % G) / P, src_reg = ch < 0 ? -1 : (ch / G) * P + ch % P;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float t = __shfl_sync(0xffffffffu, v[e], src_lane);
      if (e == src_reg) ov = t;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) vt[e] = v[e];
    // zero this lane's channels that are outlier slots (a register bit mask, so
    // that v is never indexed by a run-time value)
    uint32_t zmask = 0;
#pragma unroll 4
    for (int sl = 0; sl < 32; ++sl) {
      const int cs = __shfl_sync(0xffffffffu, ch, sl);
      if (cs >= 0 && (cs % G) / P == lane) zmask |= 1u << ((cs / G) * P + cs % P);
    }
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = ((zmask >> e) & 1u) ? 0.0f : v[e];
  }
  if (rot) {
    const float s = inv_sqrt_group<G>();
    warp_fwht<D, G>(v, lane);
#pragma unroll
    for (int j = 0; j < E; ++j) v[j] *= s;
    if (outl && to_tail) {
      warp_fwht<D, G>(vt, lane);
#pragma unroll
      for (int j = 0; j < E; ++j) vt[j] *= s;
    }
  }
  const int qt = which ? c.v_type : c.k_type;
  const long long brow = body_row(row_map(c), b, h, pos);
  if (brow < 0) {  // page id outside the pool: the body row is not written
    if (lane == 0) atomicOr(&c.status[0], KVQ_DEV_ERR_PAGE);
  } else {
    const size_t row = size_t(brow);
    uint8_t* qs = static_cast<uint8_t*>(which ? c.v_qs : c.k_qs) + row * qs_row_bytes(qt, D);
    void* qh = which ? c.v_qh : c.k_qh;
    uint8_t* dp = static_cast<uint8_t*>(which ? c.v_d : c.k_d) + row * NB * (type_has_min(qt) ? 4 : 2);
    constexpr int L = 32 / P;
    const int r = lane % L;
#pragma unroll
    for (int gi = 0; gi < D / G; ++gi) {
      const int blk = gi * P + lane / L;
      const int blk_bytes = qt == KVQ_TYPE_Q8_0 ? 32 : 16;
      quantize_block<P>(v + gi * P, qt, r, qs + blk * blk_bytes, qh_dst(qh, which == 0, row, NB, blk),
                        dp + blk * (type_has_min(qt) ? 4 : 2));
    }
    if (outl) {  // one q8_0 block, slot = lane
      uint8_t* grp = static_cast<uint8_t*>(c.outl) + (row / 16) * kOutlTile;
      uint8_t* oqs = grp + which * 512 + (row % 16) * 32;
      uint16_t* od = reinterpret_cast<uint16_t*>(grp + 1024 + which * 32) + row % 16;
      quantize_block<1>(&ov, KVQ_TYPE_Q8_0, lane, oqs, QhDst{nullptr, nullptr, false}, od, true);
    }
  }
  if (to_tail) {
    uint16_t* tail = static_cast<uint16_t*>(which ? c.v_tail : c.k_tail) +
                     (((size_t)b * c.n_kv_heads + h) * c.tail_len + pos % c.tail_len) * D;
#pragma unroll
    for (int gi = 0; gi < D / G; ++gi) {  // (two calls: a selected array pointer would force v into local memory)
      if (outl) store_bf16<P>(tail + gi * G + lane * P, vt + gi * P);
      else store_bf16<P>(tail + gi * G + lane * P, v + gi * P);
    }
  }
}

}  // namespace
}  // namespace kvq
