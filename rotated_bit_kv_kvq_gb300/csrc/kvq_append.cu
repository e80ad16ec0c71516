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

#include <algorithm>
#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_quant.cuh"

namespace kvq {
namespace {

constexpr int kAppendWarps = 8;
constexpr long long kRowsMinVectors = 2048;  // appends of at least this many vectors use append_rows_kernel

// The last CTA of an append advances seq_len: every CTA has read seq_len before
// it counts itself in.  Called by all threads of every CTA at its end.
__device__ __forceinline__ void finish_append(const kvq_cache& c, int n_new, const int32_t* n_new_per_seq) {
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

template <int D, int G>
__global__ void __launch_bounds__(kAppendWarps * 32)
append_kernel(kvq_cache c, int rot_k, int rot_v, const void* __restrict__ kin, const void* __restrict__ vin,
              int in_dtype, int n_new, const int32_t* __restrict__ n_new_per_seq, int prerotated) {
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
      const bool rot = (which ? rot_v : rot_k) && !prerotated;
      const bool to_tail = c.tail_len > 0 && i >= nb - c.tail_len;
      if (c.n_outlier)
        store_vector<D, G, true>(c, which, b, h, n0 + i, to_tail, which ? vin : kin, size_t(vec) * D, in_dtype, rot,
                                 lane);
      else
        store_vector<D, G, false>(c, which, b, h, n0 + i, to_tail, which ? vin : kin, size_t(vec) * D, in_dtype, rot,
                                  lane);
    }
  }

  finish_append(c, n_new, n_new_per_seq);
}

// ---------------------------------------------------------------------------
// Block-per-lane variant for power-of-two head_dim 64 / 128 / 256 (bulk
// appends): a vector is held by R = D/32 consecutive lanes and lane l % R
// holds exactly block l % R (32 consecutive channels).  The rotation combines
// the 5 channel bits inside a lane in registers and the log2(R) block bits
// across lanes (one shuffle per value per bit); each lane then quantizes and
// stores its own block with no cross-lane reduction, 16-byte loads and stores
// throughout.  Same arithmetic as quantize_block, operation by operation.
// The grid is persistent (three CTAs per SM, grid-stride over warp tasks): the
// other resident warps' arithmetic covers a warp's loads (measured faster than
// a register prefetch of the next task, which spills at this occupancy), and
// the seq_len hand-off counts one arrival per resident CTA.
// ---------------------------------------------------------------------------

// One 32-value block held by one lane: quantize and store (qs: the block's
// bytes; qh: where the q5_x high-bit word goes; d_ptr: fp16 d or the (d, lo) word).
// Every type, one value at a time (the general path).
__device__ __forceinline__ void quantize_lane_block_scalar(const float (&y)[32], int qt, uint8_t* qs_blk,
                                                        const QhDst& qh, void* d_ptr) {
  // block parameters, then each code computed once straight into its packed byte
  float lo = 0.0f, id = 0.0f, off = 0.0f;
  int top = 0;
  const bool q8 = qt == KVQ_TYPE_Q8_0, mn = type_has_min(qt);
  if (mn) {
    float hi = y[0];
    lo = y[0];
#pragma unroll
    for (int j = 1; j < 32; ++j) {  // first index on ties: strict comparisons in ascending order
      if (y[j] < lo) lo = y[j];
      if (y[j] > hi) hi = y[j];
    }
    top = qt == KVQ_TYPE_Q5_1 ? 31 : 15;
    const float d = __fdiv_rn(__fsub_rn(hi, lo), float(top));
    id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    off = 0.5f;
    *static_cast<uint32_t*>(d_ptr) = uint32_t(__half_as_ushort(__float2half_rn(d))) |
                                     (uint32_t(__half_as_ushort(__float2half_rn(lo))) << 16);
  } else {
    float best_a = 0.0f, best_m = 0.0f;  // strict '>' scan from +0: first index on ties
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float a = fabsf(y[j]);
      if (a > best_a) { best_a = a; best_m = y[j]; }
    }
    float d;
    if (q8) {
      d = best_a / 127.0f;
    } else {
      const bool q5 = qt == KVQ_TYPE_Q5_0;
      d = q5 ? best_m / -16.0f : best_m / -8.0f;
      off = q5 ? 16.5f : 8.5f;
      top = q5 ? 31 : 15;
    }
    id = d != 0.0f ? 1.0f / d : 0.0f;
    *static_cast<__half*>(d_ptr) = __float2half_rn(d);
  }
  // code of value j, operation by operation as the block definitions state
  auto code_of = [&](int j) -> uint32_t {
    if (q8) return uint32_t(uint8_t(int8_t(int(roundf(__fmul_rn(y[j], id)))))) ^ 0x80u;  // stored offset binary
    if (mn) return uint32_t(min(top, __float2int_rz(__fadd_rn(__fmul_rn(__fsub_rn(y[j], lo), id), off))));
    return uint32_t(min(top, __float2int_rz(__fadd_rn(__fmul_rn(y[j], id), off))));
  };
  if (q8) {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      w[k] = code_of(4 * k) | (code_of(4 * k + 1) << 8) | (code_of(4 * k + 2) << 16) | (code_of(4 * k + 3) << 24);
    reinterpret_cast<uint4*>(qs_blk)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(qs_blk)[1] = make_uint4(w[4], w[5], w[6], w[7]);
    return;
  }
  // byte k = code_k | code_{k+16} << 4; high bits (q5_x) bit j = bit 4 of code_j
  uint32_t w[4] = {0u, 0u, 0u, 0u}, h = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t c0 = code_of(k), c1 = code_of(k + 16);
    w[k / 4] |= ((c0 & 0x0Fu) | ((c1 & 0x0Fu) << 4)) << (8 * (k % 4));
    h |= ((c0 >> 4) & 1u) << k;
    h |= ((c1 >> 4) & 1u) << (k + 16);
  }
  *reinterpret_cast<uint4*>(qs_blk) = make_uint4(w[0], w[1], w[2], w[3]);
  if (type_has_qh(qt)) qh_put(qh, h);
}

// trunc(x * id + off) for two values x (the code before the clamp): the
// product and the sum rounded to nearest one at a time in scalar instructions
// with explicit rounding modifiers (the compiler keeps those apart; a packed
// multiply followed by a packed add -- fp32x2 instructions, even with .rn on
// both -- came out as one fused multiply-add, which rounds once, and failed the
// bit-exact block test), then, with 0 <= u < 2^23, a packed add of
// 2^23 rounded toward zero: the sum lands on the unit grid, so its low mantissa
// bits hold floor(u) = trunc(u).
__device__ __forceinline__ void code_bits2(float x0, float x1, float id, float off, uint32_t& c0, uint32_t& c1) {
  asm("{\n\t.reg .f32 a, b;\n\t.reg .b64 x, m;\n\t"
      "mul.rn.f32 a, %2, %4;\n\tadd.rn.f32 a, a, %5;\n\t"
      "mul.rn.f32 b, %3, %4;\n\tadd.rn.f32 b, b, %5;\n\t"
      "mov.b64 x, {a, b};\n\tmov.b64 m, {%6, %6};\n\tadd.rz.f32x2 x, x, m;\n\t"
      "mov.b64 {%0, %1}, x;\n\t}"
      : "=r"(c0), "=r"(c1)
      : "f"(x0), "f"(x1), "f"(id), "f"(off), "r"(0x4B000000u));
}

// quantize_lane_block_scalar for q4_0 / q5_0, the same operations in another
// order of evaluation: the signed value of largest magnitude from a max / min
// tree (a block holding +a and -a, or no nonzero value, takes the scalar scan,
// which resolves the first-index rule); codes min(top, trunc(x*id + off)) two
// at a time by code_bits2 (scalar multiply and add, one rounding each, as
// before; the truncation packed, u > 0 here), then four codes per word: clamp to
// top, nibble pack (byte k = code_k | code_{k+16} << 4) and for q5_0 bit 4 of
// each code into the high-bit word.  q8_0, the scale + minimum types and blocks
// whose scale or inverse is not finite take the scalar path.
__device__ __forceinline__ void quantize_lane_block(float (&y)[32], int qt, uint8_t* qs_blk, const QhDst& qh,
                                                    void* d_ptr) {
  if (qt != KVQ_TYPE_Q4_0 && qt != KVQ_TYPE_Q5_0) {
    quantize_lane_block_scalar(y, qt, qs_blk, qh, d_ptr);
    return;
  }
  // four interleaved partial maxima / minima (short dependency chains, few registers)
  float mx[4], mn[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) { mx[j] = y[j]; mn[j] = y[j]; }
#pragma unroll
  for (int j = 4; j < 32; ++j) {
    mx[j & 3] = fmaxf(mx[j & 3], y[j]);
    mn[j & 3] = fminf(mn[j & 3], y[j]);
  }
  mx[0] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
  mn[0] = fminf(fminf(mn[0], mn[1]), fminf(mn[2], mn[3]));
  const float hi = mx[0], lo = mn[0];
  const bool q5 = qt == KVQ_TYPE_Q5_0;
  const float best_m = hi > -lo ? hi : lo;
  const float d = q5 ? best_m / -16.0f : best_m / -8.0f;
  const float id = d != 0.0f ? 1.0f / d : 0.0f;
  if (!(hi > -lo || -lo > hi) || !(fabsf(best_m) <= 3.0e38f) || !(fabsf(id) <= 3.0e38f)) {
    quantize_lane_block_scalar(y, qt, qs_blk, qh, d_ptr);
    return;
  }
  *static_cast<__half*>(d_ptr) = __float2half_rn(d);
  const float off = q5 ? 16.5f : 8.5f;
  const int sh = q5 ? 5 : 4;  // codes reach top + 1 at most: subtract bit log2(top + 1)
  uint32_t half16[8], h = 0;
#pragma unroll
  for (int m = 0; m < 8; ++m) {  // codes 2m, 2m+1, 2m+16, 2m+17
    uint32_t f0, f1, f16, f17;
    code_bits2(y[2 * m], y[2 * m + 1], id, off, f0, f1);
    code_bits2(y[2 * m + 16], y[2 * m + 17], id, off, f16, f17);
    const uint32_t a = __byte_perm(f0, f1, 0x0040);
    const uint32_t b = __byte_perm(f16, f17, 0x0040);
    uint32_t x = __byte_perm(a, b, 0x5410);
    x -= (x >> sh) & 0x01010101u;
    half16[m] = (x & 0x0F0Fu) | ((x >> 12) & 0xF0F0u);  // qs bytes 2m, 2m+1
    if (q5) {
      const uint32_t g = (((x >> 4) & 0x01010101u) * 0x00204081u) >> 21;  // bit 4 of the four codes
      h |= ((g & 3u) << (2 * m)) | (((g >> 2) & 3u) << (2 * m + 16));
    }
  }
  *reinterpret_cast<uint4*>(qs_blk) =
      make_uint4(__byte_perm(half16[0], half16[1], 0x5410), __byte_perm(half16[2], half16[3], 0x5410),
                 __byte_perm(half16[4], half16[5], 0x5410), __byte_perm(half16[6], half16[7], 0x5410));
  if (q5) qh_put(qh, h);
}

// Input kinds of the bulk kernel (a template parameter: no per-value select).
enum RowIn { kInBf16 = 0, kInF16 = 1, kInF32 = 2 };

// One lane's 32 input channels as raw 16-byte words (16-bit inputs: 4, fp32: 8).
template <int IN>
struct RowRaw {
  uint4 w[IN == kInF32 ? 8 : 4];
};

// Vector vec = (b * n_new + i) * H + h of K (which = 0) or V; lane sub of its R
// lanes reads channels 32*sub .. 32*sub+31 (read once: streaming loads).
template <int D, int IN>
__device__ __forceinline__ void rows_load(RowRaw<IN>& r, const void* kin, const void* vin, size_t vec, int which,
                                          int sub) {
  constexpr bool IN32 = IN == kInF32;
  const size_t e0 = vec * D + 32 * sub;
  const void* base = which ? vin : kin;
  const uint4* src = IN32 ? reinterpret_cast<const uint4*>(static_cast<const float*>(base) + e0)
                          : reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + e0);
#pragma unroll
  for (int t = 0; t < (IN32 ? 8 : 4); ++t) r.w[t] = __ldcs(src + t);
}

template <int IN>
__device__ __forceinline__ void rows_unpack(const RowRaw<IN>& r, float (&y)[32]) {
  if constexpr (IN == kInF32) {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      y[4 * t] = __uint_as_float(r.w[t].x); y[4 * t + 1] = __uint_as_float(r.w[t].y);
      y[4 * t + 2] = __uint_as_float(r.w[t].z); y[4 * t + 3] = __uint_as_float(r.w[t].w);
    }
  } else {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t w[4] = {r.w[t].x, r.w[t].y, r.w[t].z, r.w[t].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (IN == kInBf16) {
          y[8 * t + 2 * e] = __uint_as_float(w[e] << 16);
          y[8 * t + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        } else {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          y[8 * t + 2 * e] = f.x;
          y[8 * t + 2 * e + 1] = f.y;
        }
      }
    }
  }
}

// Rotate, quantize and store one lane block of new token i of (sequence b, KV
// head h), K (which = 0) or V (its values in y); `live` false: a lane past the
// end, which computes a copy and stores nothing.
template <int D, bool OUTL>
__device__ __forceinline__ void rows_task(const kvq_cache& c, int rot_k, int rot_v, int n_new,
                                          const int32_t* __restrict__ n_new_per_seq, int prerotated, bool live,
                                          int b, int i, int h, int which, float (&y)[32], int lane) {
  constexpr int R = D / 32;   // lanes per vector
  constexpr int NB = D / kQK;
  const int sub = lane % R;
  const int H = c.n_kv_heads;
  const int n0 = c.seq_len[b];
  const int nb = n_new_per_seq ? n_new_per_seq[b] : n_new;
  const bool ok = nb >= 0 && nb <= n_new && n0 >= 0 && (long long)n0 + nb <= c.max_ctx;
  if (live && !ok && i == 0 && h == 0 && which == 0 && sub == 0) atomicOr(&c.status[0], KVQ_DEV_ERR_APPEND_RANGE);

  // Outlier channels (OUTL): the raw vector is staged in shared memory; lane sub
  // takes slots sub*SL .. sub*SL+SL-1 of the head's list (their unrotated values
  // become one q8_0 block, written below), and zeroes its own block's channels
  // that are slots before the rest is rotated and quantized.
  constexpr int SL = 32 / R;  // outlier slots per lane
  float ov[OUTL ? SL : 1];
  float* raw = nullptr;
  if constexpr (OUTL) {
    __shared__ __align__(16) float s_raw[kAppendWarps][32 * 32];
    raw = &s_raw[threadIdx.x >> 5][(lane / R) * D];
    __syncwarp();  // the warp's previous task has read its staged values
#pragma unroll
    for (int t = 0; t < 8; ++t)
      *reinterpret_cast<float4*>(raw + 32 * sub + 4 * t) = make_float4(y[4 * t], y[4 * t + 1], y[4 * t + 2], y[4 * t + 3]);
    __syncwarp();
    const int32_t* idx = c.outlier_idx + (size_t)h * 32;
    uint32_t zmask = 0;
    bool bad = false;
    int prev = -1;
#pragma unroll 4
    for (int s2 = 0; s2 < 32; ++s2) {  // strictly increasing inside [0, D), as every kernel checks it
      const int ch = idx[s2];
      const bool okc = ch >= 0 && ch < D && (s2 == 0 || prev < ch);
      prev = ch;
      bad |= !okc;
      if (okc && ch / 32 == sub) zmask |= 1u << (ch % 32);
    }
#pragma unroll
    for (int k = 0; k < SL; ++k) {
      const int s2 = sub * SL + k;
      const int ch = idx[s2];
      const bool okc = ch >= 0 && ch < D && (s2 == 0 || idx[s2 - 1] < ch);
      ov[k] = okc ? raw[ch] : 0.0f;
    }
    if (bad && live && sub == 0) atomicOr(&c.status[0], KVQ_DEV_ERR_OUTLIER);
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = ((zmask >> j) & 1u) ? 0.0f : y[j];
  }
  // rotation: the R lanes of a vector rotate together; the shuffles name exactly
  // the rotating lanes (all of a bulk warp task's lanes, whose vectors are all K or
  // all V; the outlier path's second rotation covers only the tail rows)
  const bool rot = (which ? rot_v : rot_k) && !prerotated;
  const unsigned rmask = __ballot_sync(0xffffffffu, rot);
  const int qt = which ? c.v_type : c.k_type;
  if (rot) {
    lane_fwht<R>(y, lane, rmask);
    // packed scaling, except where the next operation is a subtraction (x - lo
    // of the scale + minimum types), which must not be contracted with it
    if (type_has_min(qt)) {
#pragma unroll
      for (int j = 0; j < 32; ++j) y[j] = __fmul_rn(y[j], inv_sqrt_group<D>());
    } else {
      scale32(y, inv_sqrt_group<D>());
    }
  }
  const int pos = n0 + i;
  const bool store = live && ok && i < nb;
  const long long brow = store ? body_row(row_map(c), b, h, pos) : 0;
  if (!store) {
  } else if (brow < 0) {  // page id outside the pool: the body row is not written
    if (sub == 0) atomicOr(&c.status[0], KVQ_DEV_ERR_PAGE);
  } else {
    const size_t row = size_t(brow);
    uint8_t* qs = static_cast<uint8_t*>(which ? c.v_qs : c.k_qs) + row * qs_row_bytes(qt, D) +
                  sub * (qt == KVQ_TYPE_Q8_0 ? 32 : 16);
    void* qh = which ? c.v_qh : c.k_qh;
    uint8_t* dp = static_cast<uint8_t*>(which ? c.v_d : c.k_d) + (row * NB + sub) * (type_has_min(qt) ? 4 : 2);
    quantize_lane_block(y, qt, qs, qh_dst(qh, which == 0, row, NB, sub), dp);
  }
  if constexpr (OUTL) {
    // the slots' q8_0 block: amax over the vector's R lanes, then this lane's SL codes
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < SL; ++k) amax = fmaxf(amax, fabsf(ov[k]));
#pragma unroll
    for (int m = 1; m < R; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    const float d = amax / 127.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    if (store && brow >= 0) {
      const size_t row = size_t(brow);
      uint8_t* grp = static_cast<uint8_t*>(c.outl) + (row / 16) * kOutlTile;
      uint8_t* oqs = grp + which * 512 + (row % 16) * 32 + sub * SL;
      uint32_t w[SL / 4 > 0 ? SL / 4 : 1];
#pragma unroll
      for (int k = 0; k < SL / 4; ++k) {
        w[k] = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[k] |= uint32_t(uint8_t(int8_t(int(roundf(__fmul_rn(ov[4 * k + e], id)))))) << (8 * e);
      }
      if constexpr (SL == 16) *reinterpret_cast<uint4*>(oqs) = make_uint4(w[0], w[1], w[2], w[3]);
      else if constexpr (SL == 8) *reinterpret_cast<uint2*>(oqs) = make_uint2(w[0], w[1]);
      else *reinterpret_cast<uint32_t*>(oqs) = w[0];
      if (sub == 0) reinterpret_cast<__half*>(grp + 1024 + which * 32)[row % 16] = __float2half_rn(d);
    }
    // the tail keeps the whole vector: rotate the staged raw values again
    const bool tail_row = store && c.tail_len > 0 && i >= nb - c.tail_len;
    const unsigned tmask = __ballot_sync(0xffffffffu, tail_row && rot);
    if (tail_row) {
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float4 x = *reinterpret_cast<const float4*>(raw + 32 * sub + 4 * t);
        y[4 * t] = x.x; y[4 * t + 1] = x.y; y[4 * t + 2] = x.z; y[4 * t + 3] = x.w;
      }
      if (rot) {
        lane_fwht<R>(y, lane, tmask);
        scale32(y, inv_sqrt_group<D>());
      }
    }
  }
  if (store && c.tail_len > 0 && i >= nb - c.tail_len) {
    uint16_t* tail = static_cast<uint16_t*>(which ? c.v_tail : c.k_tail) +
                     (((size_t)b * H + h) * c.tail_len + pos % c.tail_len) * D + 32 * sub;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(y[8 * t + 2 * e]))) |
               (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(y[8 * t + 2 * e + 1]))) << 16);
      reinterpret_cast<uint4*>(tail)[t] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

constexpr int kRowsCtasPerSm = 3;  // 80 registers; 24 warps per SM hide the loads

template <int D, bool OUTL, int IN>
__global__ void __launch_bounds__(kAppendWarps * 32, kRowsCtasPerSm)
append_rows_kernel(kvq_cache c, int rot_k, int rot_v, const void* __restrict__ kin, const void* __restrict__ vin,
                   int n_new, DivU32 div_h, DivU32 div_n, const int32_t* __restrict__ n_new_per_seq, int prerotated) {
  static_assert(D == 64 || D == 128 || D == 256, "power-of-two head_dim of 64 to 256");
  constexpr int R = D / 32;   // lanes per vector
  constexpr unsigned VPW = 32u / R;  // vectors per warp task
  const int lane = threadIdx.x & 31, sub = lane % R;
  // Warp tasks hold only K vectors (tasks below Wv) or only V vectors, so every lane
  // of a warp takes the same quantizer path even when K and V formats differ: task
  // wt = which * Wv + u holds vectors u*VPW .. u*VPW+VPW-1, vector vec = (b * n_new
  // + i) * H + h (one token's heads, then the next token's: contiguous input rows).
  const unsigned nvec = unsigned(c.batch) * unsigned(n_new) * unsigned(c.n_kv_heads);
  const unsigned Wv = (nvec + VPW - 1) / VPW;
  const unsigned wtasks = 2u * Wv;
  const unsigned stride = gridDim.x * unsigned(kAppendWarps);
  const int H = c.n_kv_heads;
  const unsigned lt = unsigned(lane / R);
  // strided: the warps work on neighbouring tasks at any one time, so the partial
  // sectors of the body planes they write (one token row each) meet in L2 (contiguous
  // per-warp task ranges, which balance the warps' task counts, were 18% slower)
  unsigned wt = blockIdx.x * unsigned(kAppendWarps) + (threadIdx.x >> 5);
  for (; wt < wtasks; wt += stride) {  // warp-uniform trip count
    const int which = wt >= Wv ? 1 : 0;
    const unsigned v0 = (wt - (which ? Wv : 0u)) * VPW + lt;
    const bool live = v0 < nvec;
    const unsigned vec = live ? v0 : nvec - 1;  // a lane past the end loads a valid row
    const unsigned bi = div_u32(vec, div_h);
    const int h = int(vec - bi * unsigned(H));
    const unsigned bu = div_u32(bi, div_n);
    const int i = int(bi - bu * unsigned(n_new)), b = int(bu);
    RowRaw<IN> raw;
    rows_load<D, IN>(raw, kin, vin, vec, which, sub);
    float y[32];
    rows_unpack<IN>(raw, y);
    rows_task<D, OUTL>(c, rot_k, rot_v, n_new, n_new_per_seq, prerotated, live, b, i, h, which, y, lane);
  }
  finish_append(c, n_new, n_new_per_seq);
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
    const long long brow = body_row(row_map(c), seq, kv_head, pos);
    if (brow < 0 && lane == 0) atomicOr(&c.status[0], KVQ_DEV_ERR_PAGE);
    const size_t row = brow < 0 ? 0 : size_t(brow);  // an invalid page reads as row 0 (status set)
    const uint8_t* qs = static_cast<const uint8_t*>(is_v ? c.v_qs : c.k_qs) + row * qs_row_bytes(qt, D);
    const void* qh = is_v ? c.v_qh : c.k_qh;
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
        code = int(qs[blk * 32 + k]) - 128;  // stored offset binary
      } else {
        const uint8_t byte = qs[blk * 16 + (k & 15)];
        code = k < 16 ? (byte & 15) : (byte >> 4);
        if (type_has_qh(qt)) code |= int((qh_get(qh, !is_v, row, NB, blk) >> k) & 1u) << 4;
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
          val = uint8_t(qh_get(qh, !is_v, row, NB, blk) >> (8 * (o - hb)));
        } else {
          val = qs[blk * qsb + (o - hb - qhb)] ^ (qt == KVQ_TYPE_Q8_0 ? 0x80u : 0u);  // q8_0: back to GGUF bytes
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
  if constexpr (D == 64 || D == 128 || D == 256) {
    // one block per lane (32 / (D/32) vectors per warp) for bulk appends; a few
    // vectors (a decode step) finish sooner spread one per warp
    if (warps >= kRowsMinVectors) {
      const long long per_cta = (long long)kAppendWarps * (32 / (D / 32));
      const long long full = (warps + per_cta - 1) / per_cta;
      const int sms = device_sm_count();
      const unsigned grid = unsigned(std::min<long long>(full, (long long)(sms > 0 ? sms : 148) * kRowsCtasPerSm));
      const DivU32 div_h = make_divu32(uint32_t(c.n_kv_heads)), div_n = make_divu32(uint32_t(n_new));
      auto go = [&](auto kern) {
        kern<<<grid, kAppendWarps * 32, 0, st>>>(c, rot.k, rot.v, k, v, n_new, div_h, div_n, nps, pre);
      };
      auto by_input = [&](auto outl) {
        constexpr bool O = decltype(outl)::value;
        if (in_dtype == KVQ_F32) go(append_rows_kernel<D, O, kInF32>);
        else if (in_dtype == KVQ_F16) go(append_rows_kernel<D, O, kInF16>);
        else go(append_rows_kernel<D, O, kInBf16>);
      };
      if (c.n_outlier) by_input(std::true_type{}); else by_input(std::false_type{});
      return cudaGetLastError();
    }
  }
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
    case 288: return append_d<288>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 320: return append_d<320>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 352: return append_d<352>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 384: return append_d<384>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 416: return append_d<416>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 448: return append_d<448>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 480: return append_d<480>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
    case 512: return append_d<512>(c, rot, k, v, in_dtype, n_new, nps, flags, st);
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
    case 288: return debug_d<288>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 320: return debug_d<320>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 352: return debug_d<352>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 384: return debug_d<384>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 416: return debug_d<416>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 448: return debug_d<448>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 480: return debug_d<480>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    case 512: return debug_d<512>(c, rot, seq, kv_head, which, t0, count, original_basis, out, blocks, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
