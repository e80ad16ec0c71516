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
#include "kvq_quant.cuh"

namespace kvq {
namespace {

constexpr int kAppendWarps = 8;

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
    const long long brow = body_row(row_map(c), seq, kv_head, pos);
    if (brow < 0 && lane == 0) atomicOr(&c.status[0], KVQ_DEV_ERR_PAGE);
    const size_t row = brow < 0 ? 0 : size_t(brow);  // an invalid page reads as row 0 (status set)
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
