// Prefill (prompt) attention over the rotated, block-quantized cache and its
// bf16 tail, on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// The prompt's K/V have been appended first; query i of sequence b sits at
// p = q_pos0[b] + i and, when causal, sees keys t <= p.  Scores are dot
// products in the rotated basis (velog "fix-kv-cache-quantization-outliers",
// section 아다마르 회전: rotating q and k by the same orthogonal matrix leaves
// q.k unchanged) and the output is rotated back after P.V.  Keys at positions
// >= n - tail_len are read from the bf16 tail (aitrends.kr "KVarN과 Precision
// Tail", section 용어 해설), older ones from the q4_0 / q5_0 / q8_0 body.
//
// CTA = 128 query rows (positions x the query heads of one KV head) x one KV
// head x one sequence; 4 warps, one row per thread.  Per 64-key tile:
//   1. all threads dequantize K (rows = keys) and V^T (rows = channels) into
//      shared memory as fp16 hi + lo pairs that are exact (code * scale needs
//      15 bits), scaled by 2^-8 so every stored value stays in fp16 range;
//   2. one thread issues S = Q_hi K_hi^T + Q_hi K_lo^T + Q_lo K_hi^T
//      (tcgen05.mma kind::f16, M=128, N=64) into TMEM;
//   3. each thread loads its row of S, masks, runs the online softmax, writes
//      P (fp16 hi + lo) to shared memory and rescales its O row in TMEM when
//      its running maximum moved;
//   4. one thread issues O += P_hi V_hi + P_hi V_lo + P_lo V_hi (N = head_dim).
// The three-term products keep ~22 bits, so the result matches fp32 math.
// Operands are K-major with the 128-byte swizzle (8-row atoms of 1 KB).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tcgen05.cuh"

namespace kvq {
namespace {

constexpr int kPThreads = 128;   // one query row per thread
constexpr int kPM = 128;         // query rows per CTA (UMMA M)
constexpr int kPN = 64;          // keys per tile (UMMA N of Q K^T, K of P V)
constexpr long long kPWait = 2000000000LL;  // ~1 s at 2 GHz per MMA group
constexpr float kPLog2e = 1.4426950408889634f;
constexpr float kInvScale = 0.00390625f;    // stored K/V values are x * 2^-8
constexpr float kLazyRescale = 4.0f;        // log2: P stays <= 16 * 256 in fp16

template <int D>
struct PCfg {
  static constexpr int KA = D / 64;                 // 128-byte atoms along head_dim
  static constexpr int NB = D / 32;
  static constexpr int q_bytes = KA * kPM * 128;    // [KA][128 rows][128 B]
  static constexpr int k_bytes = KA * kPN * 128;    // [KA][64 keys][128 B]
  static constexpr int v_bytes = D * 128;           // V^T: [D channels][64 keys * 2 B]
  static constexpr int p_bytes = kPM * 128;         // [128 rows][64 keys * 2 B]
  static constexpr int off_qh = 0, off_ql = q_bytes;
  static constexpr int off_kh = 2 * q_bytes, off_kl = off_kh + k_bytes;
  static constexpr int off_vh = off_kl + k_bytes, off_vl = off_vh + v_bytes;
  static constexpr int off_ph = off_vl + v_bytes, off_pl = off_ph + p_bytes;
  static constexpr int off_bar = off_pl + p_bytes;  // 2 mbarriers + TMEM address
  static constexpr int smem = off_bar + 64 + 1024;
  static constexpr int stage_stride = D + 1;        // epilogue fp32 rows (reuses Q and K)
  static_assert(kPM * stage_stride * 4 <= off_vh, "epilogue staging must fit in the Q and K tiles");
  static constexpr uint32_t idesc_qk = tc::idesc_f16_f32(kPM, kPN);
  static constexpr uint32_t idesc_pv = tc::idesc_f16_f32(kPM, D);
  static constexpr uint32_t tmem_cols = 256;        // S: columns 0..63, O: columns 128..128+D
  static constexpr uint32_t o_col = 128;
};

struct PParams {
  const uint8_t* k_qs; const uint8_t* v_qs;
  const __half* k_d; const __half* v_d;
  const uint32_t* k_qh; const uint32_t* v_qh;
  const uint16_t* k_tail; const uint16_t* v_tail;
  const int32_t* seq_len; uint32_t* status;
  int n_kv_heads, max_ctx, tail_len, k_type, v_type;
  const void* q; void* out;
  int q_dtype, out_dtype, n_q_heads, n_tokens, group, ppt, ntiles;
  const int32_t* q_pos0;
  int causal, rot_k, rot_v;
  float scale_log2;
};

// 8 channels of one stored key/value -> fp16 hi and lo (4 + 4 pairs), value scaled by 2^-8.
__device__ __forceinline__ void split8(const float (&v)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = pack_h2(v[2 * i], v[2 * i + 1]);
    const float2 f = __half22float2(u32_as_h2(h[i]));
    l[i] = pack_h2(v[2 * i] - f.x, v[2 * i + 1] - f.y);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// The 32 stored body values of block `blk` of the key at plane row `row`, x 2^-8.
template <int D>
__device__ __forceinline__ void load_body_block(const PParams& p, bool is_v, size_t row, int blk, float (&x)[32]) {
  constexpr int NB = D / 32;
  const int qt = is_v ? p.v_type : p.k_type;
  const float sc = __half2float((is_v ? p.v_d : p.k_d)[row * NB + blk]) * kInvScale;
  const uint8_t* qs = is_v ? p.v_qs : p.k_qs;
  if (qt == KVQ_TYPE_Q8_0) {
    const uint4* src = reinterpret_cast<const uint4*>(qs + row * D + blk * 32);
    const uint4 a = src[0], b = src[1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = float(int8_t(w[i >> 2] >> (8 * (i & 3)))) * sc;
  } else {
    const uint4 a = *reinterpret_cast<const uint4*>(qs + row * (D / 2) + blk * 16);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t qh = 0;
    int off = 8;
    if (qt == KVQ_TYPE_Q5_0) {
      qh = (is_v ? p.v_qh : p.k_qh)[row * NB + blk];
      off = 16;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t byte = (w[i >> 2] >> (8 * (i & 3))) & 0xFFu;
      const int lo = int(byte & 15u) | int(((qh >> i) & 1u) << 4);
      const int hi = int(byte >> 4) | int(((qh >> (i + 16)) & 1u) << 4);
      x[i] = float(lo - off) * sc;
      x[i + 16] = float(hi - off) * sc;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kPThreads, 1) prefill_kernel(PParams p) {
  using C = PCfg<D>;
  constexpr int NB = C::NB;
  constexpr int G = (D & (D - 1)) == 0 ? D : 64;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar_s = reinterpret_cast<uint64_t*>(smem + C::off_bar);
  uint64_t* bar_o = bar_s + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::off_bar + 16);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = p.ntiles - 1 - blockIdx.x;  // the longest (latest) query tiles first
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int g = p.group;
  const int n = p.seq_len[b];
  const int T = p.tail_len;
  const int p0 = p.q_pos0 ? p.q_pos0[b] : n - p.n_tokens;

  // this thread's query row
  const int li = tid / g, hh = tid % g;
  const int qi = tile * p.ppt + li;
  const bool row_ok = li < p.ppt && qi < p.n_tokens && p0 >= 0;
  const int pos = p0 + qi;
  const int head = kvh * g + hh;
  const int kv_end_row = row_ok ? (p.causal ? min(n, pos + 1) : n) : 0;
  // keys any row of the CTA can see
  const int last_q = min(p.n_tokens, (tile + 1) * p.ppt) - 1;
  const int kv_end = p0 < 0 ? 0 : (p.causal ? min(n, p0 + last_q + 1) : n);
  const int nkv = (kv_end + kPN - 1) / kPN;
  if (p0 < 0 && tid == 0 && blockIdx.x == 0 && kvh == 0) atomicOr(p.status, KVQ_DEV_ERR_PREFILL_RANGE);

  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, C::tmem_cols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_barrier_init();
  }

  // ---- Q rows: load, rotate, scale, split into hi / lo tiles ---------------
  {
    constexpr int P = G / 32;
    for (int rr = 0; rr < 32; ++rr) {
      const int r = warp * 32 + rr;
      const int rli = r / g, rhh = r % g, rqi = tile * p.ppt + rli;
      const bool ok = rli < p.ppt && rqi < p.n_tokens;
      float v[D / 32];
      const size_t base = (((size_t)b * p.n_tokens + (ok ? rqi : 0)) * p.n_q_heads + kvh * g + rhh) * D;
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        const int c = fwht_channel<D, G>(lane, j);
        float x = 0.0f;
        if (ok) {
          if (p.q_dtype == KVQ_F32) x = static_cast<const float*>(p.q)[base + c];
          else if (p.q_dtype == KVQ_BF16) x = bf16_bits_to_f32(static_cast<const uint16_t*>(p.q)[base + c]);
          else x = __half2float(static_cast<const __half*>(p.q)[base + c]);
        }
        v[j] = x;
      }
      float s = p.scale_log2;
      if (p.rot_k) {
        warp_fwht<D, G>(v, lane);
        s *= inv_sqrt_group<G>();
      }
      // lane holds P consecutive channels per G-group: write them as fp16 hi / lo
#pragma unroll
      for (int gi = 0; gi < D / G; ++gi) {
#pragma unroll
        for (int j0 = 0; j0 < P; j0 += 2) {
          const int c = gi * G + lane * P + j0;
          const float a = v[gi * P + j0] * s, bq = v[gi * P + j0 + 1] * s;
          uint32_t hi, lo;
          hi = pack_h2(a, bq);
          const float2 f = __half22float2(u32_as_h2(hi));
          lo = pack_h2(a - f.x, bq - f.y);
          const uint32_t off = (c / 64) * (kPM * 128) + tc::sw128_chunk(r, (c % 64) / 8) + (c % 8) * 2;
          *reinterpret_cast<uint32_t*>(smem + C::off_qh + off) = hi;
          *reinterpret_cast<uint32_t*>(smem + C::off_ql + off) = lo;
        }
      }
    }
  }
  fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // ---- main loop over 64-key tiles -------------------------------------------
  float m_used = -INFINITY, l = 0.0f;
  bool timed_out = false;
  uint64_t* pend_bar = bar_s;
  uint32_t pend_phase = 0;
  const size_t bh = (size_t)b * p.n_kv_heads + kvh;
  const int kk_key = tid & 63, khalf = tid >> 6;  // dequant role: key, channel half
  const uint32_t s_taddr = tmem + ((uint32_t)(warp * 32) << 16);
  const uint32_t o_taddr = s_taddr + C::o_col;

  for (int j = 0; j < nkv; ++j) {
    // 1. dequantize K and V^T of keys [64j, 64j+64) into shared memory
    {
      const int t = j * kPN + kk_key;
      const bool valid = t < kv_end;
      const bool tail = valid && t >= n - T;
      const size_t body_row = bh * p.max_ctx + (valid ? t : 0);
      const size_t tail_row = T > 0 ? (bh * T + (tail ? t % T : 0)) * D : 0;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
#pragma unroll
        for (int bb = 0; bb < NB / 2; ++bb) {
          const int blk = khalf * (NB / 2) + bb;
          float x[32];
          if (!valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = 0.0f;
          } else if (tail) {
            const uint16_t* src = (which ? p.v_tail : p.k_tail) + tail_row + blk * 32;
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              const uint4 w = *reinterpret_cast<const uint4*>(src + i);
              const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                x[i + 2 * e] = __uint_as_float(ww[e] << 16) * kInvScale;
                x[i + 2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u) * kInvScale;
              }
            }
          } else {
            load_body_block<D>(p, which == 1, body_row, blk, x);
          }
          if (which == 0) {
            // K tile: row = key, 16-byte chunks of 8 channels
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              const int c = blk * 32 + c8 * 8;
              float v8[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) v8[e] = x[c8 * 8 + e];
              uint4 hi, lo;
              split8(v8, hi, lo);
              const uint32_t off = (c / 64) * (kPN * 128) + tc::sw128_chunk(kk_key, (c % 64) / 8);
              *reinterpret_cast<uint4*>(smem + C::off_kh + off) = hi;
              *reinterpret_cast<uint4*>(smem + C::off_kl + off) = lo;
            }
          } else {
            // V^T tile: row = channel, this key's 2-byte element in it
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const int c = blk * 32 + e;
              const uint32_t h2 = pack_h2(x[e], x[e + 1]);
              const float2 f = __half22float2(u32_as_h2(h2));
              const uint32_t l2 = pack_h2(x[e] - f.x, x[e + 1] - f.y);
              const uint32_t o0 = tc::sw128_chunk(c, kk_key / 8) + (kk_key % 8) * 2;
              const uint32_t o1 = tc::sw128_chunk(c + 1, kk_key / 8) + (kk_key % 8) * 2;
              *reinterpret_cast<uint16_t*>(smem + C::off_vh + o0) = uint16_t(h2 & 0xFFFFu);
              *reinterpret_cast<uint16_t*>(smem + C::off_vh + o1) = uint16_t(h2 >> 16);
              *reinterpret_cast<uint16_t*>(smem + C::off_vl + o0) = uint16_t(l2 & 0xFFFFu);
              *reinterpret_cast<uint16_t*>(smem + C::off_vl + o1) = uint16_t(l2 >> 16);
            }
          }
        }
      }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // 2. S = Q K^T (three fp16 products)
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t qa = smem_u32(smem) + (ks / 4) * (kPM * 128) + (ks % 4) * 32;
        const uint32_t ka = smem_u32(smem) + (ks / 4) * (kPN * 128) + (ks % 4) * 32;
        const uint64_t aqh = tc::sdesc_sw128(qa + C::off_qh), aql = tc::sdesc_sw128(qa + C::off_ql);
        const uint64_t bkh = tc::sdesc_sw128(ka + C::off_kh), bkl = tc::sdesc_sw128(ka + C::off_kl);
        tc::mma_f16(tmem, aqh, bkh, C::idesc_qk, ks > 0 ? 1u : 0u);
        tc::mma_f16(tmem, aqh, bkl, C::idesc_qk, 1u);
        tc::mma_f16(tmem, aql, bkh, C::idesc_qk, 1u);
      }
      tc::commit(bar_s);
    }
    if (!mbar_wait_bounded(bar_s, j & 1, kPWait)) { timed_out = true; }
    if (__syncthreads_or(timed_out)) { timed_out = true; pend_bar = bar_s; pend_phase = j & 1; break; }
    tc::fence_after_sync();

    // 3. softmax of this thread's row; P -> shared memory; O rescale in TMEM
    float sv[kPN];
#pragma unroll
    for (int c = 0; c < kPN; c += 16) {
      float t16[16];
      tc::ld_x16(s_taddr + c, t16);
#pragma unroll
      for (int e = 0; e < 16; ++e) sv[c + e] = t16[e];
    }
    tc::wait_ld();
    float mt = -INFINITY;
#pragma unroll
    for (int c = 0; c < kPN; ++c) {
      const int t = j * kPN + c;
      sv[c] = (t < kv_end_row) ? sv[c] * 256.0f : -INFINITY;  // keys were stored x 2^-8
      mt = fmaxf(mt, sv[c]);
    }
    // lazy rescale: move the row's reference maximum only when it grew by more
    // than 2^4, so P stays <= 16 (x 256) in fp16
    float alpha = 1.0f;
    const bool move = mt > m_used + kLazyRescale || (m_used == -INFINITY && mt > -INFINITY);
    if (move) {
      alpha = m_used == -INFINITY ? 0.0f : exp2f(m_used - mt);
      l *= alpha;
      m_used = mt;
    }
    if (j > 0 && __any_sync(0xffffffffu, move)) {  // TMEM access is warp-collective
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        float t16[16];
        tc::ld_x16(o_taddr + c, t16);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) t16[e] *= alpha;
        tc::st_x16(o_taddr + c, t16);
      }
      tc::wait_st();
    }
    const float ms = m_used == -INFINITY ? 0.0f : m_used;
#pragma unroll
    for (int c8 = 0; c8 < kPN / 8; ++c8) {
      float v8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float pe = exp2f(sv[c8 * 8 + e] - ms);  // 0 for masked keys
        l += pe;
        v8[e] = pe * 256.0f;                            // values were stored x 2^-8
      }
      uint4 hi, lo;
      split8(v8, hi, lo);
      const uint32_t off = tc::sw128_chunk(tid, c8);
      *reinterpret_cast<uint4*>(smem + C::off_ph + off) = hi;
      *reinterpret_cast<uint4*>(smem + C::off_pl + off) = lo;
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // 4. O += P V (three fp16 products)
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < kPN / 16; ++ks) {
        const uint32_t pa = smem_u32(smem) + ks * 32;
        const uint64_t aph = tc::sdesc_sw128(pa + C::off_ph), apl = tc::sdesc_sw128(pa + C::off_pl);
        const uint64_t bvh = tc::sdesc_sw128(pa + C::off_vh), bvl = tc::sdesc_sw128(pa + C::off_vl);
        tc::mma_f16(tmem + C::o_col, aph, bvh, C::idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        tc::mma_f16(tmem + C::o_col, aph, bvl, C::idesc_pv, 1u);
        tc::mma_f16(tmem + C::o_col, apl, bvh, C::idesc_pv, 1u);
      }
      tc::commit(bar_o);
    }
    if (!mbar_wait_bounded(bar_o, j & 1, kPWait)) { timed_out = true; }
    if (__syncthreads_or(timed_out)) { timed_out = true; pend_bar = bar_o; pend_phase = j & 1; break; }
    tc::fence_after_sync();
  }

  if (timed_out) {
    if (tid == 0) atomicOr(p.status, KVQ_DEV_ERR_TIMEOUT);
    // let the MMA group still in flight finish (bounded) before the TMEM is released
    mbar_wait_bounded(pend_bar, pend_phase, kPWait);
  }

  // ---- epilogue: O / l -> staging -> inverse rotation -> output -------------
  float* stage = reinterpret_cast<float*>(smem);  // [128][D + 1], reuses Q and K
  {
    const float inv = (l > 0.0f && nkv > 0 && !timed_out) ? 1.0f / l : 0.0f;
#pragma unroll
    for (int c = 0; c < D; c += 16) {
      float t16[16];
      if (nkv > 0) {
        tc::ld_x16(o_taddr + c, t16);
        tc::wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) t16[e] = 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) stage[tid * C::stage_stride + c + e] = t16[e] * inv;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, C::tmem_cols);
  for (int rr = 0; rr < 32; ++rr) {
    const int r = warp * 32 + rr;
    const int rli = r / g, rhh = r % g, rqi = tile * p.ppt + rli;
    if (!(rli < p.ppt && rqi < p.n_tokens)) continue;
    float v[D / 32];
#pragma unroll
    for (int j = 0; j < D / 32; ++j) v[j] = stage[r * C::stage_stride + fwht_channel<D, G>(lane, j)];
    if (p.rot_v) {
      warp_fwht<D, G>(v, lane);
#pragma unroll
      for (int j = 0; j < D / 32; ++j) v[j] *= inv_sqrt_group<G>();
    }
    const size_t base = (((size_t)b * p.n_tokens + rqi) * p.n_q_heads + kvh * g + rhh) * D;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      const size_t e = base + fwht_channel<D, G>(lane, j);
      if (p.out_dtype == KVQ_F32) static_cast<float*>(p.out)[e] = v[j];
      else if (p.out_dtype == KVQ_BF16) static_cast<__nv_bfloat16*>(p.out)[e] = __float2bfloat16_rn(v[j]);
      else static_cast<__half*>(p.out)[e] = __float2half_rn(v[j]);
    }
  }
  (void)row_ok; (void)head;
}

template <int D>
cudaError_t run_prefill(const kvq_cache& c, Rot rot, const void* q, int q_dtype, int n_q_heads, int n_tokens,
                        const int32_t* q_pos0, int causal, float scale, void* out, int out_dtype, cudaStream_t st) {
  using Cf = PCfg<D>;
  PParams p{};
  p.k_qs = static_cast<const uint8_t*>(c.k_qs); p.v_qs = static_cast<const uint8_t*>(c.v_qs);
  p.k_d = static_cast<const __half*>(c.k_d); p.v_d = static_cast<const __half*>(c.v_d);
  p.k_qh = static_cast<const uint32_t*>(c.k_qh); p.v_qh = static_cast<const uint32_t*>(c.v_qh);
  p.k_tail = static_cast<const uint16_t*>(c.k_tail); p.v_tail = static_cast<const uint16_t*>(c.v_tail);
  p.seq_len = c.seq_len; p.status = c.status;
  p.n_kv_heads = c.n_kv_heads; p.max_ctx = c.max_ctx; p.tail_len = c.tail_len;
  p.k_type = c.k_type; p.v_type = c.v_type;
  p.q = q; p.out = out; p.q_dtype = q_dtype; p.out_dtype = out_dtype;
  p.n_q_heads = n_q_heads; p.n_tokens = n_tokens;
  p.group = n_q_heads / c.n_kv_heads;
  p.ppt = kPM / p.group;
  p.ntiles = (n_tokens + p.ppt - 1) / p.ppt;
  p.q_pos0 = q_pos0; p.causal = causal ? 1 : 0;
  p.rot_k = rot.k; p.rot_v = rot.v;
  p.scale_log2 = scale * kPLog2e;
  auto kern = prefill_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.ntiles, c.n_kv_heads, c.batch);
  kern<<<grid, kPThreads, Cf::smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int d, int group) { return (d == 64 || d == 128) && group >= 1 && group <= kPM; }

cudaError_t launch_prefill(const kvq_cache& c, Rot rot, const void* q, int q_dtype, int n_q_heads, int n_tokens,
                           const int32_t* q_pos0, int causal, float scale, void* out, int out_dtype,
                           cudaStream_t st) {
  switch (c.head_dim) {
    case 64: return run_prefill<64>(c, rot, q, q_dtype, n_q_heads, n_tokens, q_pos0, causal, scale, out, out_dtype, st);
    case 128: return run_prefill<128>(c, rot, q, q_dtype, n_q_heads, n_tokens, q_pos0, causal, scale, out, out_dtype, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
