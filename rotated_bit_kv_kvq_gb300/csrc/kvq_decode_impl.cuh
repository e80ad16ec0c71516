// Decode kernels and their host-side launch templates, included by one
// translation unit per head_dim (kvq_decode_d*.cu) so the format pairs compile
// in parallel.
#pragma once

// Decode attention over the rotated, block-quantized cache plus its bf16 tail.
//
// Scores are dot products in the rotated basis: rotating q and k by the same
// orthogonal Hadamard matrix leaves q.k unchanged, and the softmax-weighted
// sum of rotated values is rotated back at the end (velog
// "fix-kv-cache-quantization-outliers", section 아다마르 회전).  Keys and values
// of the most recent tail_len positions come from the bf16 tail, older ones
// from the q4_0 / q5_0 / q8_0 body (aitrends.kr "KVarN과 Precision Tail",
// section 용어 해설).
//
// Kernel 1 (split-K): CTA = (split, KV head x head group, sequence), 4 warps.
// Every warp streams its own 16-token tiles through a ring of shared-memory
// stages filled by TMA (tensor copies with hardware swizzle, one per plane, for the packed
// codes and bf16 rows, 1-D bulk copies for scales and q5_0 high bits).  Codes
// are turned into exact fp16 integers in registers and multiplied on the
// tensor cores (mma.m16n8k16, fp32 accumulate):
//   S[t][h]  = sum_blocks Dk[t][blk] * (codes_K[t][blk] . q[h][blk])   (q as fp16 hi + lo)
//   O[c][h] += codes_V[t][c] . (P[t][h] * Dv[t][blk(c)])                 (P as fp16)
// with an online softmax (base 2) per head.  Each CTA writes (m, l, acc).
// Kernel 2: merges the splits per query head (log-sum-exp), normalizes,
// rotates back with a warp FWHT and stores the output.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_quant.cuh"

namespace kvq {
namespace {

template <bool B>
struct BoolTag { static constexpr bool value = B; };
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxHeads = 8;                 // query heads per CTA (mma N)
constexpr long long kWaitCycles = 1000000000LL;  // ~0.5 s at 2 GHz; a TMA tile lands in microseconds
constexpr float kLog2e = 1.4426950408889634f;
// Lazy softmax reference (log2 units): the weight of a tile's largest score is at
// least 2^-kLazyMax, so P's fp16 hi / lo split keeps its relative precision.
constexpr float kLazyMax = 2.0f;
constexpr int kTailChunkMax = 4096;  // tail slots per CTA
constexpr int kSmemBudget = 64 * 1024;       // stages; leaves room for 3 CTAs per SM
constexpr int kCtasPerSm = 3;
// Outlier-channel kernels at head_dim 256 run 2 CTAs per SM: at 3 the extra
// block's registers spill inside the tile loop.
// Above head_dim 256 the accumulators alone take 80+ registers: 2 CTAs per SM as well.
constexpr int ctas_per_sm(int d, bool outl) { return (outl && d >= 256) || d > 256 ? 2 : kCtasPerSm; }

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }
// widest TMA swizzle box (128, 64 or 32 bytes) that tiles a row exactly
constexpr int box_w(int row_bytes) { return row_bytes % 128 == 0 ? 128 : (row_bytes % 64 == 0 ? 64 : 32); }

template <int D, int KT, int VT, bool OL = false>
struct Cfg {
  static constexpr int NB = D / 32;
  static constexpr int rowK = KT == KVQ_TYPE_Q8_0 ? D : D / 2;
  static constexpr int rowV = VT == KVQ_TYPE_Q8_0 ? D : D / 2;
  static constexpr int WK = box_w(rowK), WV = box_w(rowV);
  static constexpr bool K5 = type_has_qh(KT), V5 = type_has_qh(VT);
  static constexpr bool K1 = type_has_min(KT), V1 = type_has_min(VT);   // scale + minimum blocks
  static constexpr int KH = K1 ? 4 : 2, VH = V1 ? 4 : 2;                // block header bytes
  // tail stage: TT tokens of bf16 K and V
  static constexpr int TT = D >= 256 ? 8 : 16;
  static constexpr int WT = box_w(2 * D);
  static constexpr int off_kt = 0;
  static constexpr int off_vt = align_up(TT * 2 * D, 1024);
  static constexpr int tail_bytes = off_vt + TT * 2 * D;
  // body stage: RB tokens.  Up to head_dim 128 (no outlier channels) a body tile holds
  // 32 tokens, two 16-row halves, when that fits the tail stage's size: twice the
  // independent work per tile and half the per-tile overhead per token.
  static constexpr int body32 = align_up(32 * rowK, 1024) + align_up(32 * rowV, 16) + 32 * NB * (KH + VH) +
                                (K5 ? 32 * NB * 4 : 0) + (V5 ? 32 * NB * 4 : 0);
  static constexpr int RB = (D <= 128 && !OL && body32 <= tail_bytes) ? 32 : 16;
  static constexpr int HB = RB / 16;  // 16-row halves of a body tile
  static constexpr int off_kqs = 0;
  static constexpr int off_vqs = align_up(RB * rowK, 1024);
  static constexpr int off_kd = off_vqs + align_up(RB * rowV, 16);
  static constexpr int off_vd = off_kd + RB * NB * KH;
  static constexpr int off_kqh = off_vd + RB * NB * VH;
  static constexpr int off_vqh = off_kqh + (K5 ? RB * NB * 4 : 0);
  // outlier channels (OL): one 16-row group of the outlier plane (K codes, V codes, K scales, V scales)
  static constexpr int off_ko = align_up(off_vqh + (V5 ? 16 * NB * 4 : 0), 16);
  static constexpr int off_vo = off_ko + 16 * 32;
  static constexpr int off_kod = off_vo + 16 * 32;
  static constexpr int off_vod = off_kod + 16 * 2;
  static constexpr int body_bytes = OL ? off_vod + 16 * 2 : off_vqh + (V5 ? RB * NB * 4 : 0);
  static constexpr uint32_t body_tx = RB * rowK + RB * rowV + RB * NB * (KH + VH) + (K5 ? 4 * RB * NB : 0) +
                                      (V5 ? 4 * RB * NB : 0) + (OL ? 2 * 16 * 34 : 0);
  static constexpr uint32_t tail_tx = 2 * TT * 2 * D;
  static constexpr int stage = align_up(body_bytes > tail_bytes ? body_bytes : tail_bytes, 1024);
  static constexpr int NS_raw = kSmemBudget / (kWarps * stage);
  static constexpr int NS = NS_raw > 4 ? 4 : (NS_raw < 2 ? 2 : NS_raw);
  static constexpr int off_q = kWarps * NS * stage;                 // q: [8][D] fp32
  static constexpr int off_qsum = off_q + kMaxHeads * D * 4;        // [NB][8] per-block sums of q (K minimum)
  // OL: scaled, unrotated query values of the outlier slots [8][32] fp32, then their B fragments [2][32] x uint4
  static constexpr int off_qo = align_up(off_qsum + NB * kMaxHeads * 4, 16);
  static constexpr int off_qof = off_qo + kMaxHeads * 32 * 4;
  static constexpr int off_bar = OL ? off_qof + 2 * 32 * 16 : off_qsum + NB * kMaxHeads * 4;  // mbarriers [kWarps][NS]
  static constexpr int off_ml = off_bar + kWarps * NS * 8;          // [kWarps][8] m and l
  static constexpr int smem = off_ml + 2 * kWarps * kMaxHeads * 4 + 1024;  // + alignment slack
  static_assert(NB % 2 == 0, "V block headers are read in pairs of blocks");
  static_assert(kWarps * kMaxHeads * (D + (OL ? 32 : 0)) * 4 <= kWarps * NS * stage,
                "merge buffer must fit in the stages");
};

struct Params {
  const uint8_t* k_d; const uint8_t* v_d;   // fp16 d per block, or (d, lo) pairs for q4_1 / q5_1
  const uint32_t* k_qh; const uint32_t* v_qh;
  const int32_t* seq_len; uint32_t* status;
  const void* q; float* ws_acc; float* ws_ml;
  int n_kv_heads, max_ctx, tail_len;
  int q_dtype, n_q_heads, group, heads_per_cta, head_groups;
  int rot_k;
  float scale_log2;                 // softmax scale * log2(e)
  // Cost partition (DecodePlan): per plane (KV head x head group) the work of all
  // sequences -- each sequence's tail (unless the step is fused) and body, in
  // sequence order -- is one stream cut into `pieces` pieces of equal cost (bytes
  // read), at least cost_min each.  A fused step gives every tail a CTA of its own.
  // Every non-empty segment starts with a gap of cost_gap bytes that holds no data:
  // the cost of a CTA switching segments (partials, pipeline refill, queries), so a
  // piece that crosses a segment boundary carries less data, and cut points that
  // fall inside a gap move to the segment's start.
  int batch, pieces, slots;         // stream pieces and partial slots per plane
  long long cost_body, cost_tail, cost_min, cost_gap;
  int sms, wt[3];                   // piece weights by dispatch slot (Cuts), wt[0] = 0: uniform
  // fused step: new tokens written by the tail CTA (fused != 0)
  int fused, rot_v;
  FusedAppend fa;
  kvq_cache cache;
  RowMap rows;   // body row of (sequence, KV head, position): contiguous or paged
  float* ws_acco;  // outlier channels: their partials [plane][slot][head][32]
  long long* ws_hdr;  // fused step: [0] stream cost per plane, then per sequence: stream offset, tokens
};

// New tokens of sequence b in a fused step: the requested count if it fits, else 0.
__device__ __forceinline__ int fused_count(const FusedAppend& fa, int n0, int b, int max_ctx, bool& ok) {
  const int req = fa.n_new_per_seq ? fa.n_new_per_seq[b] : fa.n_new;
  ok = req >= 0 && req <= fa.n_new && n0 >= 0 && (long long)n0 + req <= max_ctx;
  return ok ? req : 0;
}

// 2^x on the special-function unit (relative error about 2^-22; results below
// 2^-126, far under any weight that matters, flush to zero)
__device__ __forceinline__ float fast_exp2(float x) { return ex2_approx(x); }

// Tokens of sequence b when the split kernel reads it (n0) and those this launch
// appends to it (nn, fused step); `flag` reports an append that does not fit.
__device__ __forceinline__ void seq_tokens(const Params& p, int b, bool flag, int& n0, int& nn) {
  n0 = p.seq_len[b];
  nn = 0;
  if (!p.fused) return;
  bool ok;
  nn = fused_count(p.fa, n0, b, p.max_ctx, ok);
  if (!ok && flag) atomicOr(p.status, KVQ_DEV_ERR_APPEND_RANGE);
}
// cost of a segment of ntok tokens of c bytes: its gap and data, nothing when empty
__device__ __forceinline__ long long seg_cost(int ntok, long long c, long long gap) {
  return ntok > 0 ? gap + (long long)ntok * c : 0LL;
}
// cost of sequence b's part of the stream: its tail (not with a fused step) and body
__device__ __forceinline__ long long stream_cost(int n, int T, int fused, long long cb, long long ct, long long gap) {
  return (fused ? 0LL : seg_cost(min(n, T), ct, gap)) + seg_cost(max(0, n - T), cb, gap);
}
// first token of a segment (ntok tokens of cost c from stream offset P) at or past
// stream offset x, rounded up to whole tiles; piece boundaries map to the same token
// in both pieces, so the pieces of a segment tile it without gaps or overlaps
__device__ __forceinline__ int seg_token(long long x, long long P, long long c, int ntok, int tile) {
  if (x <= P) return 0;
  const long long t = (x - P + c - 1) / c;
  const long long ta = (t + tile - 1) / tile * tile;
  return ta >= ntok ? ntok : int(ta);
}
// Cut points of one plane's stream into `pieces` pieces: [cut(p), cut(p + 1)).
// Uniform pieces of max(total / pieces, cost_min) bytes; or, when the grid is one
// full wave of three CTAs per SM, pieces weighted by their CTA's dispatch slot
// (the SM's first, second or third CTA: the warp scheduler favours the oldest
// warps, so equal pieces end at different times) so that an SM's CTAs end together:
// cut(p) = min(total, W(p) * unit), W(p) the weight of pieces [0, p), unit =
// ceil(total / W(pieces)).  One division per set-up; cut() is a few integer ops.
struct Cuts {
  long long total, step;  // step: bytes per piece (uniform) or per unit of weight
  int pieces, e0, e1;     // pieces below e0 run in slot 0, below e1 in slots 0-1
  int wt[3];              // wt[0] == 0: uniform
  __device__ long long wsum(int q) const {
    const int c0 = min(max(e0, 0), q), c1 = min(max(e1, 0), q);
    return (long long)wt[0] * c0 + (long long)wt[1] * (c1 - c0) + (long long)wt[2] * (q - c1);
  }
  __device__ long long cut(int q) const {
    if (q >= pieces) return total;
    return min(total, (wt[0] == 0 ? (long long)q : wsum(q)) * step);
  }
  // the last piece starting at or before stream offset pos
  __device__ int piece_of(long long pos) const {
    int lo = 0, hi = pieces - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cut(mid) <= pos) lo = mid; else hi = mid - 1;
    }
    return lo;
  }
};
// piece p of plane x runs as CTA x + (y0 + p) * planes of a grid dispatched in order
__device__ __forceinline__ Cuts make_cuts(long long total, int pieces, long long cost_min, int planes, int y0,
                                          int sms, const int (&wt)[3], int x) {
  Cuts c;
  c.total = total;
  c.pieces = pieces;
  c.e0 = (sms - x + planes - 1) / planes - y0;
  c.e1 = (2 * sms - x + planes - 1) / planes - y0;
  const bool weighted = wt[0] != 0 && total >= (long long)pieces * cost_min;
  c.wt[0] = weighted ? wt[0] : 0;
  c.wt[1] = wt[1];
  c.wt[2] = wt[2];
  if (weighted) {
    const long long W = c.wsum(pieces);
    c.step = (total + W - 1) / W;
  } else {
    c.step = max((total + pieces - 1) / pieces, cost_min);
  }
  return c;
}

// exclusive prefix sum over the CTA's threads (kThreads); *total = the sum of all
__device__ __forceinline__ long long cta_excl_scan(long long v, long long* total, long long* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  long long before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    before += w < warp ? s_warp[w] : 0LL;
    all += s_warp[w];
  }
  *total = all;
  return before + x - v;
}


// a, b -> fp16 pairs hi = fp16(a, b) and lo = fp16(a - hi, b - hi): hi + lo keeps ~22 bits.
__device__ __forceinline__ void split_h2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_h2(a, b);
  const float2 f = __half22float2(u32_as_h2(hi));
  lo = pack_h2(a - f.x, b - f.y);
}

// two adjacent fp16 values of shared memory (4-byte aligned) in one load
__device__ __forceinline__ uint32_t ld_h2(const __half* p) { return *reinterpret_cast<const uint32_t*>(p); }

// BYTES of shared memory as 32-bit words, in the widest loads the row alignment
// allows (rows of BYTES bytes from a 16-byte aligned base)
template <int BYTES>
__device__ __forceinline__ void lds_words(const uint8_t* p, uint32_t (&w)[BYTES / 4]) {
  if constexpr (BYTES % 16 == 0) {
#pragma unroll
    for (int i = 0; i < BYTES / 16; ++i) {
      const uint4 v = reinterpret_cast<const uint4*>(p)[i];
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  } else if constexpr (BYTES % 8 == 0) {
#pragma unroll
    for (int i = 0; i < BYTES / 8; ++i) {
      const uint2 v = reinterpret_cast<const uint2*>(p)[i];
      w[2 * i] = v.x; w[2 * i + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < BYTES / 4; ++i) w[i] = reinterpret_cast<const uint32_t*>(p)[i];
  }
}

// The query row `row` (of D values, f32 / bf16 / f16) as lane `lane`'s values in
// the warp FWHT layout (P = G/32 consecutive channels per group and lane): one
// vector load per group, all issued before any is used; zeros when !valid.
template <int D, int G>
__device__ __forceinline__ void load_q_fwht(const void* q, int dtype, size_t row, bool valid, int lane,
                                            float (&v)[D / 32]) {
  constexpr int P = G / 32, NG = D / G;
#pragma unroll
  for (int j = 0; j < D / 32; ++j) v[j] = 0.0f;
  if (!valid) return;
  if (dtype == KVQ_F32) {
    const float* base = static_cast<const float*>(q) + row * D + lane * P;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      const float* src = base + gi * G;
      if constexpr (P % 4 == 0) {
#pragma unroll
        for (int k = 0; k < P; k += 4) {
          const float4 x = *reinterpret_cast<const float4*>(src + k);
          v[gi * P + k] = x.x; v[gi * P + k + 1] = x.y; v[gi * P + k + 2] = x.z; v[gi * P + k + 3] = x.w;
        }
      } else if constexpr (P == 2) {
        const float2 x = *reinterpret_cast<const float2*>(src);
        v[gi * P] = x.x; v[gi * P + 1] = x.y;
      } else {
        v[gi * P] = src[0];
      }
    }
  } else {
    const uint16_t* base = static_cast<const uint16_t*>(q) + row * D + lane * P;
    uint32_t w[NG][(P + 1) / 2];
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      const uint16_t* src = base + gi * G;
      if constexpr (P == 8) {
        const uint4 x = *reinterpret_cast<const uint4*>(src);
        w[gi][0] = x.x; w[gi][1] = x.y; w[gi][2] = x.z; w[gi][3] = x.w;
      } else if constexpr (P == 4) {
        const uint2 x = *reinterpret_cast<const uint2*>(src);
        w[gi][0] = x.x; w[gi][1] = x.y;
      } else if constexpr (P == 2) {
        w[gi][0] = *reinterpret_cast<const uint32_t*>(src);
      } else {
        w[gi][0] = src[0];
      }
    }
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
#pragma unroll
      for (int k = 0; k < P; ++k) {
        const uint32_t h = (w[gi][k / 2] >> (16 * (k & 1))) & 0xFFFFu;
        v[gi * P + k] = dtype == KVQ_BF16 ? bf16_bits_to_f32(h) : __half2float(__ushort_as_half((unsigned short)h));
      }
  }
}

// half i of such a pair (0: the lower address) as fp32
__device__ __forceinline__ float h2f(uint32_t w, int i) {
  return i ? __high2float(u32_as_h2(w)) : __low2float(u32_as_h2(w));
}

// fp16 scale of block blk from a token's header words: scales only (KHH = 1, two
// blocks per word) or (scale, minimum) pairs (KHH = 2, one block per word)
template <int KHH>
__device__ __forceinline__ float hdr_scale(const uint32_t* w, int blk) {
  return KHH == 1 ? h2f(w[blk >> 1], blk & 1) : h2f(w[blk], 0);
}

// q5 high bits of one fp16 pair of K codes from a K row word already rotated by
// the lane's amount (the K plane's bit order puts the pair's two bits 16 apart):
// the mask's bits (4 / 20 or 8 / 24) with the 0x6400 magic.
__device__ __forceinline__ uint32_t khb(uint32_t h_rot, uint32_t mask) { return (h_rot & mask) | 0x64006400u; }
// q5 V high bits of one fp16 pair (two tokens, 16 bits apart) from a row-pair part
// word already rotated by the lane's amount, at the mask's bits with the 0x6400 magic
__device__ __forceinline__ uint32_t vhb(uint32_t w_rot, uint32_t mask) { return (w_rot & mask) | 0x64006400u; }

template <int D, int KT, int VT, bool OL>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(D, OL))
decode_split_kernel(Params p, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmKt, const __grid_constant__ CUtensorMap tmVt) {
  using C = Cfg<D, KT, VT, OL>;
  constexpr int NB = C::NB;
  constexpr int NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  // the warp index through a shuffle from lane 0: visibly the same in every lane, so
  // the copy addresses derived from it can stay warp-uniform
  const int tid = threadIdx.x, lane = tid & 31, warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
  const int g = lane >> 2, tig = lane & 3;
  // grid (plane = KV head x head group, piece): piece y of every plane is dispatched
  // before piece y + 1
  const int plane = blockIdx.x;
  const int kvh = plane / p.head_groups;
  const int hg = plane % p.head_groups;
  const int head0 = kvh * p.group + hg * p.heads_per_cta;
  const int nheads = min(p.heads_per_cta, p.group - hg * p.heads_per_cta);
  const int T = p.tail_len;
  const int B = p.batch;
  const bool cta0 = blockIdx.x == 0 && blockIdx.y == 0;
  const bool own_tail = p.fused && int(blockIdx.y) < B;  // fused step: the tail of sequence y
  const long long piece = own_tail ? -1LL : (long long)blockIdx.y - (p.fused ? B : 0);

  float* sq = reinterpret_cast<float*>(smem + C::off_q);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::off_bar);
  float* sm_m = reinterpret_cast<float*>(smem + C::off_ml);
  float* sm_l = sm_m + kWarps * kMaxHeads;
  __shared__ long long s_scan[kWarps];

  // The piece's cursor (stream offset, sequence, segment kind, staged queries'
  // sequence) lives in shared memory between sub-ranges; every thread advances a
  // copy identically.
  __shared__ long long s_cur_P, s_x[2];  // cursor offset; the piece's [x0, x1)
  __shared__ int s_cur[5];  // sequence, next segment kind (0 tail, 1 body), staged sequence, slot, last
  __shared__ int s_first[3];  // the piece's first sequence and its tokens (read, appended)
  if (tid == 0) {
    for (int i = 0; i < kWarps * NS; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
    prefetch_tmap(&tmK); prefetch_tmap(&tmV);
    if (T > 0) { prefetch_tmap(&tmKt); prefetch_tmap(&tmVt); }
    s_cur_P = 0;
    s_cur[0] = own_tail ? int(blockIdx.y) : -1;
    s_cur[1] = (p.fused && !own_tail) ? 1 : 0;
    s_cur[2] = -1;
    s_first[0] = -1;
  }

  // ---- the partition: every CTA computes the same cut from seq_len ----------
  // (the merge kernel works out the same numbers, or with a fused step reads the ones CTA 0
  // records; CTA 0 also flags appends that do not fit)
  {
    constexpr int kCache = 4;  // sequences per thread kept in registers (batch <= 512)
    const int per = (B + kThreads - 1) / kThreads;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int c0[kCache], cn[kCache];
    long long mine = 0;
#pragma unroll
    for (int i = 0; i < kCache; ++i) {
      c0[i] = cn[i] = 0;
      if (b0 + i < b1) seq_tokens(p, b0 + i, cta0, c0[i], cn[i]);
      mine += stream_cost(c0[i] + cn[i], T, p.fused, p.cost_body, p.cost_tail, p.cost_gap);
    }
    for (int bb = b0 + kCache; bb < b1; ++bb) {
      int n0, nn;
      seq_tokens(p, bb, cta0, n0, nn);
      mine += stream_cost(n0 + nn, T, p.fused, p.cost_body, p.cost_tail, p.cost_gap);
    }
    long long total;
    long long P = cta_excl_scan(mine, &total, s_scan);  // (its barrier orders the cursor set-up above)
    const Cuts cu = make_cuts(total, p.pieces, p.cost_min, p.head_groups * p.n_kv_heads, p.fused ? B : 0, p.sms,
                              p.wt, plane);
    const long long x0 = piece >= 0 ? cu.cut(int(piece)) : 0;
    if (tid == 0) { s_x[0] = x0; s_x[1] = piece >= 0 ? cu.cut(int(piece) + 1) : 0; }
    for (int bb = b0; bb < b1; ++bb) {
      int n0, nn;
      if (bb - b0 < kCache) {
#pragma unroll
        for (int i = 0; i < kCache; ++i)
          if (bb - b0 == i) { n0 = c0[i]; nn = cn[i]; }
      } else {
        seq_tokens(p, bb, false, n0, nn);
      }
      const int n = n0 + nn;
      const long long c = stream_cost(n, T, p.fused, p.cost_body, p.cost_tail, p.cost_gap);
      if (cta0 && p.fused) { p.ws_hdr[1 + 2 * bb] = P; p.ws_hdr[2 + 2 * bb] = n; }
      const bool first = own_tail ? bb == int(blockIdx.y) : (piece >= 0 && c > 0 && P <= x0 && x0 < P + c);
      if (first) {
        s_cur_P = P;
        s_cur[0] = bb;
        s_first[0] = bb; s_first[1] = n0; s_first[2] = nn;
      }
      P += c;
    }
    if (cta0 && p.fused && tid == 0) p.ws_hdr[0] = total;
  }
  __syncthreads();

  // The merge kernel may launch now: its CTAs take the SM slots that this grid's
  // CTAs free as they finish and wait there for this grid's completion.  (It
  // launches only after every CTA of this grid has started and reached this point.)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- the piece's sub-ranges, one (sequence, tail or body) segment each ------
  uint32_t kk = 0;  // tiles this warp consumed (ring phases)
  // K1 (scale + minimum K blocks): B fragment of the minimum's mma, the block sums of q
  // as fp16 hi / lo for blocks 2tig, 2tig + 1 (and + 8, + 9) of head g
  uint32_t bqh[2] = {0u, 0u}, bql[2] = {0u, 0u};
  bool timed_out = false;
  for (;;) {
    // find the next non-empty sub-range of this piece (empty ones get an empty partial)
    int b = 0, n0 = 0, nn = 0, t_begin = 0, t_end = 0, slot = 0, cur_b;
    bool is_tail = false, last = true, found = false;
    {
      const long long x0 = s_x[0], x1 = s_x[1];
      long long Pseg = s_cur_P;
      int sb = s_cur[0], kind = s_cur[1];
      cur_b = s_cur[2];
      while (sb >= 0 && sb < B) {
        b = sb;
        if (b == s_first[0]) {
          n0 = s_first[1];
          nn = s_first[2];
        } else {
          seq_tokens(p, b, false, n0, nn);
        }
        const int n = n0 + nn;
        is_tail = kind == 0;
        bool use = false;
        if (own_tail) {
          t_begin = 0;
          t_end = min(n, T);
          slot = b;
          use = true;
          sb = B;  // nothing after it
        } else {
          const int ntok = is_tail ? min(n, T) : max(0, n - T);
          const long long c = is_tail ? p.cost_tail : p.cost_body;
          const long long cs = (long long)ntok * c;
          if (cs > 0) {
            const long long dstart = Pseg + p.cost_gap;  // the segment's data starts after its gap
            if (dstart < x1 && dstart + cs > x0) {
              use = true;
              const int tile = is_tail ? C::TT : C::RB;
              t_begin = seg_token(x0, dstart, c, ntok, tile);
              t_end = seg_token(x1, dstart, c, ntok, tile);
              slot = p.fused ? B + int(piece) + b : int(piece) + 2 * b + kind;
            }
            Pseg = dstart + cs;
          }
          if (p.fused || kind == 1) { kind = p.fused ? 1 : 0; ++sb; } else { kind = 1; }
          if (Pseg >= x1) sb = B;
        }
        last = sb >= B;
        if (use && t_begin < t_end) { found = true; break; }
        if (use && tid < nheads) {  // nothing to read: an empty partial
          float* ml = p.ws_ml + ((size_t)plane * p.slots + slot) * p.heads_per_cta * 2;
          ml[2 * tid] = -INFINITY;
          ml[2 * tid + 1] = 0.0f;
        }
      }
      __syncthreads();  // every thread has read the cursor
      if (tid == 0) {
        s_cur_P = Pseg; s_cur[0] = sb; s_cur[1] = kind; s_cur[2] = found ? b : cur_b;
        s_cur[3] = slot; s_cur[4] = last;
      }
    }
    if (!found) break;
  // (every thread found the same sub-range; taken from lane 0 so that the compiler
  // sees warp-uniform values in the copy addressing)
  b = __shfl_sync(0xffffffffu, b, 0);
  t_begin = __shfl_sync(0xffffffffu, t_begin, 0);
  t_end = __shfl_sync(0xffffffffu, t_end, 0);
  is_tail = __shfl_sync(0xffffffffu, int(is_tail), 0) != 0;

  // ---- this warp's tiles, and the producer (one lane) --------------------
  const int TR = is_tail ? C::TT : C::RB;                    // rows per tile
  const int ntiles = (t_end - t_begin + TR - 1) / TR;
  const int my_tiles = ntiles > warp ? (ntiles - warp + kWarps - 1) / kWarps : 0;
  uint8_t* wstage = smem + warp * NS * C::stage;
  uint64_t* wbar = bars + warp * NS;
  const size_t bh = (size_t)b * p.n_kv_heads + kvh;
  const bool paged = p.rows.page_tokens != 0;
  uint32_t bad_stage = 0;  // lane 0: bit s set when the tile in stage s came from a page outside the pool

  auto issue = [&](int k) {  // tile k of this warp's sub-range -> stage (kk + k) % NS (lane 0 only)
    const int s = (kk + k) % NS;
    uint8_t* st = wstage + s * C::stage;
    const int t0 = t_begin + (warp + k * kWarps) * TR;
    if (is_tail) {
      const int row = int(bh * T + t0);
      mbar_arrive_expect_tx(&wbar[s], C::tail_tx);
      tma_3d_g2s(st + C::off_kt, &tmKt, row, &wbar[s]);  // [column][TT rows][WT bytes]
      tma_3d_g2s(st + C::off_vt, &tmVt, row, &wbar[s]);
    } else {
      size_t row = bh * p.max_ctx + t0;
      if (paged) {  // a body tile (16 or 32 tokens, aligned) never crosses a page (a multiple of 64)
        const int pg = p.rows.page_table[(size_t)b * (p.max_ctx / p.rows.page_tokens) + t0 / p.rows.page_tokens];
        const bool bad = pg < 0 || pg >= p.rows.n_pages;
        bad_stage = (bad_stage & ~(1u << s)) | (bad ? (1u << s) : 0u);
        if (bad) {  // outside the pool: fetch row 0, the consumer masks the tile
          atomicOr(p.status, KVQ_DEV_ERR_PAGE);
          row = 0;
        } else {
          row = ((size_t)pg * p.n_kv_heads + kvh) * p.rows.page_tokens + t0 % p.rows.page_tokens;
        }
      }
      mbar_arrive_expect_tx(&wbar[s], C::body_tx);
      // one copy per plane: [box column of W bytes][RB rows][W bytes]
      tma_3d_g2s(st + C::off_kqs, &tmK, int(row), &wbar[s]);
      tma_3d_g2s(st + C::off_vqs, &tmV, int(row), &wbar[s]);
      bulk_g2s(st + C::off_kd, p.k_d + row * NB * C::KH, C::RB * NB * C::KH, &wbar[s]);
      bulk_g2s(st + C::off_vd, p.v_d + row * NB * C::VH, C::RB * NB * C::VH, &wbar[s]);
      if constexpr (C::K5) bulk_g2s(st + C::off_kqh, p.k_qh + row * NB, C::RB * NB * 4, &wbar[s]);
      if constexpr (C::V5) bulk_g2s(st + C::off_vqh, p.v_qh + row * NB, C::RB * NB * 4, &wbar[s]);
      if constexpr (OL) {  // outlier rows: 32 codes + one fp16 scale per token, K and V
        // the tile's 16-row group of the outlier plane has the stage's layout: one copy
        bulk_g2s(st + C::off_ko, static_cast<const uint8_t*>(p.cache.outl) + (row / 16) * kOutlTile, kOutlTile,
                 &wbar[s]);
      }
    }
  };

  // the query rows of a newly touched sequence: loads issued before the tile copies,
  // which would otherwise queue ahead of them
  constexpr int GQR = (D >= 64 && D % 64 == 0) ? (((D & (D - 1)) == 0) ? D : 64) : 32;
  float qv[2][D / 32];  // warp w: heads w and w + 4 in the FWHT layout
  if (b != cur_b) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int hh = warp + kWarps * i;
      load_q_fwht<D, GQR>(p.q, p.q_dtype, (size_t)b * p.n_q_heads + head0 + hh, hh < nheads, lane, qv[i]);
    }
  }

  // Fused step: this (sequence, KV head)'s only tail CTA writes the new tokens
  // (body blocks and bf16 tail rows) before any tail tile is fetched.  Body CTAs
  // never treat those positions as valid: they are >= n - T.  The proxy fence
  // makes the stores visible to the tensor copies issued after the barrier.
  if (p.fused && is_tail && nn > 0) {
    constexpr int GQ = (D >= 64 && D % 64 == 0) ? (((D & (D - 1)) == 0) ? D : 64) : 32;
    for (int t = warp; t < 2 * nn; t += kWarps) {
      const int i = t >> 1, which = t & 1;
      const bool rot = (which ? p.rot_v : p.rot_k) && !p.fa.prerotated;
      store_vector<D, GQ, OL>(p.cache, which, b, kvh, n0 + i, true, which ? p.fa.v : p.fa.k,
                          (((size_t)b * p.fa.n_new + i) * p.n_kv_heads + kvh) * D, p.fa.in_dtype, rot, lane);
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  __syncthreads();  // barriers initialised (and the fused step's tokens stored)
  if (elect_one()) {
    for (int k = 0; k < NS && k < my_tiles; ++k) issue(k);
  }

  // ---- queries: load, rotate, scale, split into fp16 hi/lo fragments ----
  // (once per sequence the piece touches)
  float* qo = reinterpret_cast<float*>(smem + C::off_qo);  // OL: [8][32] unrotated, scaled
  // B fragments: k-step (blk, half) covers channels 32*blk + 16*half + 4*tig + {0,2 | 1,3}.
  // They are the same in every warp: warp 0 builds them once and leaves them in
  // shared memory over the q staging ([blk][half][lane] x {hi b0b1, hi b2b3, lo b0b1,
  // lo b2b3}, 32*D bytes = the staging's size), so no warp holds them in registers.
  const uint4* qfs = reinterpret_cast<const uint4*>(sq);
  float* qsum = reinterpret_cast<float*>(smem + C::off_qsum);  // [blk][head]: sum of the block's q values
  if (b != cur_b) {
    constexpr int G = GQR;
    if constexpr (OL) {  // the outlier slots take the unrotated values
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < D / 32; ++j) sq[(warp + kWarps * i) * D + fwht_channel<D, G>(lane, j)] = qv[i][j];
      __syncthreads();
      if (warp == 0) {
        const int ch = outlier_channel<D>(p.cache, kvh, lane);
#pragma unroll
        for (int hh = 0; hh < kMaxHeads; ++hh) qo[hh * 32 + lane] = ch >= 0 ? sq[hh * D + ch] * p.scale_log2 : 0.0f;
      }
      __syncthreads();
    }
    {
      float sc = p.scale_log2;
      if (p.rot_k) sc *= inv_sqrt_group<G>();
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (p.rot_k) warp_fwht<D, G>(qv[i], lane);
#pragma unroll
        for (int j = 0; j < D / 32; ++j) sq[(warp + kWarps * i) * D + fwht_channel<D, G>(lane, j)] = qv[i][j] * sc;
      }
    }
    __syncthreads();
    // fragments: warp w builds blocks w, w + 4, ... from the staged values, then (after
    // every warp has read them) writes them over the staging
    constexpr int BPW = (NB + kWarps - 1) / kWarps;
    uint4 qf[BPW][2];
#pragma unroll
    for (int u = 0; u < BPW; ++u) {
      const int blk = warp + kWarps * u;
      if (blk < NB) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const float4 q4 = *reinterpret_cast<const float4*>(sq + g * D + 32 * blk + 16 * hf + 4 * tig);
          const float qx[4] = {q4.x, q4.y, q4.z, q4.w};
          float hi[4], lo[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            hi[j] = __half2float(__float2half_rn(qx[j]));
            lo[j] = qx[j] - hi[j];
          }
          qf[u][hf] = make_uint4(pack_h2(hi[0], hi[2]), pack_h2(hi[1], hi[3]), pack_h2(lo[0], lo[2]),
                                 pack_h2(lo[1], lo[3]));
        }
      }
    }
    if constexpr (C::K1) {  // the block sums of q (for the K minimum), one (block, head) per thread
      for (int i = tid; i < NB * kMaxHeads; i += kThreads) {
        const int blk = i / kMaxHeads, hh = i % kMaxHeads;
        float t = 0.0f;
        for (int c = 0; c < 32; ++c) t += sq[hh * D + blk * 32 + c];
        qsum[i] = t;
      }
    }
    if constexpr (OL) {  // the outlier slots' B fragments, same layout as one block of qf
      if (warp == 0) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const float4 q4 = *reinterpret_cast<const float4*>(qo + g * 32 + 16 * hf + 4 * tig);
          const float qx[4] = {q4.x, q4.y, q4.z, q4.w};
          float hi[4], lo[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            hi[j] = __half2float(__float2half_rn(qx[j]));
            lo[j] = qx[j] - hi[j];
          }
          reinterpret_cast<uint4*>(smem + C::off_qof)[hf * 32 + lane] =
              make_uint4(pack_h2(hi[0], hi[2]), pack_h2(hi[1], hi[3]), pack_h2(lo[0], lo[2]), pack_h2(lo[1], lo[3]));
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < BPW; ++u) {
      const int blk = warp + kWarps * u;
      if (blk < NB) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) reinterpret_cast<uint4*>(sq)[(blk * 2 + hf) * 32 + lane] = qf[u][hf];
      }
    }
    __syncthreads();
    if constexpr (C::K1) {
#pragma unroll
      for (int e = 0; e < (NB > 8 ? 2 : 1); ++e) {
        const int b0 = 2 * tig + 8 * e;
        const float x0 = b0 < NB ? qsum[b0 * kMaxHeads + g] : 0.0f;
        const float x1 = b0 + 1 < NB ? qsum[(b0 + 1) * kMaxHeads + g] : 0.0f;
        split_h2(x0, x1, bqh[e], bql[e]);
      }
    }
  }  // queries of sequence b staged
  const uint4* qofs = reinterpret_cast<const uint4*>(smem + C::off_qof);

  // ---- main loop ------------------------------------------------------------
  float acc[NB][2][4];
#pragma unroll
  for (int i = 0; i < NB; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.0f;
  float acco[OL ? 2 : 1][4];  // OL: outlier slots 0-15 / 16-31 (body tiles only)
#pragma unroll
  for (int j = 0; j < (OL ? 2 : 1); ++j)
#pragma unroll
    for (int r = 0; r < 4; ++r) acco[j][r] = 0.0f;
  // V1 (scale + minimum V blocks): sum over this lane's transposed tokens of P * lo per
  // block, for head g, in the running-max frame; added to the block's channels at the end
  // V1: sum_t P[t][h] * lo[t][blk] as one more mma accumulator, rows = blocks g, g + 8
  // (A = the tile's block minima, blocks x tokens), columns = heads 2tig, 2tig + 1
  float dmin[4] = {0.f, 0.f, 0.f, 0.f};
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  int k_stop = my_tiles;
  // per-lane ldmatrix row and swizzle constants of the body tiles
  const int mi = lane >> 3, rr = (lane & 7) + 8 * (mi & 1);
  // q5 K: rotations of a stored high-bit word bringing the lane's channel pairs
  // (4tig, 4tig+2) [kr[0]] and (4tig+1, 4tig+3) [kr[1]] to bits 4 / 20, and with the
  // same rotations (16+4tig, 18+4tig) and (17+4tig, 19+4tig) to bits 8 / 24 (their
  // nibbles are read in place, x16)
  uint32_t kr[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) kr[w] = uint32_t(8 * (tig >> 1) + 2 * (tig & 1) + w - 4) & 31u;
  // q5 V: rotations of the lane's part word (part g / 4) of a row pair bringing channel
  // 2g [vr[0]] and 2g + 1 [vr[1]] to bits 4 / 20, and with the same rotations channels
  // 2g + 16 and 2g + 17 to bits 8 / 24
  uint32_t vr[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) vr[w] = uint32_t(8 * ((g & 3) >> 1) + 2 * (g & 1) + w - 4) & 31u;
  uint32_t lbK[C::WK / 32], lbV[C::WV / 32];
  swz_lane<C::WK>(rr, mi >> 1, lbK);
  swz_lane<C::WV>(rr, mi >> 1, lbV);

  // The tile loop, compiled once for tail and once for body sub-ranges: each copy holds
  // only its own kind's code, which keeps the body loop compact in the instruction cache.
  auto tile_loop = [&](auto tail_tag) {
  constexpr bool kTail = decltype(tail_tag)::value;
  const int TR = kTail ? C::TT : C::RB;  // rows per tile (a constant in each copy)
  for (int k = 0; k < my_tiles; ++k) {
    const int s = (kk + k) % NS;
    const bool arrived = mbar_wait_bounded(&wbar[s], ((kk + k) / NS) & 1, kWaitCycles);
    if (!__all_sync(0xffffffffu, arrived)) { timed_out = true; k_stop = k; break; }
    const uint8_t* st = wstage + s * C::stage;
    const int t0 = t_begin + (warp + k * kWarps) * TR;
    // positions past the end, or a whole tile whose page id lies outside the pool, are masked
    int t_lim = t_end;
    if (paged && ((__shfl_sync(0xffffffffu, bad_stage, 0) >> s) & 1u)) t_lim = t0;
    // validity of the lane's rows 16hh + g and 16hh + g + 8 of the tile (a tail tile is
    // one half of 16 or 8 rows)
    constexpr int HB = C::HB;
    bool vv[HB][2];
#pragma unroll
    for (int hh = 0; hh < HB; ++hh) {
      vv[hh][0] = 16 * hh < TR && t0 + 16 * hh + g < t_lim;
      vv[hh][1] = 16 * hh + 8 < TR && t0 + 16 * hh + g + 8 < t_lim;
    }

    float S[HB][4];
#pragma unroll
    for (int hh = 0; hh < HB; ++hh) S[hh][0] = S[hh][1] = S[hh][2] = S[hh][3] = 0.f;
    if constexpr (!kTail) {
#pragma unroll
      for (int hh = 0; hh < HB; ++hh) {
      // ------------------------------- body: scores of rows 16hh .. 16hh + 15
      // block headers of this lane's tokens 16hh + g and 16hh + g + 8, all blocks
      constexpr int KHH = C::KH / 2;
      uint32_t kw0[NB * KHH / 2], kw8[NB * KHH / 2];
      lds_words<NB * C::KH>(st + C::off_kd + (16 * hh + g) * NB * C::KH, kw0);
      lds_words<NB * C::KH>(st + C::off_kd + (16 * hh + g + 8) * NB * C::KH, kw8);
      const uint32_t kbase = smem_u32(st + C::off_kqs) + hh * 16 * C::WK;
      if constexpr (KT == KVQ_TYPE_Q8_0) {
#pragma unroll
        for (int blk = 0; blk < NB; ++blk) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kbase + lbK[swz_lane_idx<C::WK>(2 * blk)] + swz_box_off<C::WK, C::RB>(2 * blk), r0, r1, r2, r3);
          const uint32_t alo[4] = {i8_pair<0, 2>(r0), i8_pair<0, 2>(r1), i8_pair<1, 3>(r0), i8_pair<1, 3>(r1)};
          const uint32_t ahi[4] = {i8_pair<0, 2>(r2), i8_pair<0, 2>(r3), i8_pair<1, 3>(r2), i8_pair<1, 3>(r3)};
          const uint4 qa = qfs[(blk * 2) * 32 + lane], qb = qfs[(blk * 2 + 1) * 32 + lane];
          float cc[4] = {0.f, 0.f, 0.f, 0.f};
          mma16816(cc, alo, qa.x, qa.y);
          mma16816(cc, alo, qa.z, qa.w);
          mma16816(cc, ahi, qb.x, qb.y);
          mma16816(cc, ahi, qb.z, qb.w);
          const float dk0 = hdr_scale<KHH>(kw0, blk), dk8 = hdr_scale<KHH>(kw8, blk);
          S[hh][0] += dk0 * cc[0]; S[hh][1] += dk0 * cc[1];
          S[hh][2] += dk8 * cc[2]; S[hh][3] += dk8 * cc[3];
        }
      } else {
        constexpr uint32_t OFF = (0x6400u + uint32_t(type_code_offset(KT))) * 0x10001u;
        constexpr uint32_t OFF16 = neg_off_x16_bits(type_code_offset(KT));
#pragma unroll
        for (int bp = 0; bp < NB; bp += 2) {
          uint32_t rr4[4];
          ldsm_x4(kbase + lbK[swz_lane_idx<C::WK>(bp)] + swz_box_off<C::WK, C::RB>(bp), rr4[0], rr4[1], rr4[2], rr4[3]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int blk = bp + e;
            const uint32_t ra = rr4[2 * e], rb = rr4[2 * e + 1];  // token g, token g+8
            const uint32_t ra8 = ra >> 8, rb8 = rb >> 8;
            // high bits: at bit 4 / 20 for the low nibbles, bit 8 / 24 for the x16 high nibbles
            uint32_t m00 = 0x64006400u, m01 = 0x64006400u, m02 = 0x64006400u, m03 = 0x64006400u;
            uint32_t m10 = 0x64006400u, m11 = 0x64006400u, m12 = 0x64006400u, m13 = 0x64006400u;
            if constexpr (C::K5) {
              const uint32_t* kqh = reinterpret_cast<const uint32_t*>(st + C::off_kqh);
              const uint32_t ha = kqh[(16 * hh + g) * NB + blk], hb = kqh[(16 * hh + g + 8) * NB + blk];
              const uint32_t ha0 = __funnelshift_r(ha, ha, kr[0]), ha1 = __funnelshift_r(ha, ha, kr[1]);
              const uint32_t hb0 = __funnelshift_r(hb, hb, kr[0]), hb1 = __funnelshift_r(hb, hb, kr[1]);
              m00 = khb(ha0, 0x00100010u); m01 = khb(ha1, 0x00100010u);
              m02 = khb(ha0, 0x01000100u); m03 = khb(ha1, 0x01000100u);
              m10 = khb(hb0, 0x00100010u); m11 = khb(hb1, 0x00100010u);
              m12 = khb(hb0, 0x01000100u); m13 = khb(hb1, 0x01000100u);
            }
            const uint32_t alo[4] = {nib_pair(ra, 0, m00, OFF), nib_pair(rb, 0, m10, OFF),
                                     nib_pair(ra8, 0, m01, OFF), nib_pair(rb8, 0, m11, OFF)};
            const uint32_t ahi[4] = {nib_pair_x16(ra, m02, OFF16), nib_pair_x16(rb, m12, OFF16),
                                     nib_pair_x16(ra8, m03, OFF16), nib_pair_x16(rb8, m13, OFF16)};
            const uint4 qa = qfs[(blk * 2) * 32 + lane], qb = qfs[(blk * 2 + 1) * 32 + lane];
            float cc[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816(cc, alo, qa.x, qa.y);
            mma16816(cc, alo, qa.z, qa.w);
            mma16816(cc, ahi, qb.x, qb.y);
            mma16816(cc, ahi, qb.z, qb.w);
            const float dk0 = hdr_scale<KHH>(kw0, blk), dk8 = hdr_scale<KHH>(kw8, blk);
            S[hh][0] += dk0 * cc[0]; S[hh][1] += dk0 * cc[1];
            S[hh][2] += dk8 * cc[2]; S[hh][3] += dk8 * cc[3];
          }
        }
        if constexpr (C::K1) {  // + sum_blk lo[t][blk] * (sum of block blk's q)[h]: one mma per q part
          const uint8_t* kd = st + C::off_kd;
          auto lo2 = [&](int t, int b0) -> uint32_t {  // minima of blocks b0, b0 + 1 of row t
            if (b0 >= NB) return 0u;
            const uint2 w = *reinterpret_cast<const uint2*>(kd + ((16 * hh + t) * NB + b0) * 4);
            return __byte_perm(w.x, w.y, 0x7632);
          };
          const uint32_t am[4] = {lo2(g, 2 * tig), lo2(g + 8, 2 * tig), NB > 8 ? lo2(g, 2 * tig + 8) : 0u,
                                  NB > 8 ? lo2(g + 8, 2 * tig + 8) : 0u};
          mma16816(S[hh], am, bqh[0], bqh[1]);
          mma16816(S[hh], am, bql[0], bql[1]);
        }
      }
      }  // halves
      if constexpr (OL) {  // + d_O[t] * (codes_O[t] . q_O[h]): one q8_0 block in plain 32-byte rows
        uint32_t r0, r1, r2, r3;
        ldsm_x4(smem_u32(st + C::off_ko) + rr * 32 + 16 * (mi >> 1), r0, r1, r2, r3);
        r0 ^= 0x80808080u; r1 ^= 0x80808080u; r2 ^= 0x80808080u; r3 ^= 0x80808080u;
        const uint32_t alo[4] = {i8_pair<0, 2>(r0), i8_pair<0, 2>(r1), i8_pair<1, 3>(r0), i8_pair<1, 3>(r1)};
        const uint32_t ahi[4] = {i8_pair<0, 2>(r2), i8_pair<0, 2>(r3), i8_pair<1, 3>(r2), i8_pair<1, 3>(r3)};
        const uint4 qa = qofs[lane], qb = qofs[32 + lane];
        float cc[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(cc, alo, qa.x, qa.y);
        mma16816(cc, alo, qa.z, qa.w);
        mma16816(cc, ahi, qb.x, qb.y);
        mma16816(cc, ahi, qb.z, qb.w);
        static_assert(HB == 1, "outlier-channel tiles are 16 rows");
        const __half* kod = reinterpret_cast<const __half*>(st + C::off_kod);
        const float dk0 = __half2float(kod[g]), dk8 = __half2float(kod[g + 8]);
        S[0][0] += dk0 * cc[0]; S[0][1] += dk0 * cc[1];
        S[0][2] += dk8 * cc[2]; S[0][3] += dk8 * cc[3];
      }
    } else {
      // ------------------------------- tail (bf16, stored as fp16 * 2^-8): scores
      const uint8_t* kt = st + C::off_kt;
      float cc[4] = {0.f, 0.f, 0.f, 0.f};
      auto tail_k = [&](int blk) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int xb = 2 * (32 * blk + 16 * hf + 4 * tig);
          const uint2 ka = *reinterpret_cast<const uint2*>(kt + swz_off<C::WT>(g, xb, C::TT));
          uint2 kb = make_uint2(0u, 0u);
          if (C::TT == 16) kb = *reinterpret_cast<const uint2*>(kt + swz_off<C::WT>(g + 8 < C::TT ? g + 8 : g, xb, C::TT));
          const uint32_t a[4] = {bf16x2_to_h2_scaled(__byte_perm(ka.x, ka.y, 0x5410)),
                                 C::TT == 16 ? bf16x2_to_h2_scaled(__byte_perm(kb.x, kb.y, 0x5410)) : 0u,
                                 bf16x2_to_h2_scaled(__byte_perm(ka.x, ka.y, 0x7632)),
                                 C::TT == 16 ? bf16x2_to_h2_scaled(__byte_perm(kb.x, kb.y, 0x7632)) : 0u};
          const uint4 qa = qfs[(blk * 2 + hf) * 32 + lane];
          mma16816(cc, a, qa.x, qa.y);
          mma16816(cc, a, qa.z, qa.w);
        }
      };
      if constexpr (D >= 256) {
        // kept rolled at the large head dims: tail tiles are few there (8 tokens each, a small
        // share of the tokens), and the smaller kernel keeps the body loop's instruction fetch
        // cheaper (64k workload 98.9 -> 98.0 us); below, the tail is a larger share and the
        // unrolled form is faster
#pragma unroll 1
        for (int blk = 0; blk < NB; ++blk) tail_k(blk);
      } else {
#pragma unroll
        for (int blk = 0; blk < NB; ++blk) tail_k(blk);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) S[0][r] = 256.0f * cc[r];
    }

    // ---- online softmax (base 2); rows g, g+8 = tokens, cols 2tig, 2tig+1 = heads
    // Rows past the end exist only in a warp's last tile (and in tiles of a page
    // outside the pool): a warp-uniform branch.  8-row tail tiles leave the mma's
    // rows g+8 empty in every tile.
    const bool partial = t0 + TR > t_lim;
    if (partial || TR < 16 * HB) {
#pragma unroll
      for (int hh = 0; hh < HB; ++hh) {
        if (!vv[hh][0]) { S[hh][0] = -INFINITY; S[hh][1] = -INFINITY; }
        if (!vv[hh][1]) { S[hh][2] = -INFINITY; S[hh][3] = -INFINITY; }
      }
    }
    float mx0 = fmaxf(S[0][0], S[0][2]), mx1 = fmaxf(S[0][1], S[0][3]);
#pragma unroll
    for (int hh = 1; hh < HB; ++hh) {
      mx0 = fmaxf(mx0, fmaxf(S[hh][0], S[hh][2]));
      mx1 = fmaxf(mx1, fmaxf(S[hh][1], S[hh][3]));
    }
    // m0 / m1 are reference points, not the running maxima: kLazyMax above the
    // maximum seen at the last rescale.  Weights 2^(S - m) stay <= 1, and the
    // reduction over the tile's rows and the rescale run only when a score passes
    // the reference -- a few times per head and sub-range, not at every new maximum.
    if (__any_sync(0xffffffffu, mx0 > m0 || mx1 > m1)) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float nm0 = fmaxf(m0, mx0 + kLazyMax), nm1 = fmaxf(m1, mx1 + kLazyMax);
      const float a0 = m0 == -INFINITY ? 0.0f : fast_exp2(m0 - nm0);
      const float a1 = m1 == -INFINITY ? 0.0f : fast_exp2(m1 - nm1);
      l0 *= a0; l1 *= a1;
#pragma unroll
      for (int i = 0; i < NB; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          acc[i][j][0] *= a0; acc[i][j][1] *= a1; acc[i][j][2] *= a0; acc[i][j][3] *= a1;
        }
      if constexpr (OL) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          acco[j][0] *= a0; acco[j][1] *= a1; acco[j][2] *= a0; acco[j][3] *= a1;
        }
      }
      if constexpr (C::V1) {
        dmin[0] *= a0; dmin[1] *= a1; dmin[2] *= a0; dmin[3] *= a1;
      }
      m0 = nm0; m1 = nm1;
    }
    const float ms0 = m0 == -INFINITY ? 0.0f : m0, ms1 = m1 == -INFINITY ? 0.0f : m1;
    float pp[HB][4];
#pragma unroll
    for (int hh = 0; hh < HB; ++hh) {
      pp[hh][0] = fast_exp2(S[hh][0] - ms0); pp[hh][1] = fast_exp2(S[hh][1] - ms1);
      pp[hh][2] = fast_exp2(S[hh][2] - ms0); pp[hh][3] = fast_exp2(S[hh][3] - ms1);
      l0 += pp[hh][0] + pp[hh][2]; l1 += pp[hh][1] + pp[hh][3];
    }

    // ---- P.V.  P is split into fp16 hi + lo parts and transposed once per tile
    // (movmatrix) into the B-fragment layout: tokens 2tig, 2tig+1 (ph0, pl0) and
    // 2tig+8, 2tig+9 (ph1, pl1) of head g.  Each block scales both parts by the
    // tokens' V scales in fp16 arithmetic (hscale_split: ~22 bits, like P itself);
    // the codes are exact.
    uint32_t ph0[HB], pl0[HB], ph1[HB], pl1[HB];
    bool vt0[HB], vt1[HB], vt8[HB], vt9[HB];  // validity of the lane's transposed rows
#pragma unroll
    for (int hh = 0; hh < HB; ++hh) {
      const float p0 = pp[hh][0], p1 = pp[hh][1], p2 = pp[hh][2], p3 = pp[hh][3];
      const uint32_t h0 = pack_h2(p0, p1), h1 = pack_h2(p2, p3);
      const float2 f0 = __half22float2(u32_as_h2(h0)), f1 = __half22float2(u32_as_h2(h1));
      const uint32_t r0 = pack_h2(p0 - f0.x, p1 - f0.y), r1 = pack_h2(p2 - f1.x, p3 - f1.y);
      ph0[hh] = movm_t(h0); pl0[hh] = movm_t(r0); ph1[hh] = movm_t(h1); pl1[hh] = movm_t(r1);
      const int tt = t0 + 16 * hh + 2 * tig;  // first token of this lane's transposed rows
      vt0[hh] = 16 * hh < TR && tt < t_lim;
      vt1[hh] = 16 * hh < TR && tt + 1 < t_lim;
      vt8[hh] = 16 * hh + 8 < TR && tt + 8 < t_lim;
      vt9[hh] = 16 * hh + 8 < TR && tt + 9 < t_lim;
    }
    if constexpr (!kTail) {
#pragma unroll
      for (int hh = 0; hh < HB; ++hh) {
      // V block headers of the lane's four transposed tokens (rows 16hh + ...), all blocks;
      // zero for rows past the end (their bytes may be anything, and 0 * Inf would poison the sum)
      constexpr int VHH = C::VH / 2;              // halves per block header
      constexpr int VW = NB * VHH / 2;            // header words per token
      uint32_t vh[4][VW];
      {
        const uint8_t* vd = st + C::off_vd;
        const int trow[4] = {16 * hh + 2 * tig, 16 * hh + 2 * tig + 1, 16 * hh + 2 * tig + 8, 16 * hh + 2 * tig + 9};
        const bool tok_ok[4] = {vt0[hh], vt1[hh], vt8[hh], vt9[hh]};
#pragma unroll
        for (int i = 0; i < 4; ++i) lds_words<NB * C::VH>(vd + trow[i] * NB * C::VH, vh[i]);
        if (partial) {  // full tiles hold written body rows only
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < VW; ++j) vh[i][j] = tok_ok[i] ? vh[i][j] : 0u;
        }
      }
      // scale pair of block blk for tokens (ta, tb) of the four
      auto dvpair = [&](int blk, int ta, int tb) -> uint32_t {
        if constexpr (VHH == 1) return __byte_perm(vh[ta][blk >> 1], vh[tb][blk >> 1], (blk & 1) ? 0x7632 : 0x5410);
        else return __byte_perm(vh[ta][blk], vh[tb][blk], 0x5410);
      };
      // P times the V scale of block blk, as fp16 hi + lo B fragments
      auto pscaled = [&](int blk, uint32_t& bh0, uint32_t& bl0, uint32_t& bh1, uint32_t& bl1) {
        hscale_split(ph0[hh], pl0[hh], dvpair(blk, 0, 1), bh0, bl0);
        hscale_split(ph1[hh], pl1[hh], dvpair(blk, 2, 3), bh1, bl1);
      };
      // the minimum adds sum_t P[t][h] * lo[t][blk] to every channel of the block: one mma
      // per P part with A = the minima of blocks g (and g + 8) at the lane's four transposed
      // tokens (zero for rows past the end: their bytes may be anything)
      if constexpr (C::V1) {
        const uint8_t* vd = st + C::off_vd;
        const int tr[4] = {16 * hh + 2 * tig, 16 * hh + 2 * tig + 1, 16 * hh + 2 * tig + 8, 16 * hh + 2 * tig + 9};
        const bool ok[4] = {vt0[hh], vt1[hh], vt8[hh], vt9[hh]};
        auto lo2 = [&](int blk, int i0, int i1) -> uint32_t {  // (d, lo) words -> the two lo halves
          const int bb = blk < NB ? blk : NB - 1;
          uint32_t w0 = *reinterpret_cast<const uint32_t*>(vd + (tr[i0] * NB + bb) * 4);
          uint32_t w1 = *reinterpret_cast<const uint32_t*>(vd + (tr[i1] * NB + bb) * 4);
          if (partial) { w0 = ok[i0] ? w0 : 0u; w1 = ok[i1] ? w1 : 0u; }
          return blk < NB ? __byte_perm(w0, w1, 0x7632) : 0u;
        };
        const uint32_t al[4] = {lo2(g, 0, 1), NB > 8 ? lo2(g + 8, 0, 1) : 0u, lo2(g, 2, 3),
                                NB > 8 ? lo2(g + 8, 2, 3) : 0u};
        mma16816(dmin, al, ph0[hh], ph1[hh]);
        mma16816(dmin, al, pl0[hh], pl1[hh]);
      }
      const uint32_t vbase = smem_u32(st + C::off_vqs) + hh * 16 * C::WV;
      if constexpr (VT == KVQ_TYPE_Q8_0) {
#pragma unroll
        for (int blk = 0; blk < NB; ++blk) {
          uint32_t bh0, bl0, bh1, bl1;
          pscaled(blk, bh0, bl0, bh1, bl1);
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(vbase + lbV[swz_lane_idx<C::WV>(2 * blk)] + swz_box_off<C::WV, C::RB>(2 * blk), r0, r1, r2, r3);
          const uint32_t a0[4] = {i8_pair<0, 2>(r0), i8_pair<1, 3>(r0), i8_pair<0, 2>(r1), i8_pair<1, 3>(r1)};
          const uint32_t a1[4] = {i8_pair<0, 2>(r2), i8_pair<1, 3>(r2), i8_pair<0, 2>(r3), i8_pair<1, 3>(r3)};
          mma16816(acc[blk][0], a0, bh0, bh1);
          mma16816(acc[blk][0], a0, bl0, bl1);
          mma16816(acc[blk][1], a1, bh0, bh1);
          mma16816(acc[blk][1], a1, bl0, bl1);
        }
      } else {
        constexpr uint32_t OFF = (0x6400u + uint32_t(type_code_offset(VT))) * 0x10001u;
        constexpr uint32_t OFF16 = neg_off_x16_bits(type_code_offset(VT));
#pragma unroll
        for (int bp = 0; bp < NB; bp += 2) {
          uint32_t rr4[4];
          ldsm_x4_t(vbase + lbV[swz_lane_idx<C::WV>(bp)] + swz_box_off<C::WV, C::RB>(bp), rr4[0], rr4[1], rr4[2], rr4[3]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int blk = bp + e;
            uint32_t bh0, bl0, bh1, bl1;
            pscaled(blk, bh0, bl0, bh1, bl1);
            const uint32_t ra = rr4[2 * e], rb = rr4[2 * e + 1];  // tokens 0-7, 8-15
            const uint32_t ra8 = ra >> 8, rb8 = rb >> 8;
            // high bits: at bit 4 / 20 for the low nibbles, bit 8 / 24 for the x16 high nibbles
            uint32_t ma0 = 0x64006400u, ma1 = 0x64006400u, ma2 = 0x64006400u, ma3 = 0x64006400u;
            uint32_t mb0 = 0x64006400u, mb1 = 0x64006400u, mb2 = 0x64006400u, mb3 = 0x64006400u;
            if constexpr (C::V5) {
              // the V plane's row pairs: the lane's part word of rows 2tig, 2tig+1 (pair tig)
              // and of rows 2tig+8, 2tig+9 (pair tig + 4)
              const uint32_t wa =
                  *reinterpret_cast<const uint32_t*>(st + C::off_vqh + (((8 * hh + tig) * NB + blk) * 2 + (g >> 2)) * 4);
              const uint32_t wb = *reinterpret_cast<const uint32_t*>(
                  st + C::off_vqh + (((8 * hh + tig + 4) * NB + blk) * 2 + (g >> 2)) * 4);
              const uint32_t wa0 = __funnelshift_r(wa, wa, vr[0]), wa1 = __funnelshift_r(wa, wa, vr[1]);
              const uint32_t wb0 = __funnelshift_r(wb, wb, vr[0]), wb1 = __funnelshift_r(wb, wb, vr[1]);
              ma0 = vhb(wa0, 0x00100010u); ma1 = vhb(wa1, 0x00100010u);
              ma2 = vhb(wa0, 0x01000100u); ma3 = vhb(wa1, 0x01000100u);
              mb0 = vhb(wb0, 0x00100010u); mb1 = vhb(wb1, 0x00100010u);
              mb2 = vhb(wb0, 0x01000100u); mb3 = vhb(wb1, 0x01000100u);
            }
            const uint32_t a0[4] = {nib_pair(ra, 0, ma0, OFF), nib_pair(ra8, 0, ma1, OFF),
                                    nib_pair(rb, 0, mb0, OFF), nib_pair(rb8, 0, mb1, OFF)};
            const uint32_t a1[4] = {nib_pair_x16(ra, ma2, OFF16), nib_pair_x16(ra8, ma3, OFF16),
                                    nib_pair_x16(rb, mb2, OFF16), nib_pair_x16(rb8, mb3, OFF16)};
            mma16816(acc[blk][0], a0, bh0, bh1);
            mma16816(acc[blk][0], a0, bl0, bl1);
            mma16816(acc[blk][1], a1, bh0, bh1);
            mma16816(acc[blk][1], a1, bl0, bl1);
          }
        }
      }
      }  // halves
      if constexpr (OL) {  // outlier slots += codes_O^T . (P * d_O), as one more q8_0 block
        const __half* vod = reinterpret_cast<const __half*>(st + C::off_vod);
        const uint32_t mlo = (vt0[0] ? 0x0000FFFFu : 0u) | (vt1[0] ? 0xFFFF0000u : 0u);
        const uint32_t mhi = (vt8[0] ? 0x0000FFFFu : 0u) | (vt9[0] ? 0xFFFF0000u : 0u);
        uint32_t bh0, bl0, bh1, bl1;
        hscale_split(ph0[0], pl0[0], ld_h2(vod + 2 * tig) & mlo, bh0, bl0);
        hscale_split(ph1[0], pl1[0], ld_h2(vod + 2 * tig + 8) & mhi, bh1, bl1);
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(smem_u32(st + C::off_vo) + rr * 32 + 16 * (mi >> 1), r0, r1, r2, r3);
        r0 ^= 0x80808080u; r1 ^= 0x80808080u; r2 ^= 0x80808080u; r3 ^= 0x80808080u;
        const uint32_t a0[4] = {i8_pair<0, 2>(r0), i8_pair<1, 3>(r0), i8_pair<0, 2>(r1), i8_pair<1, 3>(r1)};
        const uint32_t a1[4] = {i8_pair<0, 2>(r2), i8_pair<1, 3>(r2), i8_pair<0, 2>(r3), i8_pair<1, 3>(r3)};
        mma16816(acco[0], a0, bh0, bh1);
        mma16816(acco[0], a0, bl0, bl1);
        mma16816(acco[1], a1, bh0, bh1);
        mma16816(acco[1], a1, bl0, bl1);
      }
    } else {
      // tail values are stored as fp16 * 2^-8, so P carries the factor 256
      float pt[4];
      {
        const float2 a0 = __half22float2(u32_as_h2(ph0[0])), b0 = __half22float2(u32_as_h2(pl0[0]));
        const float2 a1 = __half22float2(u32_as_h2(ph1[0])), b1 = __half22float2(u32_as_h2(pl1[0]));
        pt[0] = a0.x + b0.x; pt[1] = a0.y + b0.y; pt[2] = a1.x + b1.x; pt[3] = a1.y + b1.y;
      }
      uint32_t bh0, bl0, bh1, bl1;
      split_h2(pt[0] * 256.0f, pt[1] * 256.0f, bh0, bl0);
      split_h2(pt[2] * 256.0f, pt[3] * 256.0f, bh1, bl1);
      // token validity of the rows this lane reads from the transposed tile
      const uint32_t mlo = (vt0[0] ? 0x0000FFFFu : 0u) | (vt1[0] ? 0xFFFF0000u : 0u);
      const uint32_t mhi = (vt8[0] ? 0x0000FFFFu : 0u) | (vt9[0] ? 0xFFFF0000u : 0u);
      const uint32_t vbase = smem_u32(st + C::off_vt);
      const int rt = (lane & 7) + (C::TT == 16 ? 8 * (mi >> 1) : 0);
#pragma unroll
      for (int blk = 0; blk < NB; ++blk)
#pragma unroll
        for (int cc2 = 0; cc2 < 2; ++cc2) {
          const int mt = 2 * blk + cc2;  // 16 channels
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(vbase + swz_off<C::WT>(rt, 2 * (16 * mt + 8 * (mi & 1)), C::TT), r0, r1, r2, r3);
          const uint32_t a[4] = {bf16x2_to_h2_scaled(r0) & mlo, bf16x2_to_h2_scaled(r1) & mlo,
                                 bf16x2_to_h2_scaled(r2) & mhi, bf16x2_to_h2_scaled(r3) & mhi};
          mma16816(acc[blk][cc2], a, bh0, bh1);
          mma16816(acc[blk][cc2], a, bl0, bl1);
        }
    }
    __syncwarp();
    if (k + NS < my_tiles && elect_one()) {
      fence_proxy_async_smem();
      issue(k + NS);
    }
  }
  };
  if (is_tail) tile_loop(BoolTag<true>{});
  else tile_loop(BoolTag<false>{});

  if (timed_out) {
    if (lane == 0) atomicOr(p.status, KVQ_DEV_ERR_TIMEOUT);
    // wait (bounded) for this warp's copies still in flight before leaving:
    // tiles k_stop .. k_stop+NS-1 were issued and not consumed
    for (int k = k_stop; k < my_tiles && k < k_stop + NS; ++k) {
      const int s = (kk + k) % NS;
      mbar_wait_bounded(&wbar[s], ((kk + k) / NS) & 1, kWaitCycles);
    }
  }
  kk += my_tiles;
  const int slot_w = s_cur[3];
  const bool last_w = s_cur[4] != 0;


  // ---- merge the 4 warps, write this CTA's partial ---------------------------
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  if (g == 0) {
    sm_m[warp * kMaxHeads + 2 * tig] = m0; sm_m[warp * kMaxHeads + 2 * tig + 1] = m1;
    sm_l[warp * kMaxHeads + 2 * tig] = l0; sm_l[warp * kMaxHeads + 2 * tig + 1] = l1;
  }
  __syncthreads();  // all warps done with their stages; sm_m / sm_l complete
  float f0, f1;
  {
    float M0 = -INFINITY, M1 = -INFINITY;
    for (int w = 0; w < kWarps; ++w) {
      M0 = fmaxf(M0, sm_m[w * kMaxHeads + 2 * tig]);
      M1 = fmaxf(M1, sm_m[w * kMaxHeads + 2 * tig + 1]);
    }
    f0 = (m0 == -INFINITY) ? 0.0f : fast_exp2(m0 - M0);
    f1 = (m1 == -INFINITY) ? 0.0f : fast_exp2(m1 - M1);
  }
  float* macc = reinterpret_cast<float*>(smem);  // [kWarps][8][D], reuses the stages
#pragma unroll
  for (int blk = 0; blk < NB; ++blk)
#pragma unroll
    for (int cc2 = 0; cc2 < 2; ++cc2) {
      const int mt = 2 * blk + cc2;
      const int cg = is_tail ? 16 * mt + g : 16 * mt + 2 * g;
      const int cg8 = is_tail ? 16 * mt + g + 8 : 16 * mt + 2 * g + 1;
      float* base = macc + (size_t)warp * kMaxHeads * D;
      base[(2 * tig) * D + cg] = acc[blk][cc2][0] * f0;
      base[(2 * tig + 1) * D + cg] = acc[blk][cc2][1] * f1;
      base[(2 * tig) * D + cg8] = acc[blk][cc2][2] * f0;
      base[(2 * tig + 1) * D + cg8] = acc[blk][cc2][3] * f1;
    }
  if constexpr (C::V1) {  // blocks g, g + 8 for heads 2tig, 2tig + 1, in this warp's merge frame
    __syncwarp();
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int blk = g + 8 * half;
      if (blk < NB) {
        const float v0 = dmin[2 * half] * f0, v1 = dmin[2 * half + 1] * f1;
        float* r0 = macc + ((size_t)warp * kMaxHeads + 2 * tig) * D + 32 * blk;
#pragma unroll 8
        for (int c = 0; c < 32; ++c) {
          r0[c] += v0;
          r0[D + c] += v1;
        }
      }
    }
  }
  float* maco = macc + (size_t)kWarps * kMaxHeads * D;  // OL: [kWarps][8][32]
  if constexpr (OL) {
#pragma unroll
    for (int cc2 = 0; cc2 < 2; ++cc2) {
      const int sl = 16 * cc2 + 2 * g;
      float* base = maco + (size_t)warp * kMaxHeads * 32;
      base[(2 * tig) * 32 + sl] = acco[cc2][0] * f0;
      base[(2 * tig + 1) * 32 + sl] = acco[cc2][1] * f1;
      base[(2 * tig) * 32 + sl + 1] = acco[cc2][2] * f0;
      base[(2 * tig + 1) * 32 + sl + 1] = acco[cc2][3] * f1;
    }
  }
  __syncthreads();
  for (int i = tid; i < nheads * D; i += kThreads) {
    const int hh = i / D, c = i % D;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += macc[((size_t)w * kMaxHeads + hh) * D + c];
    p.ws_acc[(((size_t)plane * p.slots + slot_w) * p.heads_per_cta + hh) * D + c] = v;
  }
  if constexpr (OL) {
    for (int i = tid; i < nheads * 32; i += kThreads) {
      const int hh = i / 32, c = i % 32;
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v += maco[((size_t)w * kMaxHeads + hh) * 32 + c];
      p.ws_acco[(((size_t)plane * p.slots + slot_w) * p.heads_per_cta + hh) * 32 + c] = v;
    }
  }
  if (tid < nheads) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * kMaxHeads + tid]);
    float L = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
      const float mw = sm_m[w * kMaxHeads + tid];
      if (mw != -INFINITY) L += sm_l[w * kMaxHeads + tid] * fast_exp2(mw - M);
    }
    float* ml = p.ws_ml + ((size_t)plane * p.slots + slot_w) * p.heads_per_cta * 2;
    ml[2 * tid] = M;
    ml[2 * tid + 1] = L;
  }
  __syncthreads();  // this sub-range's partial written; its stages, q and (m, l) free again
  if (last_w || timed_out) break;
  }  // sub-ranges
}

// ---------------------------------------------------------------------------
// Split merge + inverse rotation: one CTA of 256 threads per (sequence, query
// head).  The partition header (written by the split kernel) gives the sequence's
// stream offset and length, from which the slots holding its partials follow: for
// each of its segments, the pieces that intersect it.  The slot weights
// 2^(m_s - M) go to shared memory; then every thread owns channels (D <= 256: a
// group of 256 / D threads shares a channel and takes every (256/D)-th slot), so
// all partial loads of a row are independent and coalesced; warp 0 rotates the
// merged row back.
// ---------------------------------------------------------------------------

struct CombineArgs {
  const float* ws_acc; const float* ws_ml; const float* ws_acco; const long long* hdr;
  int slots, heads_per_cta, head_groups, group, batch, tail_len, fused, rot_v, out_dtype, n_q_heads;
  int pieces, planes, sms, wt[3];
  long long cost_body, cost_tail, cost_min, cost_gap;
  void* out;
  int32_t* seq_len;      // fused step: advanced to the recorded token count
  const int32_t* oidx;   // outlier channels [kv_head][32]
};

// slots of one segment: the stream pieces it intersects, as a first slot and a count
__device__ __forceinline__ void seg_slots(const Cuts& cu, long long P, long long cs, int base, int& s0, int& cnt) {
  if (cs <= 0) { s0 = 0; cnt = 0; return; }
  const int p0 = cu.piece_of(P), p1 = cu.piece_of(P + cs - 1);
  s0 = base + p0;
  cnt = p1 - p0 + 1;
}

template <int D, bool OL, int kCombineThreads>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(CombineArgs a) {
  constexpr int G = (D >= 64 && D % 64 == 0) ? (((D & (D - 1)) == 0) ? D : 64) : 32;
  constexpr int E = D / 32;
  constexpr int TPC = kCombineThreads / D >= 1 ? kCombineThreads / D : 1;  // threads per channel
  __shared__ float s_part[kCombineThreads];      // per-thread partial sums
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;  // b * Hq + h
  const int b = row / a.n_q_heads, h = row % a.n_q_heads;
  const int kvh = h / a.group, r = h % a.group;
  const int plane = kvh * a.head_groups + r / a.heads_per_cta, hh = r % a.heads_per_cta;
  // This row's slots (two runs), from the partition; lane 0 of the CTA does the cut
  // arithmetic once.  Decode alone: worked out before waiting for the split grid, from
  // seq_len (which the split kernel reads too and nobody writes; the same integer sums,
  // so the same cuts).  A fused step advances seq_len after the wait, and a merge CTA
  // that becomes resident late could read an advanced length there: it reads the
  // sequence offsets and token counts the split's CTA 0 recorded, after the wait.
  __shared__ long long s_sum[2][kCombineThreads / 32];
  __shared__ int s_runs[4], s_n;
  auto runs = [&](long long total, long long P, int n) {
    const Cuts cu = make_cuts(total, a.pieces, a.cost_min, a.planes, a.fused ? a.batch : 0, a.sms, a.wt, plane);
    const int T = a.tail_len;
    const long long ct = (long long)min(n, T) * a.cost_tail, cb = (long long)max(0, n - T) * a.cost_body;
    const long long gap = a.cost_gap;  // every non-empty segment's data follows a gap
    int q0, k0, q1, k1;
    if (a.fused) {
      q0 = b; k0 = min(n, T) > 0 ? 1 : 0;
      seg_slots(cu, P + gap, cb, a.batch + b, q1, k1);
    } else {
      seg_slots(cu, P + gap, ct, 2 * b, q0, k0);
      seg_slots(cu, P + (ct > 0 ? gap + ct : 0) + gap, cb, 2 * b + 1, q1, k1);
    }
    s_runs[0] = q0; s_runs[1] = k0; s_runs[2] = q1; s_runs[3] = k1;
  };
  if (!a.fused) {
    long long mine = 0, pre = 0;
    for (int bb = tid; bb < a.batch; bb += kCombineThreads) {
      const int n = a.seq_len[bb];
      const long long cst = stream_cost(n, a.tail_len, 0, a.cost_body, a.cost_tail, a.cost_gap);
      mine += cst;
      if (bb < b) pre += cst;
      if (bb == b) s_n = n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mine += __shfl_xor_sync(0xffffffffu, mine, o);
      pre += __shfl_xor_sync(0xffffffffu, pre, o);
    }
    if (lane == 0) { s_sum[0][warp] = mine; s_sum[1][warp] = pre; }
    __syncthreads();
    if (tid == 0) {
      long long total = 0, P = 0;
#pragma unroll
      for (int w = 0; w < kCombineThreads / 32; ++w) { total += s_sum[0][w]; P += s_sum[1][w]; }
      runs(total, P, s_n);
    }
  }
  // launched as a programmatic dependent of the split kernel: wait for its completion
  // (and memory) before reading anything it wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (a.fused && tid == 0) {
    const int n = int(a.hdr[2 + 2 * b]);
    runs(a.hdr[0], a.hdr[1 + 2 * b], n);
    if (h == 0) a.seq_len[b] = n;  // every split CTA has read seq_len: advance it (head 0's CTA)
  }
  __syncthreads();
  const int r0 = s_runs[0], c0 = s_runs[1], r1 = s_runs[2], c1 = s_runs[3];
  const int splits = c0 + c1;
  auto slot_of = [&](int j) { return j < c0 ? r0 + j : r1 + (j - c0); };
  const size_t base = (size_t)plane * a.slots;  // slot rows of this plane
  // Thread (channel c, sub) merges slots sub, sub + TPC, ... in batches of kBatch, every
  // load of a batch issued before any is used: the batch's maximum M, then the weight
  // sum L and the channel's weighted sum v, the running values rescaled when M grows.
  // A slot whose sub-range was empty holds only (m, l) = (-inf, 0); its acc row is
  // whatever an earlier call left there: read, but selected away by its weight 0 and
  // never multiplied.
  constexpr int kBatch = kCombineThreads >= 512 ? 16 : 8;  // wide CTAs serve rows with many slots
  const int c = tid % D, sub = tid / D;
  const bool has_ch = tid < D * TPC;
  float M = -INFINITY, L = 0.0f, v = 0.0f;
  for (int s0 = sub; has_ch && s0 < splits; s0 += kBatch * TPC) {
    float bm[kBatch], bl[kBatch], bx[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = s0 + u * TPC;
      bm[u] = -INFINITY; bl[u] = 0.0f; bx[u] = 0.0f;
      if (j < splits) {
        const size_t ri = (base + slot_of(j)) * a.heads_per_cta + hh;
        const float2 ml = *reinterpret_cast<const float2*>(a.ws_ml + ri * 2);
        bm[u] = ml.x; bl[u] = ml.y;
        bx[u] = a.ws_acc[ri * D + c];
      }
    }
    // (slot j is warp-uniform: a warp's threads share sub; absent slots cost nothing)
    float mb = M;
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (s0 + u * TPC < splits) mb = fmaxf(mb, bl[u] > 0.0f ? bm[u] : -INFINITY);
    const float fo = M == -INFINITY ? 0.0f : fast_exp2(M - mb);
    L *= fo;
    v *= fo;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (s0 + u * TPC < splits) {
        const float w = bl[u] > 0.0f ? fast_exp2(bm[u] - mb) : 0.0f;
        L = fmaf(bl[u], w, L);
        v += w != 0.0f ? w * bx[u] : 0.0f;
      }
    }
    M = mb;
  }
  // the TPC threads of a channel: their sums, and each sub's (M, L) (the same in all its threads)
  __shared__ float s_m[TPC], s_l[TPC];
  s_part[tid] = v;
  if (has_ch && c == 0) { s_m[sub] = M; s_l[sub] = L; }
  __syncthreads();
  // 4. warp 0: the subs combined, / L, inverse rotation, (+ outlier channels), store
  if (warp != 0) return;
  float Mg = -INFINITY;
#pragma unroll
  for (int u = 0; u < TPC; ++u) Mg = fmaxf(Mg, s_m[u]);
  float fu[TPC], Lg = 0.0f;
#pragma unroll
  for (int u = 0; u < TPC; ++u) {
    fu[u] = s_m[u] == -INFINITY ? 0.0f : fast_exp2(s_m[u] - Mg);
    Lg = fmaf(s_l[u], fu[u], Lg);
  }
  const float inv = Lg > 0.0f ? 1.0f / Lg : 0.0f;
  float x[E];
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const int ch = fwht_channel<D, G>(lane, j);
    float t = 0.0f;
#pragma unroll
    for (int u = 0; u < TPC; ++u) t += fu[u] != 0.0f ? s_part[u * D + ch] * fu[u] : 0.0f;
    x[j] = t * inv;
  }
  if (a.rot_v) {
    warp_fwht<D, G>(x, lane);
#pragma unroll
    for (int j = 0; j < E; ++j) x[j] *= inv_sqrt_group<G>();
  }
  if constexpr (OL) {  // outlier slot `lane`: its merged value (same weights), to its channel in the original basis
    float t = 0.0f;
    for (int s0 = 0; s0 < splits; s0 += 8) {
      float xo[8], wv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = s0 + u;
        xo[u] = 0.0f; wv[u] = 0.0f;
        if (j < splits) {
          const size_t ri = (base + slot_of(j)) * a.heads_per_cta + hh;
          const float2 ml = *reinterpret_cast<const float2*>(a.ws_ml + ri * 2);
          wv[u] = ml.y > 0.0f ? fast_exp2(ml.x - Mg) : 0.0f;
          xo[u] = a.ws_acco[ri * 32 + lane];
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) t += wv[u] != 0.0f ? wv[u] * xo[u] : 0.0f;
    }
    const int ch = a.oidx[(size_t)kvh * 32 + lane];
    const int prev = __shfl_up_sync(0xffffffffu, ch, 1);
    const bool ok = ch >= 0 && ch < D && (lane == 0 || prev < ch);
    const float val = t * inv;
#pragma unroll 4
    for (int sl = 0; sl < 32; ++sl) {
      const int cs = __shfl_sync(0xffffffffu, ok ? ch : -1, sl);
      const float vs = __shfl_sync(0xffffffffu, val, sl);
#pragma unroll
      for (int j = 0; j < E; ++j)
        if (fwht_channel<D, G>(lane, j) == cs) x[j] += vs;
    }
  }
#pragma unroll
  for (int j = 0; j < E; ++j) {
    const size_t e = (size_t)row * D + fwht_channel<D, G>(lane, j);
    if (a.out_dtype == KVQ_F32) static_cast<float*>(a.out)[e] = x[j];
    else if (a.out_dtype == KVQ_BF16) static_cast<__nv_bfloat16*>(a.out)[e] = __float2bfloat16_rn(x[j]);
    else static_cast<__half*>(a.out)[e] = __float2half_rn(x[j]);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

CUtensorMapSwizzle swizzle_for(int w) {
  return w == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : (w == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

// rows x row_bytes plane of `elem` sized elements, seen as three dimensions (elements
// within a box column of box_w bytes, row, box column) so that one copy of box_rows
// rows brings every column: shared memory [column][box_rows rows][box_w bytes].
bool make_map(CUtensorMap* m, void* base, CUtensorMapDataType dt, int elem, long long rows, int row_bytes,
              int box_w_bytes, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int cols = row_bytes / box_w_bytes;
  cuuint64_t dims[3] = {cuuint64_t(box_w_bytes / elem), cuuint64_t(rows), cuuint64_t(cols)};
  cuuint64_t strides[2] = {cuuint64_t(row_bytes), cuuint64_t(box_w_bytes)};
  cuuint32_t box[3] = {cuuint32_t(box_w_bytes / elem), cuuint32_t(box_rows), cuuint32_t(cols)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, dt, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(box_w_bytes),
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int KT, int VT, bool OL>
cudaError_t run_decode(const kvq_cache& c, Rot rot, const DecodePlan& plan, const void* q, int q_dtype,
                       int n_q_heads, float scale, void* out, int out_dtype, void* ws, cudaStream_t st,
                       const FusedAppend* fa) {
  using Cf = Cfg<D, KT, VT, OL>;
  Params p{};
  p.k_d = static_cast<const uint8_t*>(c.k_d); p.v_d = static_cast<const uint8_t*>(c.v_d);
  p.k_qh = static_cast<const uint32_t*>(c.k_qh); p.v_qh = static_cast<const uint32_t*>(c.v_qh);
  p.seq_len = c.seq_len; p.status = c.status; p.q = q;
  // workspace: partition header, then acc [plane][slot][head][D], (m, l) [plane][slot][head][2],
  // outlier acc [plane][slot][head][32]
  const size_t nrow = (size_t)plan.planes * plan.slots * plan.heads_per_cta;
  p.ws_hdr = static_cast<long long*>(ws);
  p.ws_acc = reinterpret_cast<float*>(static_cast<char*>(ws) + plan.hdr_bytes);
  p.ws_ml = p.ws_acc + nrow * D;
  p.ws_acco = OL ? p.ws_ml + nrow * 2 : nullptr;
  p.n_kv_heads = c.n_kv_heads; p.max_ctx = c.max_ctx; p.tail_len = c.tail_len;
  p.q_dtype = q_dtype; p.n_q_heads = n_q_heads; p.group = n_q_heads / c.n_kv_heads;
  p.heads_per_cta = plan.heads_per_cta; p.head_groups = plan.head_groups;
  p.rot_k = rot.k;
  p.rot_v = rot.v;
  p.fused = fa ? 1 : 0;
  if (fa) p.fa = *fa;
  p.cache = c;
  p.rows = row_map(c);
  p.scale_log2 = scale * kLog2e;
  p.batch = c.batch;
  p.pieces = fa ? plan.pieces_fused : plan.pieces;
  p.slots = plan.slots;
  p.cost_body = plan.cost_body; p.cost_tail = plan.cost_tail; p.cost_min = plan.cost_min;
  p.cost_gap = plan.cost_gap;
  p.sms = plan.sms;
  const bool wave = fa ? plan.weighted_fused : plan.weighted;
  for (int k = 0; k < 3; ++k) p.wt[k] = wave ? plan.slot_weight[k] : 0;

  alignas(64) CUtensorMap mk, mv, mkt, mvt;
  memset(&mk, 0, sizeof(mk)); memset(&mv, 0, sizeof(mv)); memset(&mkt, 0, sizeof(mkt)); memset(&mvt, 0, sizeof(mvt));
  const long long rows = body_rows(c);
  if (!make_map(&mk, c.k_qs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, Cf::rowK, Cf::WK, Cf::RB)) return cudaErrorInvalidValue;
  if (!make_map(&mv, c.v_qs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, Cf::rowV, Cf::WV, Cf::RB)) return cudaErrorInvalidValue;
  if (c.tail_len > 0) {
    const long long trows = (long long)c.batch * c.n_kv_heads * c.tail_len;
    if (!make_map(&mkt, c.k_tail, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, trows, 2 * D, Cf::WT, Cf::TT) ||
        !make_map(&mvt, c.v_tail, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, trows, 2 * D, Cf::WT, Cf::TT))
      return cudaErrorInvalidValue;
  }
  auto kern = decode_split_kernel<D, KT, VT, OL>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), Cf::smem);
  if (e != cudaSuccess) return e;
  dim3 grid(plan.planes, fa ? c.batch + plan.pieces_fused : plan.pieces);
  kern<<<grid, kThreads, Cf::smem, st>>>(p, mk, mv, mkt, mvt);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CombineArgs ca{};
  ca.ws_acc = p.ws_acc; ca.ws_ml = p.ws_ml; ca.ws_acco = p.ws_acco; ca.hdr = p.ws_hdr;
  ca.slots = plan.slots; ca.heads_per_cta = plan.heads_per_cta; ca.head_groups = plan.head_groups;
  ca.group = p.group; ca.batch = c.batch; ca.tail_len = c.tail_len; ca.fused = p.fused; ca.rot_v = rot.v;
  ca.out_dtype = out_dtype; ca.n_q_heads = n_q_heads;
  ca.cost_body = plan.cost_body; ca.cost_tail = plan.cost_tail; ca.cost_min = plan.cost_min;
  ca.cost_gap = plan.cost_gap;
  ca.pieces = p.pieces; ca.planes = plan.planes; ca.sms = plan.sms;
  for (int k = 0; k < 3; ++k) ca.wt[k] = p.wt[k];
  ca.out = out; ca.seq_len = c.seq_len; ca.oidx = c.outlier_idx;
  // a row merges many partials when the batch is small: 512 threads keep them all in flight;
  // with many rows, 256-thread CTAs fit twice as many rows on the GPU at once
  const bool wide = (long long)c.batch * n_q_heads <= 2LL * plan.sms;
  auto ckern = wide ? decode_combine_kernel<D, OL, 512> : decode_combine_kernel<D, OL, 256>;
  // programmatic dependent launch: the merge grid's launch overlaps the split grid's end
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.batch * n_q_heads);
  cfg.blockDim = dim3(wide ? 512 : 256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ckern, ca);
}

template <int D>
cudaError_t run_decode_d(const kvq_cache& c, Rot rot, const DecodePlan& plan, const void* q, int q_dtype, int nq,
                         float scale, void* out, int out_dtype, void* ws, cudaStream_t st, const FusedAppend* fa) {
#define KVQ_CASE(KT, VT, OL)                                                                          \
  if (c.k_type == KT && c.v_type == VT)                                                               \
    return run_decode<D, KT, VT, OL>(c, rot, plan, q, q_dtype, nq, scale, out, out_dtype, ws, st, fa);
#define KVQ_CASES_K(KT) KVQ_CASE(KT, KVQ_TYPE_Q4_0, false) KVQ_CASE(KT, KVQ_TYPE_Q5_0, false)         \
                        KVQ_CASE(KT, KVQ_TYPE_Q8_0, false) KVQ_CASE(KT, KVQ_TYPE_Q4_1, false)         \
                        KVQ_CASE(KT, KVQ_TYPE_Q5_1, false)
#define KVQ_CASES_K_OL(KT) KVQ_CASE(KT, KVQ_TYPE_Q4_0, true) KVQ_CASE(KT, KVQ_TYPE_Q5_0, true) \
                           KVQ_CASE(KT, KVQ_TYPE_Q8_0, true)
  if constexpr (D == 64 || D == 128 || D == 256) {
    if (c.n_outlier) {  // outlier channels: the q4_0 / q5_0 / q8_0 pairs
      KVQ_CASES_K_OL(KVQ_TYPE_Q4_0) KVQ_CASES_K_OL(KVQ_TYPE_Q5_0) KVQ_CASES_K_OL(KVQ_TYPE_Q8_0)
      return cudaErrorInvalidValue;
    }
  } else {
    if (c.n_outlier) return cudaErrorInvalidValue;
  }
  KVQ_CASES_K(KVQ_TYPE_Q4_0) KVQ_CASES_K(KVQ_TYPE_Q5_0) KVQ_CASES_K(KVQ_TYPE_Q8_0)
  KVQ_CASES_K(KVQ_TYPE_Q4_1) KVQ_CASES_K(KVQ_TYPE_Q5_1)
#undef KVQ_CASES_K_OL
#undef KVQ_CASES_K
#undef KVQ_CASE
  return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace kvq
