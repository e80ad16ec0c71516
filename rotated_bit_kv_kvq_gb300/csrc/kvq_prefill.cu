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
// Two kernels per call:
//
// stage_kernel   one CTA per 64-key tile of a (sequence, KV head): every key
//                the prompt can see is dequantized ONCE (code * scale, or the
//                bf16 tail value), scaled by 2^-8 and split into exact fp16
//                hi + lo parts, laid out exactly as the tensor cores read them
//                (K: rows = keys; V^T: rows = channels; 128-byte swizzle) and
//                written to the workspace with one bulk copy.  Keys past the
//                sequence are zeros.
// attn_kernel    one CTA per 128 query rows (positions x the query heads of
//                one KV head), warp-specialized:
//                  warp 8   streams K and V tiles (1-D bulk copies, two-slot
//                           rings each, released by the MMAs that read them);
//                  warp 9   issues S_j = Q K_j^T into one of two TMEM score
//                           buffers, warp 10 issues O += P_j V_j (two issuing
//                           warps keep the tensor pipe fed: one thread alone
//                           issues an MMA only every ~75 cycles); each is
//                           three fp16 products (hi.hi + hi.lo + lo.hi: ~22
//                           bits, so the result matches fp32 arithmetic);
//                  warps 0-7 (two warpgroups; row = TMEM lane, warpgroup h
//                           owns keys 32h..32h+31 of every tile and output
//                           channels h*D/2..) prepare Q (rotate, scale,
//                           split), run the online softmax on S_j while the
//                           tensor cores work on PV_{j-1} and S_{j+1} (both
//                           halves take the row maximum over all 64 scores,
//                           so they agree without exchanging it), rescale O
//                           in TMEM when a row's maximum grew by more than
//                           2^7, write P_j, and finish with O / l, the
//                           inverse rotation and the output cast.
// Every wait is bounded: a wait that gives up sets the status word's timeout
// bit and a shared abort flag that ends the other roles' loops; the CTA then
// lets its copies and MMAs in flight finish (bounded) before it releases TMEM.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tcgen05.cuh"

namespace kvq {
namespace {

constexpr int kPM = 128;               // query rows per CTA (UMMA M)
constexpr int kPN = 64;                // keys per tile
constexpr int kSoftmax = 256;          // two warpgroups, each half of a row's 64 scores
constexpr int kAttnThreads = kSoftmax + 96;  // + warp 8 producer, 9 S issue, 10 PV issue
constexpr int kStageThreads = 256;
constexpr long long kPWait = 2000000000LL;  // ~1 s at 2 GHz per wait
constexpr float kPLog2e = 1.4426950408889634f;
constexpr float kInvScale = 0.00390625f;    // staged K/V values are x * 2^-8
constexpr float kLazyRescale = 7.0f;        // log2 units: P*256 stays <= 2^15 (fp16 max 65504)

template <int D>
struct PL {
  static constexpr int KA = D / 64;             // 128-byte atoms along head_dim
  static constexpr int kt = KA * kPN * 128;     // K tile, hi or lo (stored [KA][hi, lo][64 keys][128 B])
  static constexpr int vt = D * 128;            // V^T tile, hi or lo: [D channels][64 keys * 2 B]
  static constexpr int tile = 2 * kt + 2 * vt;  // workspace bytes per tile: K hi, K lo, V hi, V lo
  static constexpr int q = KA * kPM * 128;      // Q, hi or lo: [KA][128 rows][128 B]
  static constexpr int off_qh = 0, off_ql = q;
  static constexpr int off_k = 2 * q;           // two slots of [hi | lo]
  static constexpr int off_v = off_k + 4 * kt;  // two slots of [hi | lo]
  static constexpr int off_xl = off_v + 4 * vt;  // [2][128] floats: the halves' row sums
  static constexpr int off_xm = off_xl + 2 * kPM * 4;  // [2 tiles][2 halves][128] (max, tile) words
  static constexpr int off_bar = off_xm + 2 * 2 * kPM * 8;
  static constexpr int smem = off_bar + 256 + 1024;
  static constexpr int stage_stride = D + 4;    // epilogue fp32 rows (reuse Q and K slots), 16-byte rows
  static_assert(kPM * stage_stride * 4 <= off_v, "epilogue staging must fit below the V slots");
  static constexpr uint32_t idesc_qk = tc::idesc_f16_f32(kPM, kPN);        // Q_lo . K_hi
  static constexpr uint32_t idesc_qk2 = tc::idesc_f16_f32(kPM, 2 * kPN);   // Q_hi . [K_hi; K_lo]
  static constexpr uint32_t idesc_pv = tc::idesc_f16_f32(kPM, D);
  // TMEM: two score buffers of 128 columns ([hi.hi + lo.hi | hi.lo] of 64 keys) at 0
  // and 128; two P buffers of 64 columns (P_hi: 32 columns of fp16 pairs, then P_lo)
  // at 256 and 320, the A operand of P V; O over D columns at 384
  static constexpr uint32_t tmem_cols = 512;
  static constexpr uint32_t s_cols = 2 * kPN;
  static constexpr uint32_t p_col = 256;
  static constexpr uint32_t o_col = 384;
  static_assert(o_col + D <= tmem_cols, "TMEM columns");
};
static_assert(PL<128>::smem <= 232448, "prefill shared memory over the per-CTA limit");

struct SParams {
  const uint8_t* k_qs; const uint8_t* v_qs;
  const uint8_t* k_d; const uint8_t* v_d;   // fp16 d per block, or (d, lo) pairs for q4_1 / q5_1
  const uint32_t* k_qh; const uint32_t* v_qh;
  const uint16_t* k_tail; const uint16_t* v_tail;
  const int32_t* seq_len; const int32_t* q_pos0;
  int n_kv_heads, max_ctx, tail_len, k_type, v_type, n_tokens, causal, max_tiles;
  uint8_t* ws;
  RowMap rows;   // body row of (sequence, KV head, position): contiguous or paged
  uint32_t* status;
  // outlier channels (n_outlier = 32): unrotated q8_0 slots, added back rotated like the rest
  int n_outlier, rot_k, rot_v;
  const int32_t* oidx;
  const uint8_t* outl;   // [rows / 16][kOutlTile]: K codes, V codes, K scales, V scales of 16 rows
};

struct AParams {
  const uint8_t* ws;
  const int32_t* seq_len; uint32_t* status;
  int n_kv_heads, max_tiles;
  const void* q; void* out;
  int q_dtype, out_dtype, n_q_heads, n_tokens, group, ppt, ntiles;
  const int32_t* q_pos0;
  int causal, rot_k, rot_v;
  float scale_log2;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Keys of sequence b that any of the call's queries can see: [0, kv_end).
__device__ __forceinline__ int visible_keys(int n, int p0, int n_queries, int causal) {
  if (p0 < 0) return 0;
  return causal ? min(n, p0 + n_queries) : n;
}

// fp16 hi / lo split of two values (hi = RN(x), lo = RN(x - hi); exact when x has <= 22 bits)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_h2(a, b);
  const float2 f = __half22float2(u32_as_h2(hi));
  lo = pack_h2(a - f.x, b - f.y);
}

// The raw stored words behind 8 values (channels 8*ch .. 8*ch+7) of one key:
// 16 bytes of bf16 tail values, or 8 bytes of codes with the block header
// (fp16 d, or the (d, lo) pair) and the q5_x high-bit word.  Loaded first for
// every chunk a thread handles, so that the loads overlap; decoded after.
struct Raw8 {
  uint4 w;
  uint32_t hdr, qh;
};

template <int D>
__device__ __forceinline__ Raw8 fetch8(const SParams& p, bool is_v, int qt, bool valid, bool tail, size_t body_row,
                                       size_t tail_row, int ch) {
  constexpr int NB = D / 32;
  Raw8 r{make_uint4(0u, 0u, 0u, 0u), 0u, 0u};
  if (!valid) return r;
  if (tail) {
    r.w = *reinterpret_cast<const uint4*>((is_v ? p.v_tail : p.k_tail) + tail_row * D + ch * 8);
    return r;
  }
  const int c0 = ch * 8, blk = c0 / 32, w = c0 % 32;
  const uint8_t* hd = (is_v ? p.v_d : p.k_d) + (body_row * NB + blk) * (type_has_min(qt) ? 4 : 2);
  r.hdr = type_has_min(qt) ? *reinterpret_cast<const uint32_t*>(hd) : uint32_t(*reinterpret_cast<const uint16_t*>(hd));
  const uint8_t* qs = is_v ? p.v_qs : p.k_qs;
  const uint2 a = qt == KVQ_TYPE_Q8_0 ? *reinterpret_cast<const uint2*>(qs + body_row * D + c0)
                                      : *reinterpret_cast<const uint2*>(qs + body_row * (D / 2) + blk * 16 + (w & 15));
  r.w.x = a.x;
  r.w.y = a.y;
  if (type_has_qh(qt)) r.qh = qh_get(is_v ? p.v_qh : p.k_qh, !is_v, body_row, NB, blk);
  return r;
}

// 8 stored values (channels 8*ch .. 8*ch+7) of one key, times 2^-8, from their raw words.
__device__ __forceinline__ void decode8(const Raw8& r, int qt, bool valid, bool tail, int ch, float (&x)[8]) {
  if (!valid) {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.0f;
    return;
  }
  if (tail) {
    const uint32_t ww[4] = {r.w.x, r.w.y, r.w.z, r.w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(ww[e] << 16) * kInvScale;
      x[2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u) * kInvScale;
    }
    return;
  }
  const int w = (ch * 8) % 32;
  const float sc = __half2float(__ushort_as_half(uint16_t(r.hdr & 0xFFFFu))) * kInvScale;
  const float mn = type_has_min(qt) ? __half2float(__ushort_as_half(uint16_t(r.hdr >> 16))) * kInvScale : 0.0f;
  if (qt == KVQ_TYPE_Q8_0) {
#pragma unroll
    for (int e = 0; e < 8; ++e)  // stored offset binary: code + 128
      x[e] = float(int(((e < 4 ? r.w.x : r.w.y) >> (8 * (e & 3))) & 0xFFu) - 128) * sc;
  } else {
    // byte i of a block holds element i (low nibble) and element i + 16 (high nibble)
    const int shift = w < 16 ? 0 : 4;
    const int off = type_code_offset(qt);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t byte = ((e < 4 ? r.w.x : r.w.y) >> (8 * (e & 3))) & 0xFFu;
      const int code = int((byte >> shift) & 15u) | int(((r.qh >> (w + e)) & 1u) << 4);
      x[e] = __fadd_rn(__fmul_rn(float(code - off), sc), mn);  // x = code*d + lo
    }
  }
}

// x[e] += src[e], e < 8 (src 16-byte aligned, shared memory)
__device__ __forceinline__ void add8(const float* src, float (&x)[8]) {
  const float4 a = reinterpret_cast<const float4*>(src)[0], c = reinterpret_cast<const float4*>(src)[1];
  x[0] += a.x; x[1] += a.y; x[2] += a.z; x[3] += a.w;
  x[4] += c.x; x[5] += c.y; x[6] += c.z; x[7] += c.w;
}

// ---------------------------------------------------------------------------
// stage_kernel: one 64-key tile of one (sequence, KV head) -> workspace
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kStageThreads, 3) stage_kernel(SParams p) {
  using L = PL<D>;
  constexpr int NCH = D / 8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int j = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int n = min(max(p.seq_len[b], 0), p.max_ctx);  // reads stay inside the planes
  const int p0 = p.q_pos0 ? p.q_pos0[b] : n - p.n_tokens;
  if (j * kPN >= visible_keys(n, p0, p.n_tokens, p.causal)) return;
  const int T = p.tail_len;
  const size_t bh = (size_t)b * p.n_kv_heads + kvh;
  const int key = threadIdx.x & (kPN - 1);   // a warp covers 32 consecutive keys
  const int t = j * kPN + key;
  bool valid = t < n;
  const bool tail = valid && T > 0 && t >= n - T;
  long long brow = 0;
  if (valid && !tail) {
    brow = kvq::body_row(p.rows, b, kvh, t);
    if (brow < 0) {  // page id outside the pool: the key reads as empty
      atomicOr(p.status, KVQ_DEV_ERR_PAGE);
      valid = false;
      brow = 0;
    }
  }
  const size_t body_row = size_t(brow);
  const size_t tail_row = tail ? bh * T + t % T : 0;
  // Outlier channels: per body key, the 32 dequantized slot values (x 2^-8) are
  // scattered to their channels and rotated like the rest (warp FWHT), for K
  // and V, into [2][64 keys][D] fp32 after the tile in shared memory; the
  // loop below adds them to the dequantized rest.
  float* obuf = reinterpret_cast<float*>(sm + L::tile);
  const bool ol = p.n_outlier != 0;
  if (ol) {
    for (int i = threadIdx.x; i < 2 * kPN * D / 4; i += kStageThreads)
      reinterpret_cast<float4*>(obuf)[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int chn = p.oidx[(size_t)kvh * 32 + lane];
    const int prev = __shfl_up_sync(0xffffffffu, chn, 1);
    const bool ok = chn >= 0 && chn < D && (lane == 0 || prev < chn);
    if (__ballot_sync(0xffffffffu, !ok) && lane == 0) atomicOr(p.status, KVQ_DEV_ERR_OUTLIER);
    for (int kk = warp; kk < kPN; kk += kStageThreads / 32) {
      const int tt = j * kPN + kk;
      if (tt >= n || (T > 0 && tt >= n - T)) continue;  // past the end, or a tail key (whole vector in bf16)
      const long long br = kvq::body_row(p.rows, b, kvh, tt);
      if (br < 0) continue;
      const uint8_t* grp = p.outl + (size_t)(br / 16) * kOutlTile;
      auto part = [&](int which, int rot, float* row) {
        const float dd = __half2float(reinterpret_cast<const __half*>(grp + 1024 + which * 32)[br % 16]);
        if (ok) row[chn] = float(reinterpret_cast<const int8_t*>(grp + which * 512 + (br % 16) * 32)[lane]) * dd * kInvScale;
        __syncwarp();
        if (rot) {
          constexpr int P = D / 32;
          float v[P];
#pragma unroll
          for (int e = 0; e < P; ++e) v[e] = row[lane * P + e];
          warp_fwht<D, D>(v, lane);
#pragma unroll
          for (int e = 0; e < P; ++e) row[lane * P + e] = v[e] * inv_sqrt_group<D>();
          __syncwarp();
        }
      };
      part(0, p.rot_k, obuf + (size_t)kk * D);
      part(1, p.rot_v, obuf + (size_t)(kPN + kk) * D);
    }
    __syncthreads();
  }
  // every chunk's raw words first (K and V), then decode, split and store
  constexpr int IT = NCH / (kStageThreads / kPN);  // chunks per thread
  static_assert(NCH % (kStageThreads / kPN) == 0, "chunks per thread");
  Raw8 rk[IT], rv[IT];
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int ch = threadIdx.x / kPN + it * (kStageThreads / kPN);
    rk[it] = fetch8<D>(p, false, p.k_type, valid, tail, body_row, tail_row, ch);
    rv[it] = fetch8<D>(p, true, p.v_type, valid, tail, body_row, tail_row, ch);
  }
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int ch = threadIdx.x / kPN + it * (kStageThreads / kPN);
    // K: row = key, 16-byte chunks of 8 channels
    float x[8];
    decode8(rk[it], p.k_type, valid, tail, ch, x);
    if (ol) add8(obuf + (size_t)key * D + ch * 8, x);
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split2(x[2 * e], x[2 * e + 1], h[e], l[e]);
    // per 128-byte atom: 64 hi rows then 64 lo rows, so one N=128 operand holds both
    const uint32_t off = (ch / 8) * (2 * kPN * 128) + tc::sw128_chunk(key, ch % 8);
    *reinterpret_cast<uint4*>(sm + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(sm + kPN * 128 + off) = make_uint4(l[0], l[1], l[2], l[3]);
    // V^T: row = channel, this key's 2-byte element in it
    decode8(rv[it], p.v_type, valid, tail, ch, x);
    if (ol) add8(obuf + (size_t)(kPN + key) * D + ch * 8, x);
#pragma unroll
    for (int e = 0; e < 4; ++e) split2(x[2 * e], x[2 * e + 1], h[e], l[e]);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t o = tc::sw128_chunk(ch * 8 + e, key / 8) + (key % 8) * 2;
      *reinterpret_cast<uint16_t*>(sm + 2 * L::kt + o) = uint16_t(h[e / 2] >> (16 * (e & 1)));
      *reinterpret_cast<uint16_t*>(sm + 2 * L::kt + L::vt + o) = uint16_t(l[e / 2] >> (16 * (e & 1)));
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    bulk_s2g(p.ws + (bh * p.max_tiles + j) * (size_t)L::tile, sm, L::tile);
    bulk_commit();
    bulk_wait_all();
  }
}

// ---------------------------------------------------------------------------
// attn_kernel
// ---------------------------------------------------------------------------
struct Sync {
  uint64_t kfull[2], kempty[2], vfull[2], vempty[2], sfull[2], sfree[2];
  // One barrier per P buffer for P-ready and PV-done: the softmax may finish P_{j+1}
  // before the PV issuer has observed P_j, and a single barrier would then pass two
  // phases under the waiter (same parity: the wait would never see its phase end).
  uint64_t pfull[2], odone[2], qready, fin[2];
  uint32_t tmem;
  int abort;
};

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool role_wait(uint64_t* bar, uint32_t parity, Sync* sy, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity, 20000u)) {
    if (*reinterpret_cast<volatile int*>(&sy->abort)) return false;
    if (clock64() - t0 > kPWait) {
      *reinterpret_cast<volatile int*>(&sy->abort) = 1;
      atomicOr(status, KVQ_DEV_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Hint: bring `bytes` (a multiple of 16) at the 16-byte aligned `src` into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(AParams p) {
  using L = PL<D>;
  constexpr int G = D;  // head_dim 64 and 128 rotate as one Hadamard group
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  Sync* sy = reinterpret_cast<Sync*>(sm + L::off_bar);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = p.ntiles - 1 - blockIdx.x;  // the longest (latest) query tiles first
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int g = p.group;
  // Warps 0-7 start loading their query rows before any set-up, so that the
  // load latency overlaps the TMEM allocation and barrier initialisation.  A
  // row is held by QR = D/32 consecutive lanes, 32 consecutive channels each
  // (one aligned 64- or 128-byte run: q is 16-byte aligned); a warp's 16 rows
  // take QPASS passes of 32/QR rows.
  constexpr int QR = D / 32, QRP = 32 / QR, QPASS = (kPM / 8) / QRP;
  const int qsub = lane % QR;
  uint32_t qraw[QPASS][32];
  const bool qwide = p.q_dtype == KVQ_F32;
  if (warp < kSoftmax / 32) {
#pragma unroll
    for (int pp = 0; pp < QPASS; ++pp) {
      const int r = warp * (kPM / 8) + pp * QRP + lane / QR;
      const int rli = r / g, rhh = r % g, rqi = tile * p.ppt + rli;
      const bool ok = rli < p.ppt && rqi < p.n_tokens;
      const size_t e = (((size_t)b * p.n_tokens + (ok ? rqi : 0)) * p.n_q_heads + kvh * g + rhh) * D + qsub * 32;
      const uint4* src = qwide ? reinterpret_cast<const uint4*>(static_cast<const float*>(p.q) + e)
                               : reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + e);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (t >= 4 && !qwide) break;  // 16-bit rows: 64 bytes
        const uint4 w = src[t];
        qraw[pp][4 * t] = w.x; qraw[pp][4 * t + 1] = w.y; qraw[pp][4 * t + 2] = w.z; qraw[pp][4 * t + 3] = w.w;
      }
    }
  }

  const int n = min(max(p.seq_len[b], 0), p.max_tiles * kPN);  // as the stage kernel
  const int p0 = p.q_pos0 ? p.q_pos0[b] : n - p.n_tokens;
  const int last_q = min(p.n_tokens, (tile + 1) * p.ppt) - 1;
  const int kv_end = visible_keys(n, p0, last_q + 1, p.causal);
  const int nkv = (kv_end + kPN - 1) / kPN;
  if (p0 < 0 && tid == 0 && blockIdx.x == 0 && kvh == 0) atomicOr(p.status, KVQ_DEV_ERR_PREFILL_RANGE);

  if (warp == 0) {
    tc::tmem_alloc(&sy->tmem, L::tmem_cols);
    tc::tmem_relinquish();
  }
  if (tid == kSoftmax) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sy->kfull[i], 1); mbar_init(&sy->kempty[i], 1);
      mbar_init(&sy->vfull[i], 1); mbar_init(&sy->vempty[i], 1);
      mbar_init(&sy->sfull[i], 1); mbar_init(&sy->sfree[i], kSoftmax);
    }
    mbar_init(&sy->pfull[0], kSoftmax);
    mbar_init(&sy->pfull[1], kSoftmax);
    mbar_init(&sy->odone[0], 1);
    mbar_init(&sy->odone[1], 1);
    mbar_init(&sy->qready, kSoftmax);
    mbar_init(&sy->fin[0], 1);
    mbar_init(&sy->fin[1], 1);
    sy->abort = 0;
    fence_barrier_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sy->tmem;

  if (warp == kSoftmax / 32) {
    // ---- L2 prefetch of the query rows of the CTA one SM-count further in the
    // launch order (about the one that takes over an SM after this wave) -------
    {
      uint32_t nsm;
      asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
      const uint32_t nx = gridDim.x, ny = gridDim.y;
      const uint32_t lin = blockIdx.x + nx * (blockIdx.y + ny * blockIdx.z) + nsm;
      if (lin < nx * ny * gridDim.z) {
        const int t2 = p.ntiles - 1 - int(lin % nx), h2 = int((lin / nx) % ny), b2 = int(lin / (nx * ny));
        const size_t esz = qwide ? 4 : 2;
        for (int i = lane; i < p.ppt; i += 32) {
          const int qi = t2 * p.ppt + i;
          if (qi >= p.n_tokens) break;
          const size_t e = (((size_t)b2 * p.n_tokens + qi) * p.n_q_heads + (size_t)h2 * g) * D;
          bulk_prefetch_l2(static_cast<const uint8_t*>(p.q) + e * esz, uint32_t(g * D * esz));
        }
      }
    }
    // ---- producer: K and V tiles of this (sequence, KV head) ----------------
    if (lane == 0 && nkv > 0) {
      const uint8_t* base = p.ws + ((size_t)b * p.n_kv_heads + kvh) * p.max_tiles * (size_t)L::tile;
      int kiss = 0, viss = 0;
      for (int j = 0; j < nkv; ++j) {
        const int s = j & 1;
        const uint32_t u = j >> 1;
        const uint8_t* src = base + (size_t)j * L::tile;
        if (u > 0 && !role_wait(&sy->kempty[s], (u - 1) & 1, sy, p.status)) break;
        mbar_arrive_expect_tx(&sy->kfull[s], 2 * L::kt);
        bulk_g2s(sm + L::off_k + s * 2 * L::kt, src, 2 * L::kt, &sy->kfull[s]);
        ++kiss;
        if (u > 0 && !role_wait(&sy->vempty[s], (u - 1) & 1, sy, p.status)) break;
        mbar_arrive_expect_tx(&sy->vfull[s], 2 * L::vt);
        bulk_g2s(sm + L::off_v + s * 2 * L::vt, src + 2 * L::kt, 2 * L::vt, &sy->vfull[s]);
        ++viss;
      }
      // copies still landing (abort path): let them finish before the CTA can exit
      for (int j = max(0, kiss - 2); j < kiss; ++j) mbar_wait_bounded(&sy->kfull[j & 1], (j >> 1) & 1, kPWait);
      for (int j = max(0, viss - 2); j < viss; ++j) mbar_wait_bounded(&sy->vfull[j & 1], (j >> 1) & 1, kPWait);
    }
    return;
  }

  // Shared-memory descriptors: the K-step and slot offsets are added to these
  // bases (the 14-bit start-address field cannot overflow inside the buffer).
  const uint32_t sb = smem_u32(sm);
  if (warp == kSoftmax / 32 + 1) {
    // ---- S_j = Q K_j^T issue (one thread) ----------------------------------
    if (lane == 0 && nkv > 0) {
      const uint64_t dqh = tc::sdesc_sw128(sb + L::off_qh), dql = tc::sdesc_sw128(sb + L::off_ql);
      const uint64_t dk = tc::sdesc_sw128(sb + L::off_k);
      bool ok = role_wait(&sy->qready, 0, sy, p.status);
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j & 1;
        const uint32_t u = j >> 1;
        ok = role_wait(&sy->kfull[s], u & 1, sy, p.status) &&
             (u == 0 || role_wait(&sy->sfree[s], (u - 1) & 1, sy, p.status));
        if (!ok) break;
        tc::fence_after_sync();
        const uint64_t kb = dk + ((s * 2 * L::kt) >> 4);
        const uint32_t d = tmem + s * L::s_cols;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t qo = ((ks / 4) * (kPM * 128) + (ks % 4) * 32) >> 4;
          const uint32_t ko = ((ks / 4) * (2 * kPN * 128) + (ks % 4) * 32) >> 4;
          tc::mma_f16(d, dqh + qo, kb + ko, L::idesc_qk2, ks > 0 ? 1u : 0u);  // [hi.hi | hi.lo]
          tc::mma_f16(d, dql + qo, kb + ko, L::idesc_qk, 1u);                 // + lo.hi
        }
        tc::commit(&sy->sfull[s]);
        tc::commit(&sy->kempty[s]);
      }
      tc::commit(&sy->fin[0]);  // arrives once every MMA issued above has completed
    }
    return;
  }

  if (warp == kSoftmax / 32 + 2) {
    // ---- O += P_j V_j issue (one thread; runs beside the S issue) ------------
    if (lane == 0 && nkv > 0) {
      const uint64_t dv = tc::sdesc_sw128(sb + L::off_v);
      bool ok = true;
      for (int j = 0; ok && j < nkv; ++j) {
        ok = role_wait(&sy->pfull[j & 1], (j >> 1) & 1, sy, p.status) &&
             role_wait(&sy->vfull[j & 1], (j >> 1) & 1, sy, p.status);
        if (!ok) break;
        tc::fence_after_sync();
        const uint64_t vh = dv + (((j & 1) * 2 * L::vt) >> 4), vl = vh + (L::vt >> 4);
        const uint32_t ph = tmem + L::p_col + (j & 1) * kPN, pl = ph + kPN / 2;
#pragma unroll
        for (int ks = 0; ks < kPN / 16; ++ks) {
          const uint32_t o = (ks * 32) >> 4;
          tc::mma_f16_ts(tmem + L::o_col, ph + ks * 8, vh + o, L::idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
          tc::mma_f16_ts(tmem + L::o_col, ph + ks * 8, vl + o, L::idesc_pv, 1u);
          tc::mma_f16_ts(tmem + L::o_col, pl + ks * 8, vh + o, L::idesc_pv, 1u);
        }
        tc::commit(&sy->odone[j & 1]);
        tc::commit(&sy->vempty[j & 1]);
      }
      tc::commit(&sy->fin[1]);
    }
    return;
  }

  // ---- warps 0-7: Q rows (loaded above): rotate, scale, split into hi / lo tiles
  {
    float sc = p.scale_log2;
    if (p.rot_k) sc *= inv_sqrt_group<G>();
#pragma unroll
    for (int pp = 0; pp < QPASS; ++pp) {
      const int r = warp * (kPM / 8) + pp * QRP + lane / QR;
      const int rli = r / g, rqi = tile * p.ppt + rli;
      const bool ok = rli < p.ppt && rqi < p.n_tokens;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t w = qraw[pp][i / 2];
        const uint32_t hb = (i & 1) ? (w >> 16) : (w & 0xFFFFu);
        float x;
        if (qwide) x = __uint_as_float(qraw[pp][i]);
        else if (p.q_dtype == KVQ_BF16) x = bf16_bits_to_f32(hb);
        else x = __half2float(__ushort_as_half(uint16_t(hb)));
        v[i] = ok ? x : 0.0f;
      }
      if (p.rot_k) lane_fwht<D / 32>(v, lane, 0xffffffffu);  // a row on D/32 lanes
      // the lane's 32 channels = four 16-byte chunks of 8 fp16 in each of the hi / lo tiles
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split2(v[8 * t + 2 * e] * sc, v[8 * t + 2 * e + 1] * sc, hi[e], lo[e]);
        const int c = qsub * 32 + 8 * t;
        const uint32_t off = (c / 64) * (kPM * 128) + tc::sw128_chunk(r, (c % 64) / 8);
        *reinterpret_cast<uint4*>(sm + L::off_qh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(sm + L::off_ql + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
  }
  fence_proxy_async_smem();
  mbar_arrive(&sy->qready);

  // ---- softmax: row = TMEM lane (tid % 128), half h of the 64 keys ---------
  const int row = tid & (kPM - 1), h = tid / kPM;
  // The two halves of a row swap their maxima through shared memory: slot [j & 1][h][row]
  // holds (maximum, tile j), written by half h, polled (bounded) by the other half.
  // A slot is rewritten for tile j + 2 only after its writer has seen the other
  // half's tile j + 1 value, which comes after that half read tile j's.
  unsigned long long* xm = reinterpret_cast<unsigned long long*>(sm + L::off_xm);
  xm[(0 * 2 + h) * kPM + row] = ~0ull;
  xm[(1 * 2 + h) * kPM + row] = ~0ull;
  named_sync(1, kSoftmax);
  const int li = row / g;
  const int qi = tile * p.ppt + li;
  const bool row_ok = li < p.ppt && qi < p.n_tokens && p0 >= 0;
  const int kv_end_row = row_ok ? (p.causal ? min(n, p0 + qi + 1) : n) : 0;
  const uint32_t lane_taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  constexpr int HN = kPN / 2;  // keys of a tile owned by this thread
  constexpr int HD = D / 2;    // output channels owned by this thread
  float m_used = -INFINITY;    // reference maximum of the row, log2 units
  float l = 0.0f;              // sum of this half's P * 256
  bool ok = true;
  for (int j = 0; j < nkv; ++j) {
    const int s = j & 1;
    ok = __all_sync(0xffffffffu, role_wait(&sy->sfull[s], (j >> 1) & 1, sy, p.status));
    if (!ok) break;
    tc::fence_after_sync();
    float sv[HN];  // this half's 32 scores
    {
      float t[HN];
      const uint32_t sa = lane_taddr + s * L::s_cols;
      tc::ld_x16(sa + h * HN, *reinterpret_cast<float(*)[16]>(&sv[0]));
      tc::ld_x16(sa + h * HN + 16, *reinterpret_cast<float(*)[16]>(&sv[16]));
      tc::ld_x16(sa + kPN + h * HN, *reinterpret_cast<float(*)[16]>(&t[0]));
      tc::ld_x16(sa + kPN + h * HN + 16, *reinterpret_cast<float(*)[16]>(&t[16]));
      tc::wait_ld();
#pragma unroll
      for (int c = 0; c < HN; ++c) sv[c] += t[c];
    }
    tc::fence_before_sync();
    mbar_arrive(&sy->sfree[s]);
    // mask keys past this row's end (partial tiles only)
    if (j * kPN + kPN > kv_end_row) {
      const int own0 = j * kPN + h * HN;
#pragma unroll
      for (int c = 0; c < HN; ++c)
        if (own0 + c >= kv_end_row) sv[c] = -INFINITY;
    }
    float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
    for (int c = 4; c < HN; ++c) mx[c & 3] = fmaxf(mx[c & 3], sv[c]);
    const float mo = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    // the row's maximum: this half's and the other half's
    float mp;
    {
      volatile unsigned long long* mine = xm + ((j & 1) * 2 + h) * kPM + row;
      volatile unsigned long long* other = xm + ((j & 1) * 2 + 1 - h) * kPM + row;
      *mine = (static_cast<unsigned long long>(uint32_t(j)) << 32) | __float_as_uint(mo);
      unsigned long long w = *other;
      if (uint32_t(w >> 32) != uint32_t(j)) {
        const long long t0 = clock64();
        while (uint32_t((w = *other) >> 32) != uint32_t(j)) {
          if (*reinterpret_cast<volatile int*>(&sy->abort) || clock64() - t0 > kPWait) {
            *reinterpret_cast<volatile int*>(&sy->abort) = 1;
            atomicOr(p.status, KVQ_DEV_ERR_TIMEOUT);
            break;
          }
        }
      }
      mp = __uint_as_float(uint32_t(w));
    }
    ok = __all_sync(0xffffffffu, !*reinterpret_cast<volatile int*>(&sy->abort));
    if (!ok) break;
    const float mt = fmaxf(mo, mp) * 256.0f;  // keys were staged x 2^-8
    // lazy rescale: move the reference maximum only when it grew by more than 2^7
    float alpha = 1.0f;
    const bool move = mt > m_used + kLazyRescale || (m_used == -INFINITY && mt > -INFINITY);
    if (move) {
      alpha = m_used == -INFINITY ? 0.0f : ex2_approx(m_used - mt);
      l *= alpha;
      m_used = mt;
    }
    // P * 256 (values were staged x 2^-8): 2^(s*256 - (m - 8))
    const float mb = m_used == -INFINITY ? 0.0f : m_used - 8.0f;
    uint32_t ph[HN / 2], pl[HN / 2];
    float ls[2] = {0.0f, 0.0f};
#pragma unroll
    for (int c = 0; c < HN; c += 2) {
      const float e0 = ex2_approx(fmaf(sv[c], 256.0f, -mb));
      const float e1 = ex2_approx(fmaf(sv[c + 1], 256.0f, -mb));
      ls[0] += e0;
      ls[1] += e1;
      split2(e0, e1, ph[c / 2], pl[c / 2]);
    }
    l += ls[0] + ls[1];
    // A rescale needs O stable (PV_{j-1} complete); otherwise only this P buffer's
    // previous reader (PV_{j-2}) must be complete.  One barrier per P buffer, so a
    // wait is never more than one phase behind.
    const bool resc = j > 0 && __any_sync(0xffffffffu, move);  // TMEM access is warp-collective
    if (resc) {
      ok = __all_sync(0xffffffffu, role_wait(&sy->odone[(j - 1) & 1], ((j - 1) >> 1) & 1, sy, p.status));
      if (!ok) break;
      tc::fence_after_sync();
#pragma unroll
      for (int c = 0; c < HD; c += 16) {
        float t16[16];
        tc::ld_x16(lane_taddr + L::o_col + h * HD + c, t16);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) t16[e] *= alpha;
        tc::st_x16(lane_taddr + L::o_col + h * HD + c, t16);
      }
    } else if (j > 1) {
      ok = __all_sync(0xffffffffu, role_wait(&sy->odone[j & 1], ((j >> 1) - 1) & 1, sy, p.status));
      if (!ok) break;
      tc::fence_after_sync();
    }
    // P_j -> TMEM buffer j & 1: this half's 32 keys = 16 columns of fp16 pairs, hi then lo
    const uint32_t pb = lane_taddr + L::p_col + s * kPN + h * (HN / 2);
    tc::st_x16(pb, *reinterpret_cast<float(*)[16]>(&ph[0]));
    tc::st_x16(pb + kPN / 2, *reinterpret_cast<float(*)[16]>(&pl[0]));
    tc::wait_st();
    tc::fence_before_sync();
    mbar_arrive(&sy->pfull[s]);
  }
  // every MMA of the CTA has completed once both `fin` barriers arrive (also on the abort path)
  if (nkv > 0 && !(mbar_wait_bounded(&sy->fin[0], 0, kPWait) && mbar_wait_bounded(&sy->fin[1], 0, kPWait))) ok = false;
  ok = ok && !*reinterpret_cast<volatile int*>(&sy->abort);
  tc::fence_after_sync();

  // ---- epilogue: l of both halves, O / l -> staging -> inverse rotation -----
  float* xl = reinterpret_cast<float*>(sm + L::off_xl);
  xl[h * kPM + row] = l;
  named_sync(1, kSoftmax);
  const float lt = l + xl[(1 - h) * kPM + row];
  float* stage = reinterpret_cast<float*>(sm);  // [128][D + 4], reuses the Q and K slots
  // Thread (row, h) holds half a row of O / l.  With V rotated, the row's inverse
  // rotation is H_D = [[H, H], [H, -H]] with H = H_{D/2}: each half is transformed
  // in registers, the halves are exchanged through shared memory, and thread h
  // writes a + b (h = 0) or a - b (h = 1), a and b the transformed halves.
  float v[HD];
  {
    const float inv = (lt > 0.0f && nkv > 0 && ok) ? 256.0f / lt : 0.0f;
    const bool ld = __any_sync(0xffffffffu, nkv > 0 && ok);
#pragma unroll
    for (int c = 0; c < HD; c += 16) {
      float t16[16];
      if (ld) {
        tc::ld_x16(lane_taddr + L::o_col + h * HD + c, t16);
        tc::wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) t16[e] = 0.0f;
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) v[c + e] = t16[e] * inv;
    }
  }
  tc::fence_before_sync();
  if (p.rot_v) {
#pragma unroll
    for (int hh = 1; hh < HD; hh <<= 1)
#pragma unroll
      for (int j = 0; j < HD; ++j)
        if ((j & hh) == 0) {
          const float a = v[j], bq = v[j + hh];
          v[j] = a + bq;
          v[j + hh] = a - bq;
        }
  }
#pragma unroll
  for (int e = 0; e < HD; e += 4)
    *reinterpret_cast<float4*>(&stage[row * L::stage_stride + h * HD + e]) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
  named_sync(1, kSoftmax);
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, L::tmem_cols);
  }
  {
    const int rli = row / g, rhh = row % g, rqi = tile * p.ppt + rli;
    if (rli < p.ppt && rqi < p.n_tokens) {
      const float* part = &stage[row * L::stage_stride + (1 - h) * HD];
      const float sc = inv_sqrt_group<G>();
      const size_t e0 = (((size_t)b * p.n_tokens + rqi) * p.n_q_heads + kvh * g + rhh) * D + h * HD;
#pragma unroll
      for (int c = 0; c < HD; c += 8) {
        float o[8];
        if (p.rot_v) {
          const float4 x0 = *reinterpret_cast<const float4*>(part + c), x1 = *reinterpret_cast<const float4*>(part + c + 4);
          const float pv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = (h == 0 ? v[c + e] + pv[e] : pv[e] - v[c + e]) * sc;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = v[c + e];
        }
        if (p.out_dtype == KVQ_F32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + e0 + c);
          dst[0] = make_float4(o[0], o[1], o[2], o[3]);
          dst[1] = make_float4(o[4], o[5], o[6], o[7]);
        } else {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (p.out_dtype == KVQ_BF16) {
              const __nv_bfloat162 t2 = __floats2bfloat162_rn(o[2 * e], o[2 * e + 1]);
              w[e] = *reinterpret_cast<const uint32_t*>(&t2);
            } else {
              const __half2 t2 = __floats2half2_rn(o[2 * e], o[2 * e + 1]);
              w[e] = *reinterpret_cast<const uint32_t*>(&t2);
            }
          }
          *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + e0 + c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
}

template <int D>
cudaError_t run_prefill(const kvq_cache& c, Rot rot, const void* q, int q_dtype, int n_q_heads, int n_tokens,
                        const int32_t* q_pos0, int causal, float scale, void* out, int out_dtype, void* ws,
                        cudaStream_t st) {
  using L = PL<D>;
  const int max_tiles = c.max_ctx / kPN;
  SParams sp{};
  sp.k_qs = static_cast<const uint8_t*>(c.k_qs); sp.v_qs = static_cast<const uint8_t*>(c.v_qs);
  sp.k_d = static_cast<const uint8_t*>(c.k_d); sp.v_d = static_cast<const uint8_t*>(c.v_d);
  sp.k_qh = static_cast<const uint32_t*>(c.k_qh); sp.v_qh = static_cast<const uint32_t*>(c.v_qh);
  sp.k_tail = static_cast<const uint16_t*>(c.k_tail); sp.v_tail = static_cast<const uint16_t*>(c.v_tail);
  sp.seq_len = c.seq_len; sp.q_pos0 = q_pos0;
  sp.n_kv_heads = c.n_kv_heads; sp.max_ctx = c.max_ctx; sp.tail_len = c.tail_len;
  sp.k_type = c.k_type; sp.v_type = c.v_type; sp.n_tokens = n_tokens; sp.causal = causal ? 1 : 0;
  sp.max_tiles = max_tiles; sp.ws = static_cast<uint8_t*>(ws);
  sp.rows = row_map(c); sp.status = c.status;
  sp.n_outlier = c.n_outlier; sp.rot_k = rot.k; sp.rot_v = rot.v;
  sp.oidx = c.outlier_idx;
  sp.outl = static_cast<const uint8_t*>(c.outl);
  AParams p{};
  p.ws = static_cast<const uint8_t*>(ws);
  p.seq_len = c.seq_len; p.status = c.status;
  p.n_kv_heads = c.n_kv_heads; p.max_tiles = max_tiles;
  p.q = q; p.out = out; p.q_dtype = q_dtype; p.out_dtype = out_dtype;
  p.n_q_heads = n_q_heads; p.n_tokens = n_tokens;
  p.group = n_q_heads / c.n_kv_heads;
  p.ppt = kPM / p.group;
  p.ntiles = (n_tokens + p.ppt - 1) / p.ppt;
  p.q_pos0 = q_pos0; p.causal = sp.causal;
  p.rot_k = rot.k; p.rot_v = rot.v;
  p.scale_log2 = scale * kPLog2e;
  // + the rotated outlier parts of the tile's keys and values, [2][64][D] fp32
  const int stage_smem = L::tile + 1024 + (c.n_outlier ? 2 * kPN * D * 4 : 0);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(stage_kernel<D>), stage_smem);
  if (e != cudaSuccess) return e;
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(attn_kernel<D>), L::smem);
  if (e != cudaSuccess) return e;
  stage_kernel<D><<<dim3(max_tiles, c.n_kv_heads, c.batch), kStageThreads, stage_smem, st>>>(sp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_kernel<D><<<dim3(p.ntiles, c.n_kv_heads, c.batch), kAttnThreads, L::smem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int d, int group) { return (d == 64 || d == 128) && group >= 1 && group <= kPM; }

size_t prefill_workspace_bytes(const kvq_cache& c) {
  if (c.head_dim != 64 && c.head_dim != 128) return 0;
  return (size_t)c.batch * c.n_kv_heads * (c.max_ctx / kPN) * (size_t)(512 * c.head_dim);
}

cudaError_t launch_prefill(const kvq_cache& c, Rot rot, const void* q, int q_dtype, int n_q_heads, int n_tokens,
                           const int32_t* q_pos0, int causal, float scale, void* out, int out_dtype, void* ws,
                           cudaStream_t st) {
  switch (c.head_dim) {
    case 64:
      return run_prefill<64>(c, rot, q, q_dtype, n_q_heads, n_tokens, q_pos0, causal, scale, out, out_dtype, ws, st);
    case 128:
      return run_prefill<128>(c, rot, q, q_dtype, n_q_heads, n_tokens, q_pos0, causal, scale, out, out_dtype, ws, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
