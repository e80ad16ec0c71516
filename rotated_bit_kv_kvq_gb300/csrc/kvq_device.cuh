// Device helpers shared by the kvq kernels (sm_103a).
//
//  * warp Walsh-Hadamard transform of one head vector held in registers
//  * shared-memory barrier (mbarrier) + bulk / tensor copy wrappers with
//    bounded waits
//  * warp tensor-core fragments: ldmatrix, movmatrix, mma.m16n8k16 (f16)
//  * byte -> fp16 code conversions used by the dequantizing loaders
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

// Outlier-channel plane: groups of 16 body rows, 1088 bytes each (K codes
// int8 [16][32], V codes int8 [16][32], K scales fp16 [16], V scales fp16 [16]).
constexpr int kOutlTile = 1088;

constexpr int kQK = 32;  // values per quantization block

// ---------------------------------------------------------------------------
// Format traits (GGUF q4_0 / q5_0 / q8_0 payloads split into planes)
// ---------------------------------------------------------------------------
template <int QT> struct Fmt;
template <> struct Fmt<KVQ_TYPE_Q4_0> { static constexpr int qs_per_block = 16; static constexpr bool has_qh = false; };
template <> struct Fmt<KVQ_TYPE_Q5_0> { static constexpr int qs_per_block = 16; static constexpr bool has_qh = true; };
template <> struct Fmt<KVQ_TYPE_Q8_0> { static constexpr int qs_per_block = 32; static constexpr bool has_qh = false; };

// per-type facts used by every kernel
__host__ __device__ constexpr bool type_has_qh(int qt) { return qt == KVQ_TYPE_Q5_0 || qt == KVQ_TYPE_Q5_1; }
__host__ __device__ constexpr bool type_has_min(int qt) { return qt == KVQ_TYPE_Q4_1 || qt == KVQ_TYPE_Q5_1; }
// code offset of the _0 types (value = (code - offset) * d); 0 for q8_0 and the _1 types
__host__ __device__ constexpr int type_code_offset(int qt) {
  return qt == KVQ_TYPE_Q4_0 ? 8 : (qt == KVQ_TYPE_Q5_0 ? 16 : 0);
}
// bytes of one GGUF array-of-structs block
__host__ __device__ constexpr int type_block_bytes(int qt) {
  return qt == KVQ_TYPE_Q4_0 ? 18 : qt == KVQ_TYPE_Q5_0 ? 22 : qt == KVQ_TYPE_Q8_0 ? 34 : qt == KVQ_TYPE_Q4_1 ? 20 : 24;
}

__host__ __device__ inline int qs_row_bytes(int qt, int d) { return qt == KVQ_TYPE_Q8_0 ? d : d / 2; }

// Where the body row of logical position t of (sequence b, KV head h) lives:
// contiguous rows [batch][kv_heads][max_ctx], or in the paged layout
// [page][kv_heads][page_tokens] through the page table.
struct RowMap {
  int n_kv_heads, max_ctx, page_tokens, n_pages;
  const int32_t* page_table;
};
__host__ __device__ inline RowMap row_map(const kvq_cache& c) {
  return RowMap{c.n_kv_heads, c.max_ctx, c.page_tokens, c.n_pages, c.page_table};
}
// rows of the body planes (what a tensor map over a plane spans)
__host__ __device__ inline long long body_rows(const kvq_cache& c) {
  return c.page_tokens ? (long long)c.n_pages * c.n_kv_heads * c.page_tokens
                       : (long long)c.batch * c.n_kv_heads * c.max_ctx;
}
// -1 when the page id is outside the pool
__device__ __forceinline__ long long body_row(const RowMap& m, int b, int h, int t) {
  if (m.page_tokens == 0) return ((long long)b * m.n_kv_heads + h) * m.max_ctx + t;
  const int pg = m.page_table[(long long)b * (m.max_ctx / m.page_tokens) + t / m.page_tokens];
  if (pg < 0 || pg >= m.n_pages) return -1;
  return ((long long)pg * m.n_kv_heads + h) * m.page_tokens + t % m.page_tokens;
}

// ---------------------------------------------------------------------------
// Bit order of the K high-bit plane (q5_0 / q5_1 K).  A block's 32-bit word
// holds bit 4 of code c at bit c in GGUF order.  The K plane stores the bit of
// channel c (index bits c4..c0) at bit 16*c1 + 8*c3 + 4*c4 + 2*c2 + c0: channels
// c and c + 2 (one fp16 pair of the decode's score operand) sit 16 bits apart,
// and the pairs (c, c + 2) and (c + 16, c + 18) that one lane converts sit 4 bits
// apart, so one rotation serves both.  Four delta swaps of the bit index (bits
// 1<->2, 2<->3, 3<->4, then 2<->3 again) give the order; the inverse applies them
// in reverse.
// The V plane stores rows in pairs (2r, 2r + 1) and a row's bits in two 16-bit
// parts: per (pair, block) one 32-bit word [part 0 of row 2r | part 0 of row
// 2r + 1 << 16], then one of their parts 1, so that the two consecutive tokens of
// one transposed P.V operand arrive in one word.  Part c3 of a row holds channel c
// (index bits c4..c0) at bit 8*c2 + 4*c4 + 2*c1 + c0: the four channels 2g, 2g + 1,
// 2g + 16, 2g + 17 that one lane converts sit in one part, the pairs 4 bits apart,
// so two rotations serve them.  Two delta swaps of the bit index (bits 3<->4, then
// 2<->3) give the order.
// ---------------------------------------------------------------------------
__host__ __device__ inline uint32_t delta_swap(uint32_t x, int d, uint32_t m) {
  const uint32_t t = ((x >> d) ^ x) & m;
  return x ^ t ^ (t << d);
}
__host__ __device__ inline uint32_t qh_k_from_gguf(uint32_t x) {
  x = delta_swap(x, 2, 0x0C0C0C0Cu);
  x = delta_swap(x, 4, 0x00F000F0u);
  x = delta_swap(x, 8, 0x0000FF00u);
  return delta_swap(x, 4, 0x00F000F0u);
}
__host__ __device__ inline uint32_t qh_k_to_gguf(uint32_t x) {
  x = delta_swap(x, 4, 0x00F000F0u);
  x = delta_swap(x, 8, 0x0000FF00u);
  x = delta_swap(x, 4, 0x00F000F0u);
  return delta_swap(x, 2, 0x0C0C0C0Cu);
}
__host__ __device__ inline uint32_t qh_v_from_gguf(uint32_t x) {
  x = delta_swap(x, 8, 0x0000FF00u);
  return delta_swap(x, 4, 0x00F000F0u);
}
__host__ __device__ inline uint32_t qh_v_to_gguf(uint32_t x) {
  x = delta_swap(x, 4, 0x00F000F0u);
  return delta_swap(x, 8, 0x0000FF00u);
}
// 16-bit element index of part h (0: bits 0-15, 1: bits 16-31 of the word
// qh_v_from_gguf gives) of the V word of (row, block); nb blocks per row.
__host__ __device__ inline size_t qh_v_half(size_t row, int nb, int blk, int h) {
  return ((((row >> 1) * size_t(nb) + size_t(blk)) * 2 + size_t(h)) * 2) + (row & 1);
}
// Where one block's high-bit word goes: its two 16-bit halves (lo == nullptr: none).
struct QhDst {
  uint16_t* lo;
  uint16_t* hi;
  bool k;
};
__device__ __forceinline__ QhDst qh_dst(void* plane, bool k_plane, size_t row, int nb, int blk) {
  if (!plane) return QhDst{nullptr, nullptr, k_plane};
  uint16_t* p = static_cast<uint16_t*>(plane);
  if (k_plane) {
    uint16_t* w = p + 2 * (row * size_t(nb) + size_t(blk));
    return QhDst{w, w + 1, true};
  }
  return QhDst{p + qh_v_half(row, nb, blk, 0), p + qh_v_half(row, nb, blk, 1), false};
}
// store a high-bit word given in GGUF order
__device__ __forceinline__ void qh_put(const QhDst& d, uint32_t gguf) {
  const uint32_t w = d.k ? qh_k_from_gguf(gguf) : qh_v_from_gguf(gguf);
  *d.lo = uint16_t(w & 0xFFFFu);
  *d.hi = uint16_t(w >> 16);
}
// a stored high-bit word, in GGUF order
__device__ __forceinline__ uint32_t qh_get(const void* plane, bool k_plane, size_t row, int nb, int blk) {
  if (k_plane) return qh_k_to_gguf(static_cast<const uint32_t*>(plane)[row * size_t(nb) + size_t(blk)]);
  const uint16_t* p = static_cast<const uint16_t*>(plane);
  return qh_v_to_gguf(uint32_t(p[qh_v_half(row, nb, blk, 0)]) | (uint32_t(p[qh_v_half(row, nb, blk, 1)]) << 16));
}

// ---------------------------------------------------------------------------
// Unsigned 32-bit division by a run-time invariant divisor d >= 1 with one
// high multiply (Granlund and Montgomery, "Division by invariant integers
// using multiplication", 1994, section 4): l = ceil(log2 d),
// m = floor(2^32 (2^l - d) / d) + 1, q = (t + ((n - t) >> min(l, 1))) >>
// max(l - 1, 0) with t = mulhi(m, n); exact for every 32-bit n.
// ---------------------------------------------------------------------------
struct DivU32 {
  uint32_t d, m, s1, s2;
};
inline DivU32 make_divu32(uint32_t d) {
  uint32_t l = 0;
  while (l < 32 && (uint64_t(1) << l) < d) ++l;
  const uint32_t m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
  return DivU32{d, m, l < 1 ? l : 1u, l > 1 ? l - 1 : 0u};
}
__device__ __forceinline__ uint32_t div_u32(uint32_t n, const DivU32& v) {
  const uint32_t t = __umulhi(v.m, n);
  return (t + ((n - t) >> v.s1)) >> v.s2;
}

// ---------------------------------------------------------------------------
// small utilities
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// fp16x2 subtraction of a constant pair given as raw bits.
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// fp16x2 a * b and a * b + c, each rounded once to nearest even (never contracted
// or reassociated by the compiler).
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// P * d for an fp16 pair P = hi + lo (lo the rounding residue of hi) and an fp16
// pair d, as a new hi + lo pair: hi = RN(P_hi * d); the residue P_hi * d - hi is
// exact in one fused operation (a product of two 11-bit significands rounded to 11
// bits leaves at most 11 bits), and lo = RN(P_lo * d + residue).
__device__ __forceinline__ void hscale_split(uint32_t p_hi, uint32_t p_lo, uint32_t d, uint32_t& hi, uint32_t& lo) {
  hi = hmul2_bits(p_hi, d);
  uint32_t r;
  asm("{\n\t.reg .b32 nh;\n\tneg.f16x2 nh, %3;\n\tfma.rn.f16x2 %0, %1, %2, nh;\n\t}"
      : "=r"(r) : "r"(p_hi), "r"(d), "r"(hi));
  lo = hfma2_bits(p_lo, d, r);
}

// pack two floats into fp16x2 (round to nearest even); lo goes to bits 0..15.
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// Code conversions to fp16 pairs.  A byte value u placed in the low byte of a
// 0x64XX half is the fp16 number 1024 + u exactly, so one subtraction gives
// the signed code, exactly.
// ---------------------------------------------------------------------------
// Nibbles at bit offsets s and s+16 of r (codes 0..15) plus optional high
// bits already placed at bit 4 / bit 20 in `hb` -> fp16 pair (code - off).
__device__ __forceinline__ uint32_t nib_pair(uint32_t r, int s, uint32_t hb_or_magic, uint32_t off_bits) {
  uint32_t t = ((r >> s) & 0x000F000Fu) | hb_or_magic;
  return hsub2_bits(t, off_bits);
}
// The same for nibbles at bit offsets 4 and 20 (high bits already at bit 8 / bit 24
// in `hb16`): the half is 1024 + 16 * code exactly; one fused x / 16 - (64 + off)
// gives code - off exactly.  Saves the shift of the plain form.
__device__ __forceinline__ uint32_t nib_pair_x16(uint32_t r, uint32_t hb16_or_magic, uint32_t neg_off_bits) {
  const uint32_t t = (r & 0x00F000F0u) | hb16_or_magic;
  return hfma2_bits(t, 0x2C002C00u, neg_off_bits);  // 0x2C00 = 1/16
}
// -(64 + off) as an fp16 pair for nib_pair_x16 (off = 0, 8 or 16)
__host__ __device__ constexpr uint32_t neg_off_x16_bits(int off) {
  return (off == 8 ? 0xD480u : off == 16 ? 0xD500u : 0xD400u) * 0x10001u;
}

// Offset-binary bytes i0, i1 (0..3) of ru (code + 128: the body planes store q8_0
// codes so; the outlier plane's signed bytes are XORed with 0x80 first) -> fp16
// pair (code).
template <int I0, int I1>
__device__ __forceinline__ uint32_t i8_pair(uint32_t ru) {
  uint32_t t = __byte_perm(ru, 0x64646464u, I0 | (4 << 4) | (I1 << 8) | (4 << 12));
  return hsub2_bits(t, 0x64806480u);  // 1152 = 1024 + 128
}
// bf16 pair -> fp16 pair scaled by 2^-8 (keeps |x| < 1.6e7 finite in fp16).
__device__ __forceinline__ uint32_t bf16x2_to_h2_scaled(uint32_t b) {
  float lo = __uint_as_float(b << 16) * 0.00390625f;
  float hi = __uint_as_float(b & 0xFFFF0000u) * 0.00390625f;
  return pack_h2(lo, hi);
}

// ---------------------------------------------------------------------------
// Warp tensor-core fragments
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(a));
  return r;
}
// D = A(16x16, row) * B(16x8, col) + C, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// Shared-memory barriers and bulk copies (TMA)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// true in one lane of the (converged) warp: the lowest active one
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b32 l;\n\telect.sync l|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// One wait attempt; the thread may sleep up to ~suspend_ns inside it while the
// phase is incomplete (so waiting does not spin through issue slots).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t suspend_ns = 100000u) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns) : "memory");
  return ok != 0;
}
// Bounded wait: gives up after ~`limit_cycles` SM cycles and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit_cycles) return false;
  }
  return true;
}

// 1-D bulk copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// 1-D bulk copy shared -> global (bulk-group completion; 16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(dst), "r"(smem_u32(src)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed shared -> global bulk copy of this thread has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// plain arrive (count 1) on a shared-memory barrier
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// named barrier over `count` threads (a multiple of 32)
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// 2^x with the hardware approximation (relative error below 2^-22; 2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// 3-D tiled tensor copy global -> shared: a row-major plane seen as (x: bytes within a
// box column, y: row, z: box column), so that one copy fills [column][row][box width].
__device__ __forceinline__ void tma_3d_g2s(void* dst, const CUtensorMap* map, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(0), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Byte offset of (row r, byte x) inside a tile that a TMA box copy wrote with
// the swizzle matching its box width W (128, 64 or 32 bytes: 16-byte chunks
// XORed with address bits 7..9; 16 bytes: no swizzle).  Boxes of `rows` x W are stored one after
// another along x.  The tile base must be 1024-byte aligned.
template <int W>
__device__ __forceinline__ uint32_t swz_off(int r, int x, int rows) {
  const int box = x / W, xi = x % W;
  int chunk = xi >> 4;
  if (W == 128) chunk ^= (r & 7);
  else if (W == 64) chunk ^= ((r >> 1) & 3);
  else if (W == 32) chunk ^= ((r >> 2) & 1);  // W == 16: no swizzle
  return box * rows * W + r * W + (chunk << 4) + (xi & 15);
}

// ldmatrix rows of a 16-row tile written as W-byte boxes with their swizzle, read
// at 16-byte chunk j + h of row r, j even (compile-time), h in {0, 1} (per lane):
// j + h stays in j's box and chunk (j + h) mod (W/16) = (j mod (W/16)) ^ h, so the
// swizzled offset is a per-lane constant (one per even chunk of a box, W/32 of
// them) plus a compile-time box offset.
template <int W>
__device__ __forceinline__ void swz_lane(int r, int h, uint32_t (&lb)[W / 32]) {
  const int key = W == 128 ? (r & 7) : W == 64 ? ((r >> 1) & 3) : ((r >> 2) & 1);
#pragma unroll
  for (int i = 0; i < W / 32; ++i) lb[i] = r * W + (((2 * i) ^ (h ^ key)) << 4);
}
// byte offset of the W-byte box column holding 16-byte chunk j, R rows per column
template <int W, int R = 16>
__host__ __device__ constexpr int swz_box_off(int j) { return (16 * j / W) * R * W; }
template <int W>
__host__ __device__ constexpr int swz_lane_idx(int j) { return (j % (W / 16)) / 2; }

// ---------------------------------------------------------------------------
// Warp FWHT: a head vector of D values, lane l holding E = D/32 of them.
// Channel of value j in lane l:  c = (j / P) * G + l * P + (j % P), P = G/32,
// i.e. G-wide Hadamard groups, each spread over the warp with P consecutive
// channels per lane.  Computes the unnormalized Sylvester-order transform of
// every group (callers scale by 1/sqrt(G)).
// ---------------------------------------------------------------------------
template <int D, int G>
__device__ __forceinline__ void warp_fwht(float (&v)[D / 32], int lane) {
  constexpr int P = G / 32;      // consecutive channels per lane per group
  constexpr int NG = D / G;      // groups
  static_assert(P >= 1 && D % G == 0, "bad FWHT layout");
#pragma unroll
  for (int h = 1; h < P; h <<= 1) {          // partners inside the lane
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
#pragma unroll
      for (int j = 0; j < P; ++j)
        if ((j & h) == 0) {
          const float a = v[gi * P + j], b = v[gi * P + j + h];
          v[gi * P + j] = a + b;
          v[gi * P + j + h] = a - b;
        }
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {         // partners across lanes (stride m*P)
    // upper lane: o - v, lower lane: v + o; as o + sgn*v (sgn*v is exact, so the
    // single rounding is that of the plain sum or difference)
    const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      const float o = __shfl_xor_sync(0xffffffffu, v[j], m);
      v[j] = fmaf(sgn, v[j], o);
    }
  }
}

// Unnormalised Sylvester FWHT of a vector held by R consecutive lanes, 32
// consecutive channels each: the 5 in-lane channel bits in registers, the
// log2(R) lane bits by shuffles among the lanes of `mask`, which holds whole
// R-lane groups.  Every output is one rounding of a plain sum or difference:
// a - b is taken as fma(b, -1, a) (the product is exact), and the channel-bit
// stages above bit 0 use the packed fp32x2 forms, two channels per
// instruction with the same per-channel rounding.
template <int R>
__device__ __forceinline__ void lane_fwht(float (&r)[32], int lane, unsigned mask) {
  const float2 m1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {  // channel bit 0: the two halves of a pair
    const float a = r[j], b = r[j + 1];
    r[j] = a + b;
    r[j + 1] = a - b;
  }
#pragma unroll
  for (int hh = 2; hh < 32; hh <<= 1)
#pragma unroll
    for (int j = 0; j < 32; j += 2)
      if ((j & hh) == 0) {
        const float2 a = make_float2(r[j], r[j + 1]), b = make_float2(r[j + hh], r[j + hh + 1]);
        const float2 s2 = __fadd2_rn(a, b), d2 = __ffma2_rn(b, m1, a);
        r[j] = s2.x; r[j + 1] = s2.y;
        r[j + hh] = d2.x; r[j + hh + 1] = d2.y;
      }
#pragma unroll
  for (int m = 1; m < R; m <<= 1) {
    const float sgn = (lane & m) ? -1.0f : 1.0f;  // upper partner: o - v, lower: v + o
    const float2 sg = make_float2(sgn, sgn);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float2 o = make_float2(__shfl_xor_sync(mask, r[j], m), __shfl_xor_sync(mask, r[j + 1], m));
      const float2 t = __ffma2_rn(sg, make_float2(r[j], r[j + 1]), o);
      r[j] = t.x; r[j + 1] = t.y;
    }
  }
}

// y[j] *= s for the 32 values of a lane block (packed: the same rounding per value).
__device__ __forceinline__ void scale32(float (&y)[32], float s) {
  const float2 s2 = make_float2(s, s);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float2 t = __fmul2_rn(make_float2(y[j], y[j + 1]), s2);
    y[j] = t.x; y[j + 1] = t.y;
  }
}

// 1/sqrt(G) correctly rounded to fp32.
template <int G>
__host__ __device__ constexpr float inv_sqrt_group() {
  static_assert(G == 32 || G == 64 || G == 128 || G == 256 || G == 512, "Hadamard group of 32 to 512");
  return G == 32    ? 0.17677669529663688f
         : G == 64  ? 0.125f
         : G == 128 ? 0.088388347648318440f
         : G == 256 ? 0.0625f
                    : 0.044194173824159216f;
}
static_assert(inv_sqrt_group<256>() == 0.0625f && inv_sqrt_group<512>() * inv_sqrt_group<512>() < 0.001954f &&
                  inv_sqrt_group<512>() * inv_sqrt_group<512>() > 0.001952f,
              "");

// Channel held in slot j of lane l for the FWHT layout above.
template <int D, int G>
__device__ __forceinline__ int fwht_channel(int lane, int j) {
  constexpr int P = G / 32;
  return (j / P) * G + lane * P + (j % P);
}

}  // namespace kvq
