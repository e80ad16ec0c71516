/*
 * kvq.h -- C ABI of the rotated, block-quantized KV-cache attention library.
 *
 * What it computes.  Per attention head, K and V vectors are multiplied by a
 * normalized Walsh-Hadamard matrix H/sqrt(G) and stored rotated; queries are
 * rotated the same way, so q.k -- and the attention scores -- are unchanged,
 * and the attention output is rotated back at the end (velog post
 * "fix-kv-cache-quantization-outliers", section 아다마르 회전).  Rotation is
 * used when head_dim >= 64 and a multiple of 64, and K / V rotation can each
 * be switched off (same post, section 적용 및 배경 기술).  The rotated vectors
 * are stored in the GGUF q4_0 / q5_0 / q8_0 block formats, which the same
 * section says stay unchanged: 32 values per block with an fp16 scale; the
 * scale + minimum formats q4_1 / q5_1, which the aitrends.kr summary "KV 캐시
 * 양자화 벤치마크: KVarN과 Precision Tail" (section 섹션별 상세) benchmarks in
 * K/V type pairs beside them, are stored the same way.  A BF16 "precision
 * tail" keeps the most recent tokens unquantized (same summary, section
 * 용어 해설).
 *
 * Conventions for every entry point.
 *  - Ownership: the library never allocates, frees or synchronizes (except
 *    kvq_sync_status).  Every pointer in kvq_cache and every q / k / v / out /
 *    workspace pointer is caller-owned DEVICE memory on the current CUDA
 *    device; host pointers are marked as such.  `stream` is a cudaStream_t
 *    (NULL = legacy default stream); all work is enqueued on it and the call
 *    returns without waiting.
 *  - Errors: argument errors are detected on the host before any launch and
 *    returned synchronously; nothing is launched then.  Errors that depend on
 *    device-resident values (sequence lengths) set bits in the cache's status
 *    words; kvq_sync_status reports them.  KVQ_ERR_CUDA reports a launch
 *    error (or an earlier asynchronous error surfacing at launch).
 *  - Calls that touch the same cache must be ordered on one stream.
 *  - Layouts are row-major; [a][b] means b varies fastest.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#define KVQ_VERSION 1

/* ---- status codes ------------------------------------------------------ */
typedef int32_t kvq_status;
#define KVQ_OK                 0
#define KVQ_ERR_INVALID_ARG   -1  /* null pointer, bad size, bad alignment, bad enum  */
#define KVQ_ERR_UNSUPPORTED   -2  /* valid but not built: head_dim, type pair, rotation on an ineligible head_dim */
#define KVQ_ERR_WORKSPACE     -3  /* workspace pointer NULL or ws_bytes too small      */
#define KVQ_ERR_CUDA          -4  /* a CUDA runtime call or launch failed              */
#define KVQ_ERR_TIMEOUT       -5  /* a bounded on-device wait gave up (see status bit) */
#define KVQ_ERR_DEVICE_RANGE  -6  /* device-side range check failed (see status bits)  */

/* ---- block formats (GGUF, unchanged) ----------------------------------- */
#define KVQ_TYPE_Q4_0 0   /* fp16 d = m/-8,  code = min(15, trunc(x/d + 8.5)),  x = (code-8)*d  */
#define KVQ_TYPE_Q5_0 1   /* fp16 d = m/-16, code = min(31, trunc(x/d + 16.5)), x = (code-16)*d */
#define KVQ_TYPE_Q8_0 2   /* fp16 d = amax/127, code = roundf(x/d) in [-127,127], x = code*d     */
#define KVQ_TYPE_Q4_1 3   /* fp16 d = (hi-lo)/15, fp16 lo, code = min(15, trunc((x-lo)/d + 0.5)), x = code*d + lo */
#define KVQ_TYPE_Q5_1 4   /* fp16 d = (hi-lo)/31, fp16 lo, code = min(31, trunc((x-lo)/d + 0.5)), x = code*d + lo */
/* m = the value of largest magnitude in the 32-value block (first on ties);
 * lo / hi = its smallest / largest value (first on ties).  1/d is taken as 0
 * when d == 0.  Nibble packing (q4_x, q5_x): byte k = code_k | code_{k+16} << 4;
 * q5_x high bits: bit j of a 32-bit word = bit 4 of code_j. */

/* ---- element types of q / k / v / out ----------------------------------- */
#define KVQ_F32  0
#define KVQ_BF16 1
#define KVQ_F16  2

/* ---- cache flags (kvq_cache.flags) ------------------------------------- */
#define KVQ_ROT_AUTO   1u  /* rotate K and V when head_dim >= 64 and %64 == 0, else silently off */
#define KVQ_ROT_K_OFF  2u  /* no K rotation (queries are then not rotated either)             */
#define KVQ_ROT_V_OFF  4u  /* no V rotation (the output is then not rotated back)             */
/* flags == 0 (no KVQ_ROT_AUTO): rotation is requested explicitly; an
 * ineligible head_dim then gives KVQ_ERR_UNSUPPORTED unless both _OFF bits
 * are set. */

/* ---- append flags -------------------------------------------------------- */
#define KVQ_INPUT_PREROTATED 1u  /* k / v are already rotated: store them as given */

/* ---- planes of a cache (kvq_plane_bytes) --------------------------------- */
/* body planes: rows [batch][kv_heads][max_ctx], or [n_pages][kv_heads][page_tokens] when paged */
#define KVQ_PLANE_K_QS    0  /* uint8 [batch][kv_heads][max_ctx][qs_row]    qs_row = d (q8_0) or d/2 (the others);
                                the GGUF qs bytes of the token's blocks, except that q8_0 codes are stored offset
                                binary (code + 128, the GGUF byte XOR 0x80); kvq_dequant_debug returns GGUF bytes */
#define KVQ_PLANE_K_QH    1  /* uint32 [batch][kv_heads][max_ctx][d/32]     q5_0 / q5_1 only (0 bytes otherwise);
                                the bit of channel c (index bits c4..c0) of a block sits at bit 16*c1 + 8*c3 +
                                4*c4 + 2*c2 + c0, a permutation of the GGUF word, whose bit c is bit 4 of code c;
                                kvq_dequant_debug returns GGUF bytes                                                 */
#define KVQ_PLANE_K_D     2  /* fp16 [batch][kv_heads][max_ctx][d/32]       block scales; q4_1 / q5_1: fp16 pairs
                                (d, lo) [..][d/32][2], i.e. the GGUF block header                                   */
#define KVQ_PLANE_V_QS    3
#define KVQ_PLANE_V_QH    4  /* uint32, as K_QH in size, rows in pairs: a row's bits split in two 16-bit parts, the
                                bit of channel c (index bits c4..c0) in part c3 at bit 8*c2 + 4*c4 + 2*c1 + c0; for
                                rows (2r, 2r + 1) and block j, word 2(r*d/32 + j) holds the two rows' parts 0 (row 2r
                                in its low half) and word 2(r*d/32 + j) + 1 their parts 1 */
#define KVQ_PLANE_V_D     5
#define KVQ_PLANE_K_TAIL  6  /* bf16 [batch][kv_heads][tail_len][d]          rotated values, slot = pos % tail_len */
#define KVQ_PLANE_V_TAIL  7
#define KVQ_PLANE_SEQ_LEN 8  /* int32 [batch]                               tokens stored per sequence           */
#define KVQ_PLANE_STATUS  9  /* uint32 [4]                                  device status words; zero before use */
#define KVQ_PLANE_OUTLIER 10  /* [rows / 16][1088 B]                         outlier-channel q8_0 blocks (n_outlier > 0) */
#define KVQ_PLANE_OUTLIER_IDX 11  /* int32 [kv_heads][n_outlier]            the caller's outlier channel lists          */
#define KVQ_NUM_PLANES   12

/* device status word 0 bits (read by kvq_sync_status) */
#define KVQ_DEV_ERR_APPEND_RANGE  1u  /* an append would pass max_ctx, or n_new_per_seq[b] not in [0, n_new] */
#define KVQ_DEV_ERR_PREFILL_RANGE 2u  /* a prefill query position is negative                              */
#define KVQ_DEV_ERR_TIMEOUT       4u  /* a bounded wait on a shared-memory barrier gave up                 */
#define KVQ_DEV_ERR_PAGE          8u  /* a page_table entry lies outside [0, n_pages) (paged layout)        */
#define KVQ_DEV_ERR_OUTLIER      16u  /* an outlier_idx row is not strictly increasing inside [0, head_dim) */

/*
 * The cache descriptor.  Body planes hold the packed payload of every block:
 * block j of token t of (seq b, kv head h) has its qs bytes at
 * qs + ((b*kv_heads + h)*max_ctx + t)*qs_row + j*(16 or 32), its high-bit
 * word (q5_0) at qh[((b*kv_heads + h)*max_ctx + t)*(d/32) + j] and its scale
 * at d[same index].  The bytes of one block are exactly the GGUF block
 * payload; kvq_dequant_debug can export them in GGUF array-of-structs order.
 *
 * Requirements (checked by every call): head_dim % 32 == 0 and
 * 32 <= head_dim <= 512; max_ctx % 64 == 0 and max_ctx <= 2^30; tail_len >= 0;
 * every non-NULL plane 16-byte aligned; k_qh / v_qh non-NULL only for q5_0 and
 * q5_1 (required then);
 * k_tail / v_tail non-NULL iff tail_len > 0.  Decode supports head_dim in
 * {64, 128, 192, 256, 320} for every K / V format pair (192 and 320 rotate in
 * 64-wide blocks; with outlier channels: 64, 128, 256); prefill supports
 * head_dim 64 and 128 with up to 128 query heads per KV head; append and debug
 * support every multiple of 32 up to 512.  Prefill stores keys and values
 * internally as fp16 x 2^-8, so it needs |rotated value| < 1.6e7.
 */
typedef struct kvq_cache {
  int32_t batch;        /* sequences                                   */
  int32_t n_kv_heads;   /* KV heads per sequence                       */
  int32_t head_dim;     /* d                                           */
  int32_t max_ctx;      /* token capacity per sequence (multiple of 64, at most 2^30) */
  int32_t tail_len;     /* T: recent tokens also kept in bf16 (0 = off)*/
  int32_t k_type;       /* KVQ_TYPE_*                                  */
  int32_t v_type;       /* KVQ_TYPE_*                                  */
  uint32_t flags;       /* KVQ_ROT_*                                   */
  void* k_qs; void* k_qh; void* k_d;
  void* v_qs; void* v_qh; void* v_d;
  void* k_tail; void* v_tail;
  int32_t* seq_len;     /* device int32 [batch]                        */
  uint32_t* status;     /* device uint32 [4], zero-initialised         */
  /* Paged layout (optional; page_tokens == 0 keeps the contiguous rows
   * [batch][kv_heads][max_ctx] above).  Otherwise the body planes are one pool
   * of n_pages pages shared by all sequences, rows [n_pages][kv_heads]
   * [page_tokens], and position t of sequence b lives in page
   * page_table[b * (max_ctx / page_tokens) + t / page_tokens] at row offset
   * t % page_tokens.  max_ctx stays the logical capacity per sequence; the
   * bf16 tail stays per sequence.  A page id outside [0, n_pages) met by a
   * kernel sets KVQ_DEV_ERR_PAGE and that page reads as empty / is not
   * written.  Library addition for serving batches (block-table allocation);
   * the pages describe only the contiguous cache. */
  int32_t page_tokens;        /* 0, or a multiple of 64 that divides max_ctx   */
  int32_t n_pages;            /* pages in the pool (paged layout)              */
  const int32_t* page_table;  /* device int32 [batch][max_ctx / page_tokens]   */
  /* Outlier channels kept at 8 bits (optional; n_outlier == 0 turns them off).
   * The pages (velog "fix-kv-cache-quantization-outliers", section 적용 및
   * 배경 기술) name this direction without fixing it; the reading implemented
   * here: per KV head the caller lists n_outlier channels of the original
   * basis (outlier_idx, strictly increasing).  The write path stores their
   * values unrotated as one q8_0 block in slot order (plane `outl`, body rows
   * contiguous or paged like the body, in groups of 16 rows of 1088 bytes: K
   * codes int8 [16][32], V codes int8 [16][32], K scales fp16 [16], V scales
   * fp16 [16], so one copy moves a 16-token tile), sets them to
   * zero in the vector and rotates / quantizes the rest as usual; the bf16
   * tail keeps the whole rotated vector.  Attention adds q_O . k_O to every
   * body score and scatters sum_t p_t v_O,t back to those channels of the
   * output.  Requires head_dim >= 64 and inputs in the original basis (no
   * KVQ_INPUT_PREROTATED).  Supported by append, the fused step, decode (the
   * q4_0 / q5_0 / q8_0 pairs) and prefill (its staging adds each key's and
   * value's rotated outlier part to the dequantized rest); kvq_dequant_debug
   * reads the low-bit planes only.  A row
   * of outlier_idx that is not strictly increasing in [0, head_dim) sets
   * KVQ_DEV_ERR_OUTLIER; its invalid slots are then ignored. */
  int32_t n_outlier;           /* 0 or 32                                     */
  const int32_t* outlier_idx;  /* device int32 [kv_heads][n_outlier]          */
  void* outl;                  /* KVQ_PLANE_OUTLIER                           */
} kvq_cache;

/* Library version (KVQ_VERSION). */
KVQ_API int32_t kvq_version(void);

/* Human-readable name of a status code (static string). */
KVQ_API const char* kvq_status_string(kvq_status s);

/* Bytes the caller must allocate for plane `plane` (KVQ_PLANE_*) of a cache
 * with the given sizes and types; pointers in `c` are ignored.  Returns 0 for
 * an absent plane (qh of a type other than q5_0 / q5_1, tail of tail_len 0,
 * outlier planes of n_outlier 0) or an invalid descriptor. */
KVQ_API size_t kvq_plane_bytes(const kvq_cache* c, int32_t plane);

/* Host-side check of a descriptor (sizes, types, pointers, alignment). */
KVQ_API kvq_status kvq_cache_check(const kvq_cache* c);

/* The enable rule (velog 적용 및 배경 기술): writes 1/0 to *rot_k and *rot_v
 * (host pointers).  KVQ_ROT_AUTO turns rotation on iff head_dim >= 64 and
 * head_dim % 64 == 0; the _OFF bits switch each side off; an explicit request
 * (no AUTO bit) on an ineligible head_dim returns KVQ_ERR_UNSUPPORTED. */
KVQ_API kvq_status kvq_resolve_rotation(const kvq_cache* c, int32_t* rot_k, int32_t* rot_v);

/*
 * Rotate, quantize and append new tokens (write path).  The rotation is
 * applied where the cache is stored, so the stored K and V are rotated (velog
 * "fix-kv-cache-quantization-outliers", section 아다마르 회전); the blocks are
 * the GGUF formats, unchanged (section 적용 및 배경 기술); the most recent
 * tokens also stay in bf16 (aitrends.kr "KVarN과 Precision Tail", section
 * 용어 해설).
 *   k, v          device [batch][n_new][n_kv_heads][head_dim] of in_dtype
 *   n_new         rows per sequence in k / v (>= 0; 0 is a no-op; batch * n_new *
 *                 n_kv_heads * 2 must stay below 2^31, else KVQ_ERR_INVALID_ARG)
 *   n_new_per_seq device int32 [batch] or NULL: tokens actually appended for
 *                 sequence b (0 <= n_new_per_seq[b] <= n_new); rows past it
 *                 are ignored.  NULL means n_new for every sequence.
 *   append_flags  KVQ_INPUT_PREROTATED or 0
 * Token i of sequence b goes to position p = seq_len[b] + i: its rotated
 * values are quantized into the body planes at p, and if p is among the last
 * tail_len positions written by this call its rotated values (bf16, round to
 * nearest even) also go to tail slot p % tail_len.  Afterwards seq_len[b] has
 * grown by the tokens appended.  A sequence whose append would pass max_ctx
 * (or whose count is out of range) is left untouched and sets
 * KVQ_DEV_ERR_APPEND_RANGE.  Uses status word 1 as a completion counter.
 */
KVQ_API kvq_status kvq_rotate_quantize_append(const kvq_cache* c, const void* k, const void* v,
                                      int32_t in_dtype, int32_t n_new,
                                      const int32_t* n_new_per_seq, uint32_t append_flags,
                                      void* stream);

/* Workspace bytes kvq_decode_attention needs for this cache and n_q_heads on
 * the current device (0 on an invalid descriptor). */
KVQ_API size_t kvq_decode_workspace_bytes(const kvq_cache* c, int32_t n_q_heads);

/*
 * One decode step of attention for every sequence (read path).  The query is
 * rotated like the keys, the scores are the rotated dot products, and the
 * weighted sum of the rotated values is rotated back (velog
 * "fix-kv-cache-quantization-outliers", section 아다마르 회전); the latest
 * tail_len tokens are read from the bf16 tail (aitrends.kr "KVarN과 Precision
 * Tail", section 용어 해설).
 *   q      device [batch][n_q_heads][head_dim] of q_dtype (unrotated)
 *   out    device [batch][n_q_heads][head_dim] of out_dtype (original basis)
 *   scale  softmax scale; 0 means 1/sqrt(head_dim)
 * Query head h uses KV head h / (n_q_heads / n_kv_heads).  Scores are taken
 * in the rotated basis (q rotated when K rotation is on); keys at positions
 * [n - tail_len, n) come from the bf16 tail, older ones from the quantized
 * body (n = seq_len[b]); the softmax-weighted sum of values is rotated back
 * when V rotation is on.  A sequence with n == 0 yields zeros.
 * n_q_heads must be a multiple of n_kv_heads.  workspace: device memory of at
 * least kvq_decode_workspace_bytes(c, n_q_heads) bytes, 16-byte aligned.
 */
KVQ_API kvq_status kvq_decode_attention(const kvq_cache* c, const void* q, int32_t q_dtype,
                                int32_t n_q_heads, float scale, void* out, int32_t out_dtype,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * kvq_decode_attention without a caller-provided workspace.  The pages have
 * no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory themselves -- for example a plugin inside a host
 * application that owns every device allocation, or a runtime that works
 * within a fixed memory budget reserved up front -- and therefore cannot
 * supply the workspace kvq_decode_attention needs.
 *
 * The split partials go to one scratch array of KVQ_NOALLOC_SCRATCH_BYTES
 * that the library defines statically in device memory: every GPU that loads
 * the library holds it until the process exits.  The call allocates nothing
 * (no cudaMalloc, no allocating library routine).  Every call looks up the
 * array's device address (cudaGetSymbolAddress, a host-side lookup that
 * allocates nothing) with the caller's device current, so a call after a
 * reset of that device's context finds the array wherever it now lives.  The
 * first call in a process may load the library's device code: make it
 * before any stream capture.
 * Arguments, results and errors are those of kvq_decode_attention, except:
 * KVQ_ERR_WORKSPACE when kvq_decode_workspace_bytes(c, n_q_heads) exceeds
 * KVQ_NOALLOC_SCRATCH_BYTES (nothing is launched then).  All calls share the
 * one array and it keeps the last call's contents.  A call writes the
 * partition header and every (m, l) pair its merge reads; the partial rows of
 * a split whose token range came out empty are not written and may hold an
 * earlier call's values (even Inf or NaN): the merge reads them but drops them
 * by their weight 0, never multiplying them.  Calls that overlap on the GPU
 * (for example on two streams at once) race on the array and must not be
 * issued.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)
KVQ_API kvq_status kvq_decode_attention_noalloc(const kvq_cache* c, const void* q, int32_t q_dtype,
                                                int32_t n_q_heads, float scale, void* out,
                                                int32_t out_dtype, void* stream);

/*
 * One decode step: kvq_rotate_quantize_append(c, k, v, in_dtype, n_new,
 * n_new_per_seq, append_flags) followed by kvq_decode_attention(c, q, ...),
 * with the same arguments, results and errors as the two calls in sequence.
 * When n_new <= tail_len, the query heads of a KV head fit one CTA (up to 8)
 * and the tail fits one (tail_len <= 4096), the append runs inside the decode
 * launch: the CTA that reads a (sequence, KV head)'s bf16 tail first writes
 * the new tokens (body blocks and tail rows), and the merge kernel advances
 * seq_len after every split has read it -- one launch pair instead of three
 * kernels.  Otherwise the two calls run in sequence.  The workspace is the
 * decode's (kvq_decode_workspace_bytes).  Library addition for serving loops:
 * the pages describe the append and the attention, not this entry point.
 */
KVQ_API kvq_status kvq_append_decode(const kvq_cache* c, const void* k, const void* v, int32_t in_dtype,
                                     int32_t n_new, const int32_t* n_new_per_seq, uint32_t append_flags,
                                     const void* q, int32_t q_dtype, int32_t n_q_heads, float scale, void* out,
                                     int32_t out_dtype, void* workspace, size_t ws_bytes, void* stream);

/* Workspace bytes kvq_prefill_attention needs (a pure size query: no
 * pointer in *c is read): batch * n_kv_heads * (max_ctx / 64) tiles of
 * 512 * head_dim bytes each, i.e. 8 bytes per cached K+V element of the
 * capacity.  Every 64-key tile a call's queries can see is dequantized once
 * into it (fp16 hi + lo operand tiles) before the attention kernel streams
 * it.  0 when the shape is invalid or prefill does not support it.  The
 * library-level staging has no counterpart in the method's description; it
 * is how this implementation avoids dequantizing a key once per query tile. */
KVQ_API size_t kvq_prefill_workspace_bytes(const kvq_cache* c, int32_t n_q_heads, int32_t n_tokens);

/*
 * Chunked attention of a block of queries per sequence over the cache
 * (prompt processing), after their K/V have been appended: the prompt-side
 * use of the same rotated cache (velog "fix-kv-cache-quantization-outliers",
 * section 트레이드오프, reports its cost apart from token generation), with
 * the bf16 tail as in decode (aitrends.kr "KVarN과 Precision Tail", section
 * 용어 해설).
 *   q       device [batch][n_tokens][n_q_heads][head_dim] of q_dtype
 *   q_pos0  device int32 [batch] or NULL: absolute position of query 0 of
 *           sequence b; NULL means seq_len[b] - n_tokens (the just-appended
 *           prompt).  A negative position sets KVQ_DEV_ERR_PREFILL_RANGE and
 *           that sequence's rows are written as zeros.
 *   causal  non-zero: query at position p sees keys t <= p; always t < seq_len[b]
 *   chunk   queries per processing chunk (multiple of 64, or 0 for 512); it
 *           orders the work and does not change the result
 *   out     device [batch][n_tokens][n_q_heads][head_dim] of out_dtype
 *   workspace, ws_bytes  device scratch, 16-byte aligned, at least
 *           kvq_prefill_workspace_bytes(c, n_q_heads, n_tokens) bytes, else
 *           KVQ_ERR_WORKSPACE; owned by the caller, overwritten by the call,
 *           and must not be shared with a call running concurrently
 * Body / tail selection, rotation and scale are as in kvq_decode_attention.
 */
KVQ_API kvq_status kvq_prefill_attention(const kvq_cache* c, const void* q, int32_t q_dtype,
                                 int32_t n_q_heads, int32_t n_tokens, const int32_t* q_pos0,
                                 int32_t causal, int32_t chunk, float scale, void* out,
                                 int32_t out_dtype, void* workspace, size_t ws_bytes,
                                 void* stream);

/*
 * Inspection of stored tokens (test aid): the stored blocks in the GGUF
 * array-of-structs byte order, which rotation leaves unchanged (velog
 * "fix-kv-cache-quantization-outliers", section 적용 및 배경 기술), and their
 * dequantized values, optionally rotated back (section 아다마르 회전).
 *   which          0 = K body, 1 = V body, 2 = K tail, 3 = V tail
 *   t0, count      positions [t0, t0+count) of (seq, kv_head); body positions
 *                  must lie below max_ctx; tail reads slot p % tail_len
 *   original_basis non-zero: rotate the values back when that side is rotated
 *   out            device float [count][head_dim] (NULL allowed)
 *   blocks_ggml    device bytes [count][head_dim/32][block bytes] or NULL: the
 *                  body blocks in GGUF array-of-structs byte order (body only;
 *                  18, 20, 22, 24, 34 bytes for q4_0, q4_1, q5_0, q5_1, q8_0)
 * No range check against seq_len: positions that were never written return
 * whatever the planes hold.
 */
KVQ_API kvq_status kvq_dequant_debug(const kvq_cache* c, int32_t seq, int32_t kv_head, int32_t which,
                             int32_t t0, int32_t count, int32_t original_basis, float* out,
                             void* blocks_ggml, void* stream);

/*
 * Synchronizes `stream`, reads and clears the cache's device status word 0
 * (raw bits to *device_bits, a host pointer, if non-NULL) and reports:
 * KVQ_ERR_CUDA for a pending CUDA error, KVQ_ERR_TIMEOUT or
 * KVQ_ERR_DEVICE_RANGE for status bits, else KVQ_OK.
 */
KVQ_API kvq_status kvq_sync_status(const kvq_cache* c, void* stream, uint32_t* device_bits);

/*
 * Test aid for the failure path: launches one CTA that waits on a shared-memory
 * barrier nothing ever completes, with the same bounded wait the kernels use
 * (limit_cycles clock cycles, 1 .. 2^31), and sets KVQ_DEV_ERR_TIMEOUT in the
 * cache's status word when it gives up.  The kernel then exits normally, so the
 * context stays usable; kvq_sync_status reports KVQ_ERR_TIMEOUT.  Asynchronous.
 */
KVQ_API kvq_status kvq_selftest_wait_timeout(const kvq_cache* c, int64_t limit_cycles, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
