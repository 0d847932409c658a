/*
 * fa_rows.h — row-indexed flash attention over a unified KV pool (C ABI).
 *
 * The operation ("llama.cpp 0.9.0 inference boundaries", section 1, the
 * ggml_flash_attn_ext_rows paragraph): every sequence's K/V rows share one
 * storage pool; each query slice carries its own integer kv_rows list naming
 * the pool rows it attends to; a negative row index is padding whose mask is
 * minus infinity.  The next paragraph of that section fixes that the result is
 * exact attention over the listed rows, not a lossy summary.
 *
 * Paged KV with 64-token pages and an INT8 cache: the v100llm article,
 * sections 1-2 ("FlashAttention 1.5 SM70 kernels", "Paged KV cache").
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers, row-major and contiguous, owned
 *    by the caller.  The library never allocates device memory, never
 *    synchronises, and enqueues all work on the given stream.
 *  - Argument errors are detected on the host before anything is launched and
 *    returned as a status; nothing is thrown across this boundary.  A failed
 *    launch returns FA_ERR_CUDA; fa_last_error() then names the CUDA error.
 *  - Row indices are NOT range-checked by the attention calls (that would cost
 *    a pass over the lists); fa_rows_validate() checks them on the device and
 *    reports through a status word, without trapping.
 *  - Every wait inside the tensor-core kernels is bounded in time (1 s by
 *    default, see fa_set_wait_limit_ns).  A wait that runs out is treated as a
 *    hang: the kernel leaves its pipeline, lets its own copies and MMAs drain,
 *    frees its tensor memory and sets FA_WS_WAIT_EXPIRED in the status word of
 *    the call's workspace (fa_rows_status reads it).  That call's outputs are
 *    then invalid; the call itself has already returned FA_OK, since the wait
 *    runs on the GPU after the launch.
 */
#ifndef FA_ROWS_H
#define FA_ROWS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, inconsistent shape        */
  FA_ERR_UNSUPPORTED = 2,  /* valid but outside the shapes/dtypes built here   */
  FA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required        */
  FA_ERR_INDEX_OOB = 4,    /* reported by fa_rows_validate through its status   */
  FA_ERR_CUDA = 5,         /* a CUDA launch or runtime call failed              */
  FA_ERR_WAIT_EXPIRED = 6  /* not returned by a launch: the code to report when
                            * a workspace status word holds FA_WS_WAIT_EXPIRED */
} fa_status;

/* Bits of the workspace status word (the first uint32 of every decode and
 * prefill workspace).  Sticky: set by any call on that workspace, cleared only
 * by fa_rows_workspace_init or fa_rows_status(..., clear = 1). */
#define FA_WS_WAIT_EXPIRED 1u  /* a bounded pipeline wait ran out; that call's outputs are invalid */

typedef enum fa_dtype { FA_F16 = 0, FA_BF16 = 1, FA_F32 = 2, FA_I8 = 3, FA_I4 = 4, FA_F8E4M3 = 5 } fa_dtype;

typedef enum fa_mask_kind {
  FA_MASK_NONE = 0,
  /* additive fp32 mask [S, Nq, L], aligned with list POSITION j (not pool row);
   * minus infinity removes an entry.  Section 1's "corresponding mask". */
  FA_MASK_DENSE = 1,
  /* bottom-right causal: the slice's Nq queries are the last Nq positions of
   * its n_s list entries, so query i sees list positions j <= n_s - Nq + i. */
  FA_MASK_CAUSAL = 2
} fa_mask_kind;

/*
 * Arguments of one row-indexed attention call.
 *
 *   q        [S, Nq, Hq, D]     FA_F16 or FA_BF16
 *   k, v     [R, Hkv, D]        the unified pool: FA_F16/FA_BF16 (same as q),
 *                               FA_I8 (int8 codes, then k_scale/v_scale), or
 *            [R, Hkv, D/2]      FA_I4 (two 4-bit codes per byte, element 2t in
 *                               the low nibble of byte t; D = 128 only), or
 *            [R, Hkv, D]        FA_F8E4M3 (OCP E4M3 bytes; D = 128 only)
 *   k_scale, v_scale            quantised pools only: fp16 bit patterns laid out
 *                               [R/64, Hkv, 64], i.e. the scale of (row r,
 *                               head g) sits at ((r/64)*Hkv + g)*64 + r%64;
 *                               value = code * scale (R must be a multiple of 64)
 *   kv_rows  [S, L] int32       pool row of list entry j of slice s; negative =
 *                               padding.  Duplicates count once per occurrence.
 *   kv_len   [S] int32 or NULL  n_s: entries at positions >= kv_len[s] are
 *                               padding (NULL: n_s = L)
 *   mask     [S, Nq, L] fp32    FA_MASK_DENSE only
 *   out      [S, Nq, Hq, D]     FA_F32, FA_BF16 or FA_F16
 *   lse      [S, Nq, Hq] fp32   optional natural-log log-sum-exp of the logits
 *
 * Query head h reads KV head h / (Hq/Hkv).  Logit of entry j for query i:
 * scale * <q, K[row]> (+ mask[s,i,j]).  A query with no visible entry gets
 * out = 0 and lse = -inf.
 *
 * n_valid_hint: optional host-side count of listed entries summed over all
 * slices (0 = unknown); it only steers how the list is split across SMs.
 */
typedef struct fa_rows_args {
  const void* q;
  fa_dtype q_dtype;
  const void* k;
  const void* v;
  fa_dtype kv_dtype;
  const uint16_t* k_scale;
  const uint16_t* v_scale;
  int64_t n_pool_rows;
  const int32_t* kv_rows;
  int32_t list_len;
  const int32_t* kv_len;
  fa_mask_kind mask_kind;
  const float* mask;
  float scale;
  void* out;
  fa_dtype out_dtype;
  float* lse;
  int32_t S, Nq, Hq, Hkv, D;
  int64_t n_valid_hint;
} fa_rows_args;

/*
 * Bytes of scratch (a device buffer, 256-byte aligned) that fa_rows_decode /
 * fa_rows_prefill need for these arguments; at least 256.  Layout: bytes
 * [0, 256) are the status block, whose first uint32 is the status word
 * (FA_WS_WAIT_EXPIRED; the next words are the calls' own scratch); decode
 * then holds one arrival counter per (slice, KV
 * head) and, when the list is split over several CTAs, the per-split partial
 * results.  The buffer must be ZERO-FILLED once after allocation
 * (fa_rows_workspace_init); every call leaves the counters at zero again, an
 * aborted one included.  One workspace must not be used by two calls that can
 * run at the same time.  Returns 0 and sets fa_last_error() on invalid
 * arguments.
 */
size_t fa_rows_workspace_size(const fa_rows_args* a, int is_prefill);
fa_status fa_rows_workspace_init(void* ws, size_t ws_bytes, fa_stream_t stream);

/*
 * Kernel launches one fa_rows_decode call with these arguments makes: 1, or 2
 * when the plan merges the list's splits in a kernel of its own (a
 * latency-bound 16-bit decode: one wave of CTAs, each over at most four
 * tiles), 0 when there is nothing to do; -1 (and fa_last_error()) on invalid
 * arguments.  Host-only: no device work, no stream.
 */
int fa_rows_decode_launches(const fa_rows_args* a);

/*
 * Enqueues on `stream` a copy of the workspace's status word into *d_status
 * (a device uint32) and, if `clear` is non-zero, then zeroes the word.  The
 * caller reads d_status once the stream has reached this point; a non-zero
 * FA_WS_WAIT_EXPIRED bit means a call on this workspace since the word was
 * last cleared had a pipeline wait run out, so its outputs are invalid.
 * ws_bytes must be at least 256.  No counterpart on the pages: the pages
 * describe no failure path.
 */
fa_status fa_rows_status(void* ws, size_t ws_bytes, uint32_t* d_status, int clear, fa_stream_t stream);

/*
 * Diagnostic: the time limit, in nanoseconds, of every bounded pipeline wait
 * in kernels launched after this call by any thread of the process (0 restores
 * the default of 1 s).  Lowering it to a few nanoseconds makes waits run out
 * on purpose, which exercises the abort path and the status word in tests.
 * The drain waits of an aborting kernel keep the 1 s default.
 * No counterpart on the pages.
 */
fa_status fa_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Decode: few query rows per slice (Nq * Hq/Hkv <= 32).  Split-KV over the
 * list, online softmax per split, cross-split merge inside the same launch
 * (by the last split of each (slice, KV head) to finish), or, for a
 * latency-bound 16-bit decode, in a second kernel enqueued right after it on
 * the same stream (fa_rows_decode_launches tells which).
 * D in {64, 128, 256}; Hq/Hkv a power of two up to 32 (times Nq).
 */
fa_status fa_rows_decode(const fa_rows_args* a, void* ws, size_t ws_bytes, fa_stream_t stream);

/*
 * Decode for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call; it exists for hosts that may not call cudaMalloc
 * (or any allocating routine) where they run attention: code inside a custom
 * device allocator or its callbacks, plugins whose framework owns every device
 * allocation, and latency-critical paths that cannot afford an allocation or
 * its failure.  Same arguments and results as fa_rows_decode, but the
 * split-merge scratch comes from a static device array of 16 MiB inside this
 * library (held on every GPU that loads it, until the process exits).
 * Arguments whose scratch would exceed 16 MiB are rejected with
 * FA_ERR_WORKSPACE before anything is launched.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress), so make that
 * first call before any stream capture.  Each call zero-fills the part of the
 * array it uses; all calls share the array, so calls that overlap on the GPU
 * (other streams or threads) race and must be serialised by the caller.
 */
fa_status fa_rows_decode_static(const fa_rows_args* a, fa_stream_t stream);

/*
 * Prefill: many query rows per slice.  QK^T and PV on the tensor cores
 * (tcgen05, accumulators in tensor memory), K/V tiles gathered by row index.
 * D = 128, FA_BF16 or FA_F16 for q and the pool; Nq >= 1.  The workspace
 * (fa_rows_workspace_size(a, 1) = 256 bytes, zero-filled once) is required:
 * it holds the status word; a NULL ws is rejected with FA_ERR_WORKSPACE.
 * bf16 pools: the call first scans the listed V rows (one extra kernel, one
 * read of them) and writes words 1-3 of the status block as its own scratch:
 * when no listed V value is beyond f16's range (finite, 65536 or more) and
 * at most a quarter of the 128-entry KV tiles are gathered rather than one
 * contiguous pool run, V tiles are converted to f16 in shared memory and P
 * enters the PV product as one f16 value (11 significant bits; a bf16 V value
 * below 2^-14 in magnitude becomes an f16 subnormal, within 2^-25 of it);
 * otherwise V stays bf16 and P is the pair rn(P) + rn(P - rn(P)).
 */
fa_status fa_rows_prefill(const fa_rows_args* a, void* ws, size_t ws_bytes, fa_stream_t stream);

/*
 * Range check of the lists (section 1: negative = padding; anything else must
 * name a pool row).  d_status is a device int64[2] that this call overwrites:
 * [0] = number of entries with kv_rows >= n_pool_rows (within kv_len),
 * [1] = flat index s*L + j of the first such entry, or -1.
 * Returns FA_OK once the check is enqueued; the caller reads d_status.
 */
fa_status fa_rows_validate(const fa_rows_args* a, int64_t* d_status, fa_stream_t stream);

/*
 * Page tables -> row lists (v100llm article, section 2: 64-token pages).
 * page_table [n_seq, max_pages] int32 page ids; seq_len [n_seq] int32 (device).
 * kv_rows [n_seq, list_len] is written as page_id*page_size + j%page_size for
 * j < seq_len[s] and -1 elsewhere.  seq_len values above max_pages*page_size
 * are clamped to it.
 */
fa_status fa_kv_page_table_to_rows(const int32_t* page_table, int32_t max_pages, const int32_t* seq_len,
                                   int32_t n_seq, int32_t page_size, int32_t* kv_rows, int32_t list_len,
                                   fa_stream_t stream);

/*
 * INT8 KV quantisation, per (row, KV head) with an fp16 scale (value = q*s):
 * s = fp16_rne(min(amax/127, 65504)) with amax/127 one fp32 division;
 * q = clamp(rint_half_even(x/s), -127, 127) with x/s one fp32 division;
 * s = 0 gives q = 0.
 *   x        [n_rows, Hkv, D] FA_F16 or FA_BF16 (x_dtype)
 *   dst_rows [n_rows] int32 pool rows to write, negative or >= R = skip;
 *            NULL = row i
 *   q        [R, Hkv, D] int8 pool; scale the fp16 layout of fa_rows_args.
 * This is also the KV append of a ubatch into an INT8 pool.
 */
fa_status fa_kv_quantize_int8(const void* x, fa_dtype x_dtype, int64_t n_rows, int32_t Hkv, int32_t D,
                              const int32_t* dst_rows, int8_t* q, uint16_t* scale, int64_t n_pool_rows,
                              fa_stream_t stream);

/* out[r, g, d] = float(q[r, g, d]) * float(scale of (r, g)), exact in fp32. */
fa_status fa_kv_dequantize_int8(const int8_t* q, const uint16_t* scale, int64_t n_rows, int32_t Hkv, int32_t D,
                                float* out, fa_stream_t stream);

/*
 * INT4 KV quantisation for the paged INT4 pool the v100llm article names
 * (section 2, "INT4/INT8 paged path"; it gives no rule): the INT8 rule above
 * with 7 in place of 127 (s = fp16_rne(min(amax/7, 65504)), codes in -7..7),
 * stored as two's-complement nibbles, element 2t in the low nibble of byte t.
 *   q        [R, Hkv, D/2] uint8 pool; scale the fp16 layout of fa_rows_args.
 * D must be even and <= 256; negative dst_rows entries are skipped.
 */
fa_status fa_kv_quantize_int4(const void* x, fa_dtype x_dtype, int64_t n_rows, int32_t Hkv, int32_t D,
                              const int32_t* dst_rows, uint8_t* q, uint16_t* scale, int64_t n_pool_rows,
                              fa_stream_t stream);

/* out[r, g, d] = float(nibble code) * float(scale of (r, g)), exact in fp32. */
fa_status fa_kv_dequantize_int4(const uint8_t* q, const uint16_t* scale, int64_t n_rows, int32_t Hkv, int32_t D,
                                float* out, fa_stream_t stream);

/*
 * FP8 E4M3 KV quantisation.  "llama.cpp 0.9.0 inference boundaries"
 * (section 4) adds the OCP FP8 E4M3 type in saturating mode and leaves its KV
 * use and scaling to later work; the rule here mirrors the INT8 one:
 * s = fp16_rne(min(amax/448, 65504)); code = E4M3 of x/s (one fp32 division,
 * round to nearest even, saturating to +-448, NaN -> 0x7f); s = 0 gives 0.
 *   q        [R, Hkv, D] E4M3 bytes; scale the fp16 layout of fa_rows_args.
 */
fa_status fa_kv_quantize_fp8(const void* x, fa_dtype x_dtype, int64_t n_rows, int32_t Hkv, int32_t D,
                             const int32_t* dst_rows, uint8_t* q, uint16_t* scale, int64_t n_pool_rows,
                             fa_stream_t stream);

/* out[r, g, d] = float(E4M3 value of q[r, g, d]) * float(scale of (r, g)), exact in fp32. */
fa_status fa_kv_dequantize_fp8(const uint8_t* q, const uint16_t* scale, int64_t n_rows, int32_t Hkv, int32_t D,
                               float* out, fa_stream_t stream);

/*
 * Sparse row-list builder (v100llm article, section 5: anchor + recent + sink
 * selection; the llama.cpp-v100 README's QSA reads such a subset of a long
 * context).  For each slice s with n = min(n_len[s], n_max) positions
 * (n_len NULL: n = n_max): positions 0 .. sinks-1, the k positions of
 * [sinks, n - recent) with the largest score[s, pos], and n-recent .. n-1,
 * in increasing position order, padded with -1.  Ties in score go to the
 * smaller position; a NaN score ranks below every number.  Slices with no
 * more than k middle positions list every position.
 *   score    [S, n_max] fp32, caller-provided (the learned indexer that would
 *            produce it is not part of this library)
 *   row_map  [S, n_max] int32 position -> pool row, or NULL (row = position)
 *   kv_rows  [S, list_len] int32 output; list_len >= sinks + recent + k
 *   ws       scratch of fa_kv_sparse_rows_workspace_size(S, n_max) bytes
 *            (16-byte aligned; its contents need no initialisation): each
 *            slice is then spread over blocks of 8192 positions (several
 *            launches on the stream).  NULL: one CTA per slice, no scratch.
 * The output is bit-exact (an integer selection) either way.
 */
size_t fa_kv_sparse_rows_workspace_size(int32_t S, int32_t n_max);
fa_status fa_kv_sparse_rows(const float* score, int32_t n_max, const int32_t* n_len, int32_t S, int32_t sinks,
                            int32_t recent, int32_t k, const int32_t* row_map, int32_t* kv_rows, int32_t list_len,
                            void* ws, size_t ws_bytes, fa_stream_t stream);

/*
 * KV append for 16-bit pools: pool[dst_rows[i]] = x[i] for i < n_rows
 * (negative dst = skip).  x and pool are [*, Hkv, D] of the same 16-bit dtype.
 */
fa_status fa_kv_append(const void* x, fa_dtype dtype, int64_t n_rows, int32_t Hkv, int32_t D,
                       const int32_t* dst_rows, void* pool, int64_t n_pool_rows, fa_stream_t stream);

const char* fa_status_string(fa_status s);
/* Text of the last error seen by the calling thread ("" if none). */
const char* fa_last_error(void);
/* Library build tag, e.g. "fa_rows sm_103a". */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_ROWS_H */
