/*
 * kvq.h -- C ABI of the GB300 (sm_103a) low-bit KV-cache library.
 *
 * The library implements the data-parallel hot path of KIVI-style asymmetric
 * 2/4-bit KV-cache quantization and decode attention read directly from the
 * quantized cache:
 *
 *   - keys quantized per channel in groups of 32 tokens, values per token,
 *     each slice with an fp32 (scale, min) pair and codes in [0, 2^b - 1]
 *     ("KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
 *     second paragraph; "KV cache quantization", "Keys are harder than
 *     values");
 *   - the newest tokens (fewer than R) kept in an fp16 window that is
 *     quantized in blocks of R tokens when it fills (KIVI page, third
 *     paragraph);
 *   - optionally keys stored before RoPE with RoPE applied after
 *     dequantization, and the first token kept in fp16 as an attention sink
 *     ("KV cache quantization", "Keys are harder than values" and "What they
 *     report");
 *   - options of the cache descriptor below: keys grouped per token (the
 *     baseline KIVI compares against), per-vector dense-and-sparse outlier
 *     entries (KVQuant), a Walsh-Hadamard rotation of every token before it
 *     is quantized, and a block-paged layout of the group blocks.
 *
 * Conventions shared by every entry point:
 *   - All buffer pointers are DEVICE pointers owned by the caller.  The
 *     library allocates no memory and never synchronizes; work is enqueued on
 *     the CUDA stream passed as `stream` (a cudaStream_t, NULL = legacy
 *     default stream).
 *   - fp16 data is passed as uint16_t bit patterns (IEEE binary16).
 *   - Return value: KVQ_OK (0) or a negative KVQ_ERR_* code.  Arguments are
 *     validated before anything is launched; on error nothing is enqueued.
 *     Errors found on the device (lengths past capacity, a bounded wait that
 *     gave up) are OR-ed into the optional device word `status`.
 *   - No C++ exception and no abort crosses this boundary.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_OK                 0
#define KVQ_ERR_INVALID_ARG   -1  /* null pointer, negative size, bad geometry   */
#define KVQ_ERR_UNSUPPORTED   -2  /* head_dim != 128, bits not 2/4, group != 32, ... */
#define KVQ_ERR_CAPACITY      -3  /* max_new / max_len larger than capacity       */
#define KVQ_ERR_WORKSPACE     -4  /* workspace null or smaller than required      */
#define KVQ_ERR_ALIGNMENT     -5  /* a buffer not aligned as documented           */
#define KVQ_ERR_CUDA          -6  /* a CUDA launch failed                         */

/* bits OR-ed into *status by device code */
#define KVQ_STATUS_CAPACITY    1  /* seq_len + new_len > capacity: sequence skipped */
#define KVQ_STATUS_BAD_LEN     2  /* new_len < 0 or > max_new: sequence skipped     */
#define KVQ_STATUS_TIMEOUT     4  /* a bounded pipeline wait gave up                */
#define KVQ_STATUS_MAX_LEN     8  /* seq_len > max_len at kv_decode_attn: row zeroed */
#define KVQ_STATUS_BAD_BLOCK  16  /* a block-table entry outside [0, num_blocks):
                                     its group was not written (append) or pool
                                     block 0 was read in its place (decode)   */
#define KVQ_STATUS_BOUNDS     32  /* builds compiled with KVQ_DEBUG_BOUNDS only:
                                     an index computed on the device fell
                                     outside its buffer; the access was skipped */

/* which buffer for kvq_buffer_bytes() */
#define KVQ_BUF_BLOCKS   0
#define KVQ_BUF_K_RES    1
#define KVQ_BUF_V_RES    2
#define KVQ_BUF_K_SINK   3
#define KVQ_BUF_V_SINK   4
#define KVQ_BUF_SEQ_LEN  5
#define KVQ_BUF_BLOCK_TABLE 6  /* paged layout only */

/*
 * Cache descriptor.  Plain data; every pointer is a caller-owned device
 * buffer sized by kvq_buffer_bytes().
 *
 *   blocks   [S][Hkv][max_groups][block_bytes] u8, 128-byte aligned (may be
 *            NULL when max_groups is 0).  One
 *            block holds one group of 32 quantized tokens of one (sequence,
 *            KV head): K codes (32*D*b/8 B, token rows), V codes (same size,
 *            channel rows), K scale fp32[D], K min fp32[D], V scale fp32[32],
 *            V min fp32[32].  A code tile (keys: rows = 32 tokens, cols =
 *            D channels; values: rows = D channels, cols = 32 tokens) is 32
 *            lanes x W 32-bit little-endian words; element (row, col) is in
 *            lane 4*(row%8) + (col%8)/2, word (P*KT + kt)*(4/nu) + tau/nu at
 *            bit 16*(col%2) + 8*((col/8)%2) + b*(tau%nu), where mt = row/16,
 *            tau = 2*(mt%2) + (row/8)%2, P = mt/2, kt = col/16, KT = cols/16,
 *            nu = 8/b; word w of lane l sits at byte ((w/4)*32 + l)*16 +
 *            (w%4)*4 of the tile.
 *            max_groups = floor((capacity - num_sink) / residual) * residual / 32.
 *   k_res, v_res    [S][Hkv][residual][D] fp16, the full-precision window
 *                   (pre-RoPE keys when pre_rope).  16-byte aligned.
 *   k_sink, v_sink  [S][Hkv][num_sink][D] fp16 (may be NULL when num_sink
 *                   is 0).  16-byte aligned.
 *   seq_len  [S] int32: tokens stored per sequence.  The caller zeroes it
 *            for an empty cache; kv_quant_append advances it.
 *   status   optional device int32 (may be NULL), see KVQ_STATUS_*.
 *   block_table  optional device int32 [S][Hkv][max_groups] (may be NULL).
 *            When set the layout is paged: `blocks` is a pool of num_blocks
 *            blocks and logical group g of (s, h) lives in pool block
 *            block_table[(s*Hkv + h)*max_groups + g].  The caller assigns
 *            the entries (a paged serving engine hands out pool blocks as
 *            sequences grow) before the appends that fill them; only groups
 *            below seq_len are read.  An entry outside [0, num_blocks) is
 *            never dereferenced: KVQ_STATUS_BAD_BLOCK is set.  4-byte
 *            aligned.  NULL: the contiguous layout above.
 *
 * Token p of a sequence is in the sink if p < num_sink.  The remaining
 * n = L - num_sink tokens form the stream: the first Lq = n - (n mod
 * residual) are quantized (Lq/32 blocks), the last n mod residual sit in the
 * window at slots 0.. in order.
 *
 * hadamard (the training-free rotation lever of "2-Bit KV Cache
 * Quantization: Memory You Save, Recall You Risk", "Method map: three ways
 * to shrink the cache"): a token's D-vector x is quantized as y = fp16(H x
 * / D), H the Sylvester Walsh-Hadamard matrix (H[i][j] = (-1)^popcount(i &
 * j)), evaluated as the fast transform in fp32 with strides 1, 2, ..., D/2
 * in that order (each butterfly (a, b) -> (a + b, a - b)), then scaled by
 * 1/D and rounded to fp16; |y| <= max |x|.  The blocks hold the codes of y;
 * the sink and the window keep tokens as given.  Decode scores the groups
 * with H q and rotates their weighted value sum back by H (H H = D I), so
 * its output is attention over x_hat = H y_hat; kv_dequant returns x_hat.
 *
 * outliers (per-vector dense-and-sparse, "KV cache quantization", "What
 * they report", KVQuant paragraph): in every quantization slice (a key
 * channel's 32 tokens of a group, or a token's D channels for per-token
 * keys and for values) the element of largest magnitude (the first in slice
 * order on ties) is the outlier.  The slice's min and scale come from the
 * other elements, the outlier's code is 0, and the block gains, after V
 * min, one 32-bit entry per key slice (D, or 32 with per-token keys) and
 * then one per value token (32): the outlier's fp16 bits in bits 0-15 and
 * its index within the slice (token, or channel) at bit 16.  The
 * dequantized outlier is its fp16 value.
 */
typedef struct kvq_cache {
  int32_t  num_seqs;       /* S, >= 1                                   */
  int32_t  num_kv_heads;   /* Hkv, >= 1                                 */
  int32_t  head_dim;       /* D, must be 128                            */
  int32_t  bits;           /* 2 or 4                                    */
  int32_t  group;          /* tokens per key group, must be 32          */
  int32_t  residual;       /* R: 32, 64, 96 or 128                      */
  int32_t  num_sink;       /* 0 or 1                                    */
  int32_t  pre_rope;       /* 1: keys stored pre-RoPE, rotated at read  */
  float    rope_theta;     /* RoPE base (e.g. 10000), used if pre_rope  */
  int32_t  capacity;       /* max tokens per sequence, >= 1             */
  int32_t  key_per_token;  /* 0: keys grouped per channel over 32 tokens;
                              1: per token over its D channels (the
                              baseline KIVI compares against; not with
                              pre_rope)                                 */
  int32_t  num_blocks;     /* pool size when block_table is set         */
  int32_t  hadamard;       /* 1: every key and value token is rotated by
                              the Walsh-Hadamard transform before it is
                              quantized (see below; not with pre_rope)  */
  int32_t  outliers;       /* 1: dense-and-sparse blocks (see below; not
                              with pre_rope or hadamard)                */
  uint8_t  *blocks;
  uint16_t *k_res, *v_res;
  uint16_t *k_sink, *v_sink;
  int32_t  *seq_len;
  int32_t  *status;
  int32_t  *block_table;   /* NULL: contiguous blocks                    */
} kvq_cache;

/* Sizing helpers (plumbing of this library; the pages define no interface).
 *
 * Bytes of one group block (3328 at 2-bit, 5376 at 4-bit for D = 128 with
 * per-channel keys; 2560 / 4608 with per-token keys; plus 4 * (D + 32), or
 * 4 * 64 with per-token keys, for dense-and-sparse blocks); 0 for an
 * unsupported (bits, head_dim) or a flag other than 0 / 1. */
int32_t kvq_block_bytes(int32_t bits, int32_t head_dim, int32_t key_per_token, int32_t outliers);

/* Quantized groups per (sequence, KV head) the cache can hold; -1 on bad
 * geometry. */
int32_t kvq_max_groups(const kvq_cache *cache);

/* Size in bytes of buffer `which` (KVQ_BUF_*); 0 for a buffer that is not
 * needed (the sink when num_sink is 0); -1 on bad geometry. */
int64_t kvq_buffer_bytes(const kvq_cache *cache, int32_t which);

/*
 * kv_quant_append -- append new tokens to every sequence.
 *
 * Source: KIVI page, second and third paragraphs (per-channel keys in
 * 32-token groups, per-token values, fp16 window of the newest tokens
 * quantized in blocks of R when it fills); "KV cache quantization", "What
 * they report" (first token in fp16).
 *
 *   k_new, v_new  [S][Hkv][max_new][D] fp16, 16-byte aligned; token j of
 *                 sequence s is k_new[s][h][j] for j < new_len[s] (pre-RoPE
 *                 keys when pre_rope).  Read only.
 *   new_len       device int32 [S], 0 <= new_len[s] <= max_new.
 *   max_new       host bound on new_len, 0 <= max_new <= capacity.
 *
 * New tokens take positions seq_len[s] .. seq_len[s] + new_len[s] - 1.
 * Positions below num_sink fill the sink; the rest enter the window, and each
 * time the window holds `residual` tokens its contents are quantized into
 * residual/32 blocks (scale = (max - min) / (2^b - 1) in fp32, code =
 * round-half-even of (x - min) / scale by IEEE fp32 subtract and divide,
 * clamped; scale 0 gives code 0) and the window empties.  The result is the
 * same for any split of a token stream into appends.  A sequence whose
 * new_len is out of range or would exceed capacity is left unchanged and the
 * matching KVQ_STATUS_* bit is set.  When max_new <= residual (at most one
 * window fills), capacity < 2^22 and num_kv_heads < 512, enqueues one
 * kernel, which counts its finished blocks in the high bits of
 * seq_len while it runs (seq_len is exact again when the kernel ends);
 * otherwise two kernels (quantize, then copy and advance seq_len).
 */
int kv_quant_append(const kvq_cache *cache, const uint16_t *k_new,
                    const uint16_t *v_new, const int32_t *new_len,
                    int32_t max_new, void *stream);

/*
 * kv_decode_workspace_bytes -- scratch size for kv_decode_attn (plumbing of
 * this library's split-K schedule; not on the pages).
 *
 *   num_q_heads  query heads (a multiple of num_kv_heads, ratio 1, 2 or 4).
 *   max_len      host bound on every seq_len at the time of the call
 *                (1 <= max_len <= capacity); pass capacity if unknown.
 * Returns bytes (a multiple of 256), or -1 on invalid arguments.
 */
int64_t kv_decode_workspace_bytes(const kvq_cache *cache, int32_t num_q_heads,
                                  int32_t max_len);

/*
 * kv_decode_attn -- attention of one query token per (sequence, query head)
 * over that sequence's whole cache: sink, quantized groups and window.
 *
 * Source: "KV cache quantization", "Keys are harder than values" (the
 * grouped part and the full-precision part are combined when computing
 * attention scores; keys stored pre-RoPE are rotated after dequantization).
 *
 *   q       [S][Hq][D] fp16 (already rotated for its own position when
 *           keys are stored pre-RoPE); query head j reads KV head
 *           j / (Hq / Hkv).
 *   softmax_scale  multiplier of q.k; <= 0 selects 1/sqrt(D).
 *   out     [S][Hq][D] fp16, written for every row (zeros when seq_len is 0).
 *   workspace, workspace_bytes  device scratch of at least
 *           kv_decode_workspace_bytes(cache, num_q_heads, max_len) bytes,
 *           256-byte aligned, owned by the library between calls.  It must
 *           be zero-filled before its first use with a given cache geometry
 *           and num_q_heads: the call's merge counters live in it, and every
 *           call that ends without KVQ_STATUS_TIMEOUT leaves them zero again
 *           (so no clearing step runs per call).  After a timeout, or before
 *           reusing it for another geometry, zero it again.
 *   max_len host bound on every seq_len (sizes the RoPE table); a
 *           sequence longer than max_len gets a zero output row and sets
 *           KVQ_STATUS_MAX_LEN.
 *
 * Keys are k_hat = code * scale + min (pre-RoPE keys then rotated by
 * rotate-half RoPE at their absolute position); values likewise.  The work
 * of all (sequence, KV head) pairs -- 32-token passes over the fp16 sink and
 * window, then packed groups -- is cut into equal contiguous ranges, one per
 * warp; the kernel dequantizes in registers, forms scores, runs an online
 * softmax over each range, and the last range of a pair to finish merges its
 * partials (log-sum-exp).  Every option of the descriptor is honoured:
 * per-token key scales, outlier entries (each adds q . (x - min) to its
 * token's score, or p (x - min) to its channel's output), the rotation
 * (groups scored with H q, their value sum rotated back), and the block
 * table.  Enqueues the decode kernel, plus a plan kernel (work prefix over
 * the sequences) when S > 256 and a RoPE table kernel when pre_rope.
 */
int kv_decode_attn(const kvq_cache *cache, int32_t num_q_heads,
                   const uint16_t *q, float softmax_scale, uint16_t *out,
                   void *workspace, size_t workspace_bytes, int32_t max_len,
                   void *stream);

/*
 * kv_decode_attn_noalloc -- kv_decode_attn for callers that cannot allocate
 * device memory.
 *
 * The pages describe no such interface; it has no counterpart in the method.
 * It exists for callers that cannot hand the library a workspace: code
 * running inside a host program whose device memory is owned and planned by
 * another runtime (a plugin in an inference server or engine with a fixed
 * memory budget), and paths where a cudaMalloc is not allowed because it can
 * synchronize the device.
 *
 * Same arguments and results as kv_decode_attn, minus the workspace: the
 * arguments are checked first and give the same error codes.  The scratch
 * is a 16 MiB array compiled into this library (every GPU that loads the
 * library keeps it until the process exits).  A valid call whose
 * kv_decode_workspace_bytes(cache, num_q_heads, max_len) exceeds 16 MiB
 * returns KVQ_ERR_WORKSPACE and enqueues nothing.  Nothing is allocated: no
 * cudaMalloc, no cudaFree, no allocating library call.
 *
 * Every call looks up the array's device address in the current device's
 * context (nothing is cached, so a cudaDeviceReset in between is harmless).
 * The first lookup on a device loads the array's module there: make the
 * first call on each device before any stream capture.  All calls on a
 * device share the one array and it keeps
 * the previous call's contents (each call clears the part that must start
 * at zero, on its own stream, before using it): calls
 * whose work overlaps on the GPU (different streams, or different host
 * threads without ordering) race on the scratch and must be serialized by
 * the caller.
 */
int kv_decode_attn_noalloc(const kvq_cache *cache, int32_t num_q_heads,
                           const uint16_t *q, float softmax_scale,
                           uint16_t *out, int32_t max_len, void *stream);

/*
 * kv_dequant -- test aid: write the dequantized cache.
 *
 * Source: "KV cache quantization", "What they report" (asymmetric
 * quantization: a value is rebuilt as code * scale + min from its slice's
 * scale and minimum); "KIVI: A Tuning-Free Asymmetric 2bit Quantization for
 * KV Cache", second paragraph (which slice a key or value code belongs to).
 *
 *   k_out, v_out  [S][Hkv][capacity][D] fp32.  For every stored position p <
 *                 seq_len[s]: sink and window tokens are converted exactly,
 *                 quantized tokens are code * scale + min (one fused
 *                 multiply-add in fp32), an outlier entry's position its fp16
 *                 value, and with the rotation the group rows are rotated
 *                 back (H y_hat in fp32); keys are pre-RoPE.  Positions at or
 *                 past seq_len are not written.  Through a block table, a
 *                 group whose entry lies outside the pool is not written and
 *                 sets KVQ_STATUS_BAD_BLOCK.
 */
int kv_dequant(const kvq_cache *cache, float *k_out, float *v_out, void *stream);

/* Message for a KVQ_ERR_* code (static storage).  Plumbing; not on the
 * pages, like the two calls below. */
const char *kvq_strerror(int err);

/* Number of kernels this library has launched in this process (for
 * launch accounting in benchmarks). */
uint64_t kvq_launch_count(void);

/* Warps a decode launch cuts its work into (1..2560); 0 restores the
 * built-in choice (every resident warp of the device, at most 2560).
 * Affects kv_decode_attn calls made afterwards in this process; the
 * workspace size does not depend on it.  Returns KVQ_OK or
 * KVQ_ERR_INVALID_ARG. */
int kvq_set_decode_warps(int32_t warps);

/* Test aid (not on the pages) for the bounded waits of the decode kernel.
 * limit_cycles: SM clock cycles a pipeline wait may last before it gives up,
 * records KVQ_STATUS_TIMEOUT, lets its own copies in flight land (those
 * waits keep the default bound) and ends its warp's work; 0 restores the
 * default of about two seconds (4e9 cycles).  wait_before_fetch = 1 makes
 * each warp's first wait come before its first copy is issued, on a barrier
 * that nothing completes, so that it runs out: this is how tests exercise the
 * timeout path without a fault (in normal operation every copy of a valid
 * block lands).  It needs limit_cycles > 0.  Affects kv_decode_attn calls made
 * afterwards in this process.  Returns KVQ_OK, or KVQ_ERR_INVALID_ARG for a
 * limit that is negative or above the default, or a bad flag. */
int kvq_set_wait_test(int64_t limit_cycles, int32_t wait_before_fetch);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
