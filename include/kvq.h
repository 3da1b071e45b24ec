/*
 * kvq.h -- C ABI of libkvq: an FP4 (E2M1 codes, one E4M3 scale per 16
 * channels) key/value cache, an FP8 E4M3 sliding-window cache beside it, and
 * the split-K decode attention that reads both back.
 *
 * Sources (page title, section):
 *   "Quantising the KV cache", section "Code": the block quantiser
 *       (s = RNE_e4m3(amax/6) saturating, s == 0 -> E4M3 min subnormal 2^-9,
 *       codes = RNE_e2m1(v/s) saturating) and the place of the quantised K/V
 *       between projection and an unchanged attention.
 *   "Quantising the KV cache", section "FP4 with a fine-grained scale" and
 *       section "Maths": E2M1 with an E4M3 scale per 16 costs 4.5 bits/number.
 *   "Quantising the KV cache", section "Concept": decode reads the whole cache
 *       for every new token, so decode time is mostly spent reading it.
 *   "KV Cache Quantisation", section "Common questions": the win holds only if
 *       the attention kernel handles the scales and dequantisation itself.
 *   "Week 6 -- FP4 KV Caches and Bounded Replay", "Overview": global KV goes
 *       ~4-bit, sliding-window (SWA) KV stays FP8.
 *
 * Conventions shared by every entry point
 *   - All pointers named d_* or documented as "device" are CUDA device memory
 *     owned by the caller.  The library allocates nothing at call time.  Two
 *     things are held by the library itself: a fixed 8 MiB device array on
 *     every device that loads it (the scratch of kvq_decode_attn_noalloc, used
 *     by that entry point only, whose calls must be serialised -- see its
 *     comment), and the process-wide wait limit a test can set with
 *     kvq_test_set_wait_limit_ns.  Apart from kvq_decode_attn_noalloc, calls
 *     on different streams with disjoint buffers are independent.
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  The return value reports only host-side
 *     argument checks and launch errors:
 *       KVQ_ERR_INVALID_ARGUMENT  a size, pointer or layout is invalid; nothing
 *                                 was enqueued.
 *       KVQ_ERR_UNSUPPORTED       valid but outside what the kernels handle
 *                                 (e.g. head_dim not 64/128 in decode); nothing
 *                                 was enqueued.
 *       KVQ_ERR_WORKSPACE         workspace too small; nothing was enqueued.
 *       KVQ_ERR_CUDA              a CUDA call or launch failed.
 *   - Data-dependent problems found on the device set bits (atomicOr) in the
 *     caller's int32 device word `d_err_flag` (may be NULL: then they are not
 *     reported).  Kernels never trap or assert; the offending element is
 *     skipped (append, dequant) or contributes nothing (decode).  Read the flag
 *     after synchronising the stream.
 *   - Key/value inputs are bf16; query heads h use kv head h / (Hq / Hkv).
 *
 * FP4 paged cache layout (format KVQ_FORMAT_FP4_E2M1_E4M3_G16).
 *   Codes: nibble = sign<<3 | E2M1 magnitude (0..7 -> 0, .5, 1, 1.5, 2, 3, 4,
 *   6); the sign of zero is kept.  Scales: one E4M3FN byte per 16-channel
 *   block of one token (never 0x00: an all-zero block stores 0x01).
 *   The pool `data` is uint8 [num_pages][num_kv_heads][page_size/G][group],
 *   G = min(page_size, 128) tokens per group, NB = head_dim/16 blocks, and one
 *   group of G tokens of one kv head is a contiguous block of G*9*head_dim/8
 *   bytes (4.5 bits per number), so a decode stage fetches it with one copy:
 *     K codes  [G][head_dim/2] at 0: byte j of token t holds channels 2j (low
 *              nibble) and 2j+1 (high nibble).
 *     K scales [G][NB] at G*head_dim/2.
 *     V codes  [G/2][head_dim] at G*(head_dim/2 + NB): row i holds tokens 2i
 *              (low nibbles) and 2i+1 (high nibbles), byte c = channel c.  The
 *              row's bytes are stored permuted so that decode reads them without
 *              shared-memory bank conflicts: head_dim 64 moves 8-byte chunk u to
 *              u ^ (((i >> 1) & 1) << 2); head_dim 128 and 256 move 16-byte chunk
 *              u to u ^ ((i & 3) << 1).
 *     V scales [G/2][NB][2] at G*(head_dim + NB): pair i, block j holds the
 *              scales of tokens 2i and 2i+1.
 *   Position p of sequence b lives in page page_table[b*max_pages_per_seq +
 *   p/page_size], slot p % page_size (group slot/G, token slot%G).  With
 *   page_table == NULL the cache is contiguous: page p/page_size of sequence b
 *   is b*max_pages_per_seq + p/page_size.
 *
 * NVFP4 cache (format KVQ_FORMAT_NVFP4): the FP4 layout above plus one fp32
 *   second-level scale per kv head, k_scale and v_scale: float [num_kv_heads]
 *   ("KV Cache Quantisation": FP8 or NVFP4 with the scales handled at read
 *   time).  Codes and block scales are those of x / S (fp32 division), and a
 *   value reads back as fp32(fp32(E2M1(code) * E4M3(s)) * S).  S is set from
 *   calibration tokens by kvq_fp8_set_scales (S = amax / (6*448), so the
 *   largest block lands on the top E4M3 scale and small tensors keep their
 *   resolution instead of underflowing the E4M3 scale).
 *
 * FP8 window cache layout (format KVQ_FORMAT_FP8_E4M3_HEAD), K in `data`, V in
 * `v_data`:
 *   uint8 [num_pages][num_kv_heads][page_size][head_dim], one E4M3FN byte per
 *   value; here num_pages counts rings (one per sequence b) and page_size is
 *   the window length W: position p of sequence b lives in slot p % W of ring b.
 *   k_scale, v_scale: float [num_kv_heads], one fp32 scale per kv head:
 *   value = fp32(E4M3(code) * scale).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_VERSION 1

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARGUMENT = 1,
    KVQ_ERR_UNSUPPORTED = 2,
    KVQ_ERR_WORKSPACE = 3,
    KVQ_ERR_CUDA = 4
} kvq_status;

/* Bits OR-ed into *d_err_flag by the kernels. */
#define KVQ_FLAG_NONFINITE 0x1 /* a key/value/query input held Inf or NaN */
#define KVQ_FLAG_PAGE_OOB 0x2  /* a page id outside [0, num_pages) or a page index
                                  outside [0, max_pages_per_seq) */
#define KVQ_FLAG_TIMEOUT 0x4   /* a bounded wait inside a kernel gave up (~2 s) */
#define KVQ_FLAG_BAD_LENGTH 0x8 /* a negative sequence length or start position */
#define KVQ_FLAG_BOUNDS 0x10    /* an index outside its buffer; raised only by a
                                   bounds-checked build of the library
                                   (-DKVQ_DEBUG_BOUNDS), which then skips the
                                   access */

typedef enum kvq_format {
    KVQ_FORMAT_FP4_E2M1_E4M3_G16 = 1,
    KVQ_FORMAT_FP8_E4M3_HEAD = 2,
    KVQ_FORMAT_NVFP4 = 3
} kvq_format;

typedef struct kvq_stream_opaque *kvq_stream; /* a cudaStream_t */

/* Description of one cache (K and V of one layer).  All buffers are device
 * memory owned by the caller; see the layouts above.  kvq_fp4_pool_bytes gives
 * the size of an FP4 pool. */
typedef struct kvq_cache {
    int32_t format;            /* kvq_format */
    int32_t num_kv_heads;      /* Hkv >= 1 */
    int32_t head_dim;          /* FP4: 64, 128 or 256; FP8: multiple of 16, <= 512 */
    int32_t page_size;         /* FP4: tokens per page, one of 16, 32, 64, 128, 256;
                                  FP8: window length W, 1..1024 */
    int64_t num_pages;         /* FP4: pages in the pool; FP8: number of rings */
    int32_t max_pages_per_seq; /* FP4: row length of page_table (or pages per
                                  sequence when contiguous); FP8: ignored */
    int32_t reserved;          /* must be 0 */
    const int32_t *page_table; /* FP4: device int32 [batch][max_pages_per_seq] or NULL;
                                  FP8: must be NULL */
    void *data;                /* FP4: the page pool; FP8: K codes (16-byte aligned) */
    void *v_data;              /* FP8: V codes (16-byte aligned); FP4: must be NULL */
    void *k_scale;             /* FP8, NVFP4: float [Hkv]; FP4: must be NULL */
    void *v_scale;             /* FP8, NVFP4: float [Hkv]; FP4: must be NULL */
} kvq_cache;

/*
 * kvq_append -- quantise n_new new tokens per sequence into `cache`.
 * ("Quantising the KV cache", section "Code": per 16-channel block, scale
 * RNE_e4m3(amax/6) saturating with 0 -> 2^-9, codes RNE_e2m1(v/s) saturating,
 * IEEE fp32 divisions; NVFP4 caches: the same on x / S_h; FP8 caches: code
 * RNE_e4m3(x / s_h) saturating.)
 *   cache       FP4, NVFP4 or FP8 cache (NVFP4 and FP8 caches need their
 *               scales set first, e.g. by kvq_fp8_set_scales).
 *   batch       number of sequences (rows of page_table / rings), >= 0.
 *   n_new       new tokens per sequence, >= 0.
 *   d_start_pos device int32 [batch]: position of each sequence's first new
 *               token; token t goes to position d_start_pos[b] + t.
 *   k, v        device bf16 [batch][n_new][num_kv_heads][head_dim], contiguous.
 * FP8 caches keep a ring of W slots: when n_new > W only the last W new
 * tokens are written (the earlier ones would be overwritten in the same call).
 * Device flags: NONFINITE (the block's codes and scale are whatever the
 * conversion produces), PAGE_OOB (token skipped), BAD_LENGTH (negative start;
 * sequence skipped).  Host errors: INVALID_ARGUMENT (bad cache or sizes, NULL
 * or non-16-byte-aligned k/v), UNSUPPORTED (FP4: n_new * num_kv_heads *
 * head_dim / 16 above 2^30 in one call; split the tokens over several calls).
 */
kvq_status kvq_append(const kvq_cache *cache, int32_t batch, int32_t n_new,
                      const int32_t *d_start_pos, const void *k, const void *v,
                      int32_t *d_err_flag, kvq_stream stream);

/*
 * kvq_fp8_set_scales -- set a cache's per-head fp32 scales from a calibration
 * set of tokens, over every value of kv head h in k (resp. v), 1 where
 * amax == 0: an FP8 window cache gets s_h = amax / 448 ("Week 6 -- FP4 KV
 * Caches and Bounded Replay": SWA KV stays FP8; "Quantising the KV cache"
 * table row "FP8 E4M3, one scale per tensor", here one scale per head); an
 * NVFP4 cache gets its second-level scales S_h = amax / (6*448).  Both are
 * fp32 divisions.
 *   k, v   device bf16 [batch][n][num_kv_heads][head_dim].
 * Writes cache->k_scale and cache->v_scale (float [Hkv]).  Device flags:
 * NONFINITE.
 */
kvq_status kvq_fp8_set_scales(const kvq_cache *cache, int32_t batch, int32_t n,
                              const void *k, const void *v, int32_t *d_err_flag,
                              kvq_stream stream);

/*
 * kvq_decode_workspace_bytes -- bytes of device workspace kvq_decode_attn
 * needs for these sizes on the current device (it depends on the device's SM
 * count).  Returns 0 for invalid sizes.
 */
size_t kvq_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim);

/*
 * kvq_decode_attn -- one decode step of attention for every sequence and
 * query head, reading keys and values from the FP4 cache (dequantised in the
 * kernel) and, when `swa` is given, the last min(W, T) positions from the FP8
 * window cache instead; one softmax over the union.  ("Quantising the KV
 * cache", section "Code": quantised K/V feed an unchanged attention;
 * "Concept": decode reads the whole cache.)
 *   out[b][h][:] = sum_t softmax_t(softmax_scale * q[b][h] . K^[b][t]) V^[b][t]
 *   global       FP4 or NVFP4 cache with head_dim 64 or 128 (NVFP4: the
 *                second-level scales multiply the scores and the values).
 *   swa          FP8 window cache with the same num_kv_heads/head_dim, or NULL.
 *   batch        sequences, >= 1.
 *   num_q_heads  Hq, a multiple of num_kv_heads with Hq/Hkv <= 8.
 *   d_seq_lens   device int32 [batch]: T_b, positions 0..T_b-1 are attended
 *                (T_b == 0 gives a zero output row).
 *   q            device bf16 [batch][num_q_heads][head_dim].
 *   softmax_scale scale applied to q.k (usually 1/sqrt(head_dim)), > 0.
 *   out          device float [batch][num_q_heads][head_dim].
 *   workspace    device scratch of at least kvq_decode_workspace_bytes(...)
 *                bytes, 16-byte aligned; needs no initialisation; must not be
 *                shared by calls that may run concurrently.
 * Device flags: PAGE_OOB (the page's tokens are left out), BAD_LENGTH,
 * TIMEOUT.
 */
kvq_status kvq_decode_attn(const kvq_cache *global, const kvq_cache *swa, int32_t batch,
                           int32_t num_q_heads, const int32_t *d_seq_lens, const void *q,
                           float softmax_scale, float *out, void *workspace,
                           size_t workspace_bytes, int32_t *d_err_flag, kvq_stream stream);

/*
 * kvq_decode_attn_noalloc -- kvq_decode_attn for callers that cannot allocate
 * device memory on their call path: a plug-in running inside a host framework
 * that owns every device allocation through its own pool, or code under a hard
 * memory budget where an extra cudaMalloc (which may also synchronise the
 * device) is not allowed.  The pages describe no such entry point; it exists
 * only for these callers.  Same arguments and results as kvq_decode_attn,
 * without `workspace`: the scratch is a fixed 8 MiB device array inside the
 * library, which every GPU that loads the library keeps until the process
 * exits.  Sizes whose kvq_decode_workspace_bytes exceed 8 MiB are refused with
 * KVQ_ERR_WORKSPACE (nothing is enqueued).  The first call on each device looks
 * up the array's device address (cudaGetSymbolAddress), so make that first call
 * before any stream capture.  With CUDA's lazy module loading (the default),
 * the first libkvq call on a device -- or that address lookup -- is also what
 * loads the library's device module and reserves its memory, the 8 MiB array
 * included; a caller that must not allocate on its call path makes one call
 * (of this entry point, or any libkvq call on that device) during its setup.
 * The array needs no clearing (each call writes the scratch it reads), but
 * all calls share it: calls whose kernels can overlap on
 * the GPU (different streams, or a second call before the first finished on
 * another stream) race and give wrong results; serialise them on one stream.
 * Allocates nothing and calls no allocating routine.
 */
kvq_status kvq_decode_attn_noalloc(const kvq_cache *global, const kvq_cache *swa, int32_t batch,
                                   int32_t num_q_heads, const int32_t *d_seq_lens, const void *q,
                                   float softmax_scale, float *out, int32_t *d_err_flag,
                                   kvq_stream stream);

/*
 * kvq_append_decode_attn -- one decode step with its append fused in:
 * kvq_append of one new token per sequence at position T_b - 1 followed by
 * kvq_decode_attn over positions 0..T_b-1, in one decode launch (plus the
 * merge).  ("Quantising the KV cache", section "Code": each new K/V row is
 * quantised as it enters the cache, and attention reads it back.)  The codes
 * and scale bytes written equal those of kvq_append (same quantiser, same
 * placement).  The output is that of kvq_append followed by kvq_decode_attn
 * with the same products summed in another order: the fused kernel adds each
 * stage's PV products straight into its fp32 accumulator, so the two differ
 * by fp32 reassociation only (at most about 3 n 2^-24 max|V^| after n
 * 128-token stages of one CTA range).  The producer warp of the CTA that
 * reads a sequence's last chunk stores that sequence's new token a few
 * chunks before copying it, so no separate append launch is needed.  When
 * the cache's capacity (max_pages_per_seq * page_size) gives the CTA ranges
 * fewer than 16 chunks each, the append runs as its own launch before the
 * decode instead, and the output then equals the two calls' bit for bit.
 *   global       FP4 or NVFP4 cache (head_dim 64 or 128), as kvq_decode_attn.
 *   d_seq_lens   device int32 [batch]: T_b including the new token; T_b == 0
 *                appends nothing and gives a zero output row.
 *   k_new, v_new device bf16 [batch][num_kv_heads][head_dim], 16-byte aligned:
 *                the new token of every sequence (row b is ignored when
 *                T_b == 0).
 *   other arguments, workspace and device flags as kvq_decode_attn, plus the
 *   append's NONFINITE flag.  There is no FP8 window form: with a sliding
 *   window, call kvq_append on both caches and then kvq_decode_attn.
 */
kvq_status kvq_append_decode_attn(const kvq_cache *global, int32_t batch, int32_t num_q_heads,
                                  const int32_t *d_seq_lens, const void *k_new, const void *v_new,
                                  const void *q, float softmax_scale, float *out, void *workspace,
                                  size_t workspace_bytes, int32_t *d_err_flag, kvq_stream stream);

/*
 * kvq_decode_attn_tc -- kvq_decode_attn for head_dim 128 with both products
 * on the 5th-generation tensor cores: per 128-token stage the E2M1 x E4M3
 * expansion of K^ (tokens on TMEM lanes) and of V^T (channels on TMEM lanes)
 * goes to tensor memory, S = K^ Q^T and O^T += V^T P^T run as tcgen05.mma
 * M=128 N=16 (8 query rows padded), O stays in tensor memory, and three
 * independent pipelines share an SM.  ("Quantising the KV cache", section
 * "Code"; "KV Cache Quantisation", section "Common questions".)  Same
 * arguments, workspace, results (within the decode tolerance) and device flags
 * as kvq_decode_attn; head_dim 64 returns KVQ_ERR_UNSUPPORTED.  It is a
 * measured alternative, not the default: on GB300 at 32k context it runs
 * about 1.6x slower than kvq_decode_attn (the channel split of V^T that
 * tensor-memory lanes impose costs more instructions than the tensor-core
 * products save, and the per-stage warpgroup barriers stall).
 */
kvq_status kvq_decode_attn_tc(const kvq_cache *global, const kvq_cache *swa, int32_t batch,
                              int32_t num_q_heads, const int32_t *d_seq_lens, const void *q,
                              float softmax_scale, float *out, void *workspace,
                              size_t workspace_bytes, int32_t *d_err_flag, kvq_stream stream);

/*
 * kvq_test_set_wait_limit_ns -- for tests of the timeout path only: every
 * bounded wait of the mma.sync decode kernel on its own pipeline (a consumer
 * waiting for a stage to land, the producer waiting for a free stage) gives
 * up after `ns` nanoseconds instead of about 2 s, for kvq_decode_attn,
 * kvq_decode_attn_noalloc and kvq_append_decode_attn calls enqueued after
 * this one; 0 restores the default.  A wait that gives up sets
 * KVQ_FLAG_TIMEOUT, the CTA stops consuming, its producer waits (always up to
 * about 2 s) for the copies it already issued, and the call's output is
 * undefined.  A non-zero limit selects a separate instantiation of the
 * kernel that reads the limit at run time; 0 selects the production one,
 * whose limit is a compile-time constant.  Process-wide; not for production
 * use.
 */
void kvq_test_set_wait_limit_ns(uint64_t ns);

/*
 * kvq_prefill_attn -- attention of a chunk of new query tokens over the FP4 or
 * NVFP4 cache that already holds their keys and values (chunked prefill):
 * query token i of sequence b (0 <= i < chunk) sits at position
 * T_b - chunk + i and attends positions 0..T_b - chunk + i (causal), every
 * one dequantised from the cache.  ("Quantising the KV cache", section
 * "Code": the quantised K and V feed an unchanged attention.)  Runs on the
 * tensor cores: one CTA per 256 query rows (G query heads x 256/G tokens, as
 * two 128-row tiles), cache tiles of 128 positions dequantised once into
 * shared memory and shared by both.  Query values are used at f16 precision
 * after an exact power-of-two rescale of each row; dequantised K and V are
 * exact in f16; P is rounded to f16; accumulation is fp32.
 *   cache        FP4 or NVFP4 cache, head_dim 64 or 128.
 *   num_q_heads  Hq, a multiple of num_kv_heads with G = Hq/Hkv in {1,2,4,8}.
 *   d_seq_lens   device int32 [batch]: T_b >= chunk, the positions in the
 *                cache including the chunk's.
 *   q            device bf16 [batch][chunk][num_q_heads][head_dim].
 *   out          device float [batch][chunk][num_q_heads][head_dim].
 * Host errors: INVALID_ARGUMENT; UNSUPPORTED (head_dim, G).  Device flags:
 * BAD_LENGTH (T_b < chunk: the sequence's rows are written as 0), PAGE_OOB,
 * TIMEOUT.
 */
kvq_status kvq_prefill_attn(const kvq_cache *cache, int32_t batch, int32_t num_q_heads, int32_t chunk,
                            const int32_t *d_seq_lens, const void *q, float softmax_scale, float *out,
                            int32_t *d_err_flag, kvq_stream stream);

/*
 * kvq_dequant -- expand a cache to dense values (value = E2M1(code) * E4M3(s)
 * for FP4, exact in fp32 and bf16; fp32(that * S) for NVFP4;
 * fp32(E4M3(code) * s_h) for FP8).
 * ("Quantising the KV cache", section "Code": the dequantised value is the
 * code times its scale.)
 *   FP4, NVFP4: k_out, v_out [batch][max_len][num_kv_heads][head_dim]; positions
 *        >= d_seq_lens[b] are written as 0.
 *   FP8: max_len must equal the window W; the rings are written in slot order
 *        [batch][W][num_kv_heads][head_dim] and d_seq_lens is ignored (NULL ok).
 *   out_dtype 0 = float32, 1 = bfloat16.
 * Device flags: PAGE_OOB, BAD_LENGTH.
 */
kvq_status kvq_dequant(const kvq_cache *cache, int32_t batch, const int32_t *d_seq_lens,
                       int32_t max_len, int32_t out_dtype, void *k_out, void *v_out,
                       int32_t *d_err_flag, kvq_stream stream);

/* ------------------------------------------------------------------ bit-width sweep
 * Layouts of the formats compared in the results table of "Quantising the KV
 * cache" (section "Concept"; storage b + s/g bits per number, section
 * "Maths"), for measuring what each does to attention -- not cache formats.
 * Readings (the pages give the INT formats' storage, not their rounding):
 *   FP8_TENSOR       E4M3, one scale per tensor: s = amax/448 in fp32 over the
 *                    whole tensor (1 if amax == 0), code RNE_e4m3(x/s)
 *                    saturating, x^ = E4M3(code) * s in fp32.
 *   INT_PER_TOKEN    symmetric INT-b, one FP16 scale per (sequence, token,
 *                    head) group of head_dim channels;
 *   INT_PER_CHANNEL  ... one FP16 scale per (sequence, head, channel) group
 *                    over the tokens (section "Per token or per channel?").
 *                    Both: s = FP16_RNE(amax/qmax), qmax = 2^(bits-1)-1, fp32
 *                    division, saturating at 65504, 0 -> 2^-24; code
 *                    clamp(RNE(x/s), -qmax, qmax) (fp32 division, NaN -> 0);
 *                    x^ = code * s.
 *   FP4_G16          the cache's E2M1 + E4M3-per-16 block quantiser. */
enum {
  KVQ_LAYOUT_FP8_TENSOR = 1,
  KVQ_LAYOUT_INT_PER_TOKEN = 2,
  KVQ_LAYOUT_INT_PER_CHANNEL = 3,
  KVQ_LAYOUT_FP4_G16 = 4
};

/*
 * kvq_fake_quant -- quantise x in one sweep layout and write the dequantised
 * values ("Quantising the KV cache", section "Code": the quantised K and V
 * replace the real ones ahead of the attention).
 *   layout, bits  FP8_TENSOR: 8; INT_*: 2..8; FP4_G16: 4.
 *   x       device bf16 [batch][tokens][heads][head_dim], head_dim % 16 == 0,
 *           16-byte aligned.
 *   x_hat   device float, same shape (required).
 *   codes   device int8, same shape, or NULL: INT codes; E4M3 bytes (FP8);
 *           E2M1 nibbles 0..15 (FP4).
 *   scales  FP8_TENSOR: device float[2], required (scales[0] is scratch,
 *           scales[1] receives s); INT_PER_TOKEN: uint16 FP16 bit patterns
 *           [batch][tokens][heads] or NULL; INT_PER_CHANNEL: uint16
 *           [batch][heads][head_dim] or NULL; FP4_G16: uint8 E4M3 bytes, one
 *           per 16 values in order, or NULL.
 * Host errors: INVALID_ARGUMENT (sizes, layout/bits, pointers).  Device flag:
 * NONFINITE.  No counterpart on the pages for the entry point itself.
 */
kvq_status kvq_fake_quant(int32_t layout, int32_t bits, int32_t batch, int32_t tokens, int32_t heads,
                          int32_t head_dim, const void *x, float *x_hat, int8_t *codes, void *scales,
                          int32_t *d_err_flag, kvq_stream stream);

/*
 * kvq_attn_dense -- decode attention over dense float K and V with every
 * product, the softmax and the sums in fp64 (the measuring stick of the
 * sweep: "Quantising the KV cache", section "Code", the attention the
 * quantised K and V feed is unchanged).
 *   out[b][h] = sum_t softmax_t(softmax_scale * q[b][h] . k[b][t][h/G]) v[b][t][h/G]
 *   q    device bf16 [batch][num_q_heads][head_dim].
 *   k, v device float [batch][tokens][num_kv_heads][head_dim].
 *   out  device float [batch][num_q_heads][head_dim].
 *   top  device int32 [batch][num_q_heads] or NULL: the position with the
 *        largest score (the lowest on a tie; -1 when tokens == 0).
 * Host errors: INVALID_ARGUMENT; UNSUPPORTED for tokens > 16384 or head_dim
 * > 512.
 */
kvq_status kvq_attn_dense(int32_t batch, int32_t tokens, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, const void *q, const float *k, const float *v,
                          float softmax_scale, float *out, int32_t *top, kvq_stream stream);

/*
 * kvq_swa_replay_workspace_bytes / kvq_swa_replay -- replay of a toy
 * multilayer sliding-window (SWA) network over a range of positions,
 * rebuilding each layer's window state: the K and V rows of the last n_win
 * positions.  ("Week 6 -- FP4 KV Caches and Bounded Replay", Core Concepts
 * "Bounded replay" and Lab: an exact replay reaches back about L n_win
 * positions -- precisely n_win + (L - 1)(n_win - 1) -- while a bounded replay
 * starts only n_win back.)  The pages give the toy no shapes; it is: L layers
 * of width d, one head each; per position i of the replayed range
 *   u = x_i / sqrt(mean(x_i^2) + 1e-6),  q, k, v = Wq u, Wk u, Wv u
 *   a_i = sum over s = max(0, i - n_win + 1) .. i of
 *         softmax_s(q_i . k_s / sqrt(d)) v_s,   x_i += Wo a_i
 * with every layer's k, v, q taken from that layer's input.
 *   w          device float [layers][4][d][d], row-major Wq, Wk, Wv, Wo
 *              ((W u)[r] = sum_c W[r][c] u[c]).
 *   emb        device float [n][d]: the inputs of the n replayed positions.
 *   states     device float [layers][2][n_win][d]: out, each layer's K rows
 *              then V rows of positions n - n_win .. n - 1.
 *   hidden     device float [n][d] or NULL: out, the last layer's x.
 *   workspace  device, at least kvq_swa_replay_workspace_bytes(layers, n, d)
 *              bytes, 16-byte aligned, owned by the caller.
 * d is 64 or 128; 1 <= n_win <= min(n, 4096); layers >= 1.  fp32 arithmetic.
 * A position's result depends only on the inputs of its window (in a fixed
 * order), so a replay that starts at the exact start reproduces the state of
 * a forward pass over the whole sequence bit for bit.
 * Host errors: INVALID_ARGUMENT (pointers, sizes, alignment), WORKSPACE
 * (too small).  No device flags.
 */
size_t kvq_swa_replay_workspace_bytes(int32_t layers, int64_t n, int32_t d);
kvq_status kvq_swa_replay(const float *w, int32_t layers, int32_t d, const float *emb, int64_t n, int32_t n_win,
                          float *states, float *hidden, void *workspace, size_t workspace_bytes,
                          kvq_stream stream);

/* Bytes of an FP4 page pool: num_pages * num_kv_heads * page_size *
 * 9 * head_dim / 8 (0 for invalid sizes). */
size_t kvq_fp4_pool_bytes(int64_t num_pages, int32_t num_kv_heads, int32_t page_size, int32_t head_dim);

/* A static, human-readable name for a status code. */
const char *kvq_status_string(kvq_status status);

/* KVQ_VERSION of the built library. */
int32_t kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
