/*
 * libmlaq -- MLA decode attention over a jointly low-bit, dual-path, paged KV
 * cache (QuantMLA C4R4 / C2R4), plus the fused writer that fills the cache.
 *
 * The method: "QuantMLA: Function-Aligned Dual-Path Quantization for Low-Bit
 * MLA KV Caching" (arXiv 2609.36760), as summarised on
 *   - ai.info "AI summary": "Key Contributions" item 4 (native low-bit MLA
 *     backend: unpack + dequant fused into attention, BF16 buffers for 4 sink
 *     and 128 recent tokens, one global softmax over all valid tokens) and
 *     "Methodology in Plain English" (packed data and metadata buffered apart
 *     from the reconstructed tiles; per-token asymmetric affine quantizer,
 *     group size 64);
 *   - onedev.kr summary, section "어떻게 쓰나" (the fused writer keeps a
 *     packed copy of every token plus the pre-quantization BF16 values of the
 *     4 sink and 128 most recent tokens; each token is read in exactly one
 *     representation; a token leaving the recent window switches to its
 *     existing packed copy with no re-quantization).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers to caller-owned memory. The
 *     library never allocates, frees or retains caller tensors beyond the
 *     cache handle's lifetime (the handle records the pool pointers given to
 *     mlaq_cache_create).
 *   - bf16 tensors are passed as uint16_t bit patterns; row-major, densely
 *     packed, 16-byte aligned.
 *   - Calls that take a stream are asynchronous on that stream (NULL = the
 *     legacy default stream) and do no host<->device synchronisation, so they
 *     may be captured in a CUDA graph. Exceptions are documented per call.
 *   - Return value: MLAQ_OK (0) or a negative mlaq_status for an argument
 *     error detected on the host; nothing is launched in that case.
 *   - Errors found on the device (page index outside the pool, sequence past
 *     its page-table row, non-finite quantization metadata, a bounded wait
 *     that ran out) set bits in a sticky device status word, read with
 *     mlaq_get_device_status. Kernels never trap; offending tokens are skipped
 *     (writer) or masked out (decode).
 *
 * Model shapes: content latent 512 + decoupled RoPE key 64 per token; H query
 * heads absorbed into the latent (H a multiple of 16, 16 <= H <= 128); 64-token
 * pages.
 */
#ifndef MLAQ_H_
#define MLAQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t */
typedef struct mlaq_cache mlaq_cache;

/* Cache formats. C4R4: content INT4 + RoPE INT4. C2R4: content INT2 + RoPE
 * INT4 (ai.info "Key Contributions" item 3). BF16: every token kept as BF16
 * in the pages -- the uncompressed comparison cache, decoded by the same
 * kernel. */
typedef enum mlaq_mode { MLAQ_C4R4 = 0, MLAQ_C2R4 = 1, MLAQ_BF16 = 2 } mlaq_mode;

typedef enum mlaq_status {
  MLAQ_OK = 0,
  MLAQ_ERR_NULL = -1,      /* a required pointer is NULL */
  MLAQ_ERR_MODE = -2,      /* unknown mode */
  MLAQ_ERR_SHAPE = -3,     /* size outside the supported range (B, H, n_new, ...) */
  MLAQ_ERR_ALIGN = -4,     /* a pointer is not 16-byte aligned */
  MLAQ_ERR_CAPACITY = -5,  /* B > max_seqs, H > max_heads, ... */
  MLAQ_ERR_CUDA = -6,      /* a CUDA runtime call failed (launch, event, ...) */
  MLAQ_ERR_WORKSPACE = -7  /* workspace smaller than mlaq_buffer_sizes asked for */
} mlaq_status;

/* Bits of the sticky device status word. */
#define MLAQ_DEV_PAGE_OOB 0x1     /* page_table entry outside [0, num_pages) */
#define MLAQ_DEV_SEQ_OVERFLOW 0x2 /* token position beyond max_pages_per_seq * 64 */
#define MLAQ_DEV_NONFINITE 0x4    /* quantization metadata not finite in fp16 */
#define MLAQ_DEV_TIMEOUT 0x8      /* a bounded wait on a bulk copy ran out */
#define MLAQ_DEV_RANGE 0x10       /* a value outside the decode's fp16 operand range
                                     (see mlaq_append and mlaq_decode) */
#define MLAQ_DEV_BAD_ROWS 0x20    /* mlaq_append: cu_new[B] != total_new, or cu_new is
                                     not a non-decreasing prefix sum from 0 */

#define MLAQ_PAGE_TOKENS 64
#define MLAQ_SINK 4
#define MLAQ_RECENT 128
#define MLAQ_D_LATENT 512
#define MLAQ_D_ROPE 64

/* Byte sizes of the four device buffers a cache needs.
 *   codes:     packed code pool, num_pages pages of 64 tokens
 *              (C4R4 288 B/token, C2R4 160 B/token, BF16 1152 B/token);
 *   meta:      fp16 (scale, min) pool kept apart from the codes, 36 B/token
 *              (0 for BF16);
 *   ring:      BF16 sink + recent buffer, 132 tokens x 1152 B per sequence
 *              slot (0 for BF16);
 * BF16 rows (ring slots, and tokens of BF16-mode pages) keep their 72
 * 16-byte chunks XOR-permuted by the row index: channel e of row r (r = ring
 * slot, or token index within its page) is element
 * ((e / 8) ^ (r % 8)) * 8 + e % 8 of the row, so that eight consecutive rows
 * read at one channel fall in eight different shared-memory bank groups.
 *   workspace: split-KV plan, partial outputs and the device status word,
 *              for batches up to max_seqs sequences and max_heads heads.
 * Limits: 1 <= max_seqs <= 16384; max_heads a multiple of 16 in [16, 128].
 * Returns MLAQ_ERR_SHAPE / MLAQ_ERR_MODE for bad sizes. Host only. */
int mlaq_buffer_sizes(int mode, int32_t num_pages, int32_t max_seqs, int32_t max_heads,
                      size_t* codes_bytes, size_t* meta_bytes, size_t* ring_bytes,
                      size_t* workspace_bytes);

/* Create a cache handle over caller-allocated device buffers (sizes from
 * mlaq_buffer_sizes; all 256-byte aligned; workspace zero-filled by the
 * caller before first use). Pages are addressed only through the page tables
 * passed to each call; row b of a page table (and seq_lens[b]) is sequence
 * slot b, which also selects ring slot b. The handle is host memory; destroy
 * it with mlaq_cache_destroy. Queries the current device's SM count.
 * MLAQ_ERR_SHAPE also when max_seqs * (32 * max_pages_per_seq + 224) reaches
 * 2^31 (the device planner's 32-bit cost sums). */
int mlaq_cache_create(mlaq_cache** out, int mode, int32_t num_pages, int32_t max_seqs,
                      int32_t max_pages_per_seq, int32_t max_heads, void* codes, void* meta,
                      void* ring, void* workspace, size_t workspace_bytes);
int mlaq_cache_destroy(mlaq_cache* cache);

/* Fused writer (onedev.kr "어떻게 쓰나"): append new tokens to B sequences.
 *   page_table [B, max_pages_per_seq] int32: physical page of each 64-token
 *       block; every page the new tokens land in must be mapped.
 *   seq_lens [B] int32, IN-OUT: length before the append; the call adds each
 *       sequence's new-token count on the device when it finishes.
 *   c_latent [N, 512] bf16, k_rope [N, 64] bf16: the new tokens.
 *   cu_new: NULL -> every sequence gets n_new tokens, rows laid out
 *       [B, n_new]; else a device int32 [B+1] prefix sum: sequence b gets rows
 *       cu_new[b] .. cu_new[b+1]-1, and total_new must equal cu_new[B]
 *       (the host value sizes the launch). A mismatch, or counts that are not
 *       a non-decreasing prefix sum from 0, sets MLAQ_DEV_BAD_ROWS; rows that
 *       cu_new does not place are skipped, and the lengths of such a call are
 *       undefined (reset them before the next append).
 * Each token t is quantized per group (8 content groups + 1 RoPE group of 64
 * channels: mn = min, s = fp16((max - mn) / (2^b - 1)), q = clamp(rint((x -
 * fp16(mn)) / s), 0, 2^b - 1), s == 0 -> q = 0, IEEE fp32), packed into page
 * page_table[b][t/64] slot t%64, and its fp16 (s, mn) written to the meta
 * pool. If t < 4 its BF16 values go to ring slot t; if t is among the last
 * 128 tokens after the append they go to ring slot 4 + t%128, overwriting the
 * token 128 positions earlier, which from then on is read from its packed
 * copy (no re-quantization). In BF16 mode the BF16 token is stored in the
 * page instead. Invalid page entries set MLAQ_DEV_PAGE_OOB and skip the token.
 * The decode computes on fp16 operands (bf16 for an all-BF16 cache, under the
 * same bound, which also keeps every score finite in fp32), so the writer
 * checks their range: a
 * BF16 copy (ring slot or BF16-mode page) holding a value beyond +-65504 or a
 * NaN, or a packed group whose largest reconstructed value mn + (2^b - 1) * s
 * reaches 65520, sets MLAQ_DEV_RANGE (non-finite metadata sets
 * MLAQ_DEV_NONFINITE instead); the token is still stored, and decodes of its
 * sequence are undefined while it is attended.
 */
int mlaq_append(mlaq_cache* cache, const int32_t* page_table, int32_t* seq_lens, int32_t B,
                const uint16_t* c_latent, const uint16_t* k_rope, int32_t n_new,
                const int32_t* cu_new, int32_t total_new, struct CUstream_st* stream);

/* Decode attention for one query token per sequence (ai.info "Key
 * Contributions" item 4; onedev.kr "어떻게 쓰나").
 *   q_latent [B, H, 512] bf16 (absorbed queries), q_rope [B, H, 64] bf16;
 *   page_table [B, max_pages_per_seq], seq_lens [B] (current lengths L);
 *   softmax_scale: multiplies q_latent.c + q_rope.k_rope;
 *   out_latent [B, H, 512] bf16: sum_t softmax_t * c_t over the 512-d latent;
 *   lse [B, H] fp32: natural log of sum_t exp(scale * score_t).
 * Token t < L is read from its BF16 ring copy iff t < 4 or t >= L - 128,
 * otherwise from its packed copy (unpacked and dequantized inside the
 * kernel); all tokens share one softmax. L == 0 gives out = 0, lse = -inf.
 * Work is split over the GPU (split-KV) by a device-side planner from
 * seq_lens, and merged by a log-sum-exp combine kernel: three launches, no
 * host sync. The kernel computes on fp16 operands (bf16 for an all-BF16
 * cache) with fp32 accumulation, and inputs must lie in fp16 range in every
 * mode; this is checked: a query element beyond
 * +-65504 or a NaN, or a per-group (64-channel) sum of one head's query
 * beyond the fp16 range, sets MLAQ_DEV_RANGE (cached tokens are checked by
 * the writer); that sequence's output is then undefined and the other
 * sequences are unaffected. The first decode call on a device
 * (any mode, any head count) opts every attention kernel variant into large
 * shared memory (a host-side attribute), so make that first call outside any
 * CUDA-graph capture; later calls capture.
 */
int mlaq_decode(mlaq_cache* cache, const uint16_t* q_latent, const uint16_t* q_rope,
                const int32_t* page_table, const int32_t* seq_lens, int32_t B, int32_t H,
                float softmax_scale, uint16_t* out_latent, float* lse,
                struct CUstream_st* stream);

/* Decode attention for Q query tokens per sequence (multi-token prediction
 * or speculative verification; the pages describe Q = 1, this is its causal
 * extension). The Q new tokens must already be appended: seq_lens[b] = L
 * counts them, and query j = 0..Q-1 (position L - Q + j) attends to tokens
 * t < L - (Q - 1 - j), each in the representation (BF16 or packed) that the
 * length-L cache gives it, under one softmax per query.
 *   q_latent [B, Q, H, 512] bf16, q_rope [B, Q, H, 64] bf16;
 *   out_latent [B, Q, H, 512] bf16, lse [B, Q, H] fp32.
 * Q >= 1, H a multiple of 16, Q * H <= 128 and <= the cache's max_heads (the
 * Q * H query rows share every unpacked page, as heads do). A query that sees
 * no token gets out = 0, lse = -inf. Same launches, status and capture rules
 * as mlaq_decode; Q = 1 is mlaq_decode. Returns MLAQ_ERR_SHAPE or
 * MLAQ_ERR_CAPACITY for sizes outside those bounds. */
int mlaq_decode_mtp(mlaq_cache* cache, const uint16_t* q_latent, const uint16_t* q_rope,
                    const int32_t* page_table, const int32_t* seq_lens, int32_t B, int32_t Q, int32_t H,
                    float softmax_scale, uint16_t* out_latent, float* lse, struct CUstream_st* stream);

/* Allocation-free variant of mlaq_decode. The pages describe no such call;
 * it exists for callers that cannot allocate device memory: code running
 * inside another runtime's allocator, plugins that may not call cudaMalloc
 * while a stream is being captured, or hosts that reserve all of HBM up
 * front. Such a caller still owns and passes the cache pools (codes, meta,
 * ring, filled by mlaq_append or an equivalent writer of the same layout),
 * the inputs and the outputs; only the split-KV scratch (plan, partial
 * outputs, status word) moves into a fixed 64 MiB array inside this library,
 * which every GPU that loads the library holds until the process exits.
 *   mode, num_pages, max_pages_per_seq: describe the pools as for
 *       mlaq_cache_create (ring holds at least B sequence slots);
 *   remaining arguments as for mlaq_decode;
 *   dev_status: optional device int32 that receives this call's device
 *       status bits (MLAQ_DEV_*), or NULL.
 * Calls nothing that allocates (no cudaMalloc / cudaFree, no allocating
 * library routine). The scratch needed for (B, H) is what mlaq_buffer_sizes
 * reports as workspace_bytes for max_seqs = B, max_heads = H: about
 * (B * H + 32768 + H) * 1028 bytes of split partials plus 36 * B + 38 KB of
 * plan; when it exceeds 64 MiB the call returns MLAQ_ERR_CAPACITY and
 * launches nothing. That admits B * H up to about 32,300: B <= 2022 at H = 16,
 * 1011 at H = 32, 505 at H = 64, 252 at H = 128. The first call on each
 * device looks up the array's device address and sets the shared-memory
 * attribute of every decode kernel variant (all modes and head counts);
 * make that first call before any stream capture. Every call uses the same
 * array and the next call
 * overwrites it (the status word is cleared at the start of each call), so
 * calls that can overlap on the GPU -- on different streams, or on two
 * threads -- race and give wrong results; serialise them on one stream. */
int mlaq_decode_noalloc(int mode, const void* codes, const void* meta, const void* ring,
                        int32_t num_pages, int32_t max_pages_per_seq, const uint16_t* q_latent,
                        const uint16_t* q_rope, const int32_t* page_table, const int32_t* seq_lens,
                        int32_t B, int32_t H, float softmax_scale, uint16_t* out_latent, float* lse,
                        int32_t* dev_status, struct CUstream_st* stream);

/* Debug / test read-back of n stored tokens in a canonical form independent
 * of the physical packing: for k < n, token token_t[k] of sequence
 * token_b[k] ->
 *   codes_out [n, 576] uint8, one code per byte (content 0..511, RoPE
 *   512..575), meta_out [n, 9, 2] uint16 fp16 bits (scale, min) per group.
 * Packed modes only. Device pointers; asynchronous. */
int mlaq_export_tokens(mlaq_cache* cache, const int32_t* page_table, int32_t B,
                       const int32_t* token_b, const int32_t* token_t, int32_t n,
                       uint8_t* codes_out, uint16_t* meta_out, struct CUstream_st* stream);

/* Persistent-cache accounting (onedev.kr system-efficiency paragraph: BF16
 * buffers + redundant packed copies + page mapping), for host seq_lens.
 * *policy_bytes: this cache's format; *bf16_bytes: the same sequences in a
 * paged all-BF16 cache. Host only. */
int mlaq_cache_bytes(const mlaq_cache* cache, const int32_t* seq_lens_host, int32_t B,
                     size_t* policy_bytes, size_t* bf16_bytes);

/* Synchronises `stream`, then returns the sticky device status word
 * (MLAQ_DEV_* bits) in *status. Blocks the host. */
int mlaq_get_device_status(mlaq_cache* cache, struct CUstream_st* stream, int32_t* status);
/* Clears the device status word (asynchronous on `stream`). */
int mlaq_clear_device_status(mlaq_cache* cache, struct CUstream_st* stream);

/* Kernel timing for measurement: when enabled, mlaq_decode records a CUDA
 * event pair around the whole call (planner, attention and combine kernels) on
 * the call's stream, up to max_calls calls. mlaq_timing_read synchronises and
 * returns the per-call durations in milliseconds (*n = number recorded) and
 * resets the counter. Host calls; events are created at enable;
 * max_calls = 0 turns timing off (an event recorded between launches keeps
 * the next kernel from starting before the previous one ends). */
int mlaq_timing_enable(mlaq_cache* cache, int32_t max_calls);
int mlaq_timing_read(mlaq_cache* cache, float* ms_out, int32_t* n);

/* Number of CTAs the decode planner aims to fill (default: one wave of the
 * attention kernel's resident CTAs: for the register-score kernel 3 per SM
 * with 16 heads per CTA, 2 per SM with 32; 1 per SM for the tcgen05-score
 * kernel). 1 <= ctas <= 1024. */
int mlaq_set_decode_ctas(mlaq_cache* cache, int32_t ctas);

/* Which attention kernel mlaq_decode / mlaq_decode_mtp use (a tuning and
 * test knob; results agree within the stated tolerances):
 *   0 (default) automatic: currently the register-score kernel for every
 *     head count (the faster one on GB300 for the tuned shapes);
 *   1 register scores (legacy m16n8k16 MMAs on exact codes, tcgen05
 *     aggregation);
 *   2 tcgen05 scores and aggregation (64, 32 or 16 heads per CTA; exact
 *     scores through split fp16 scales).
 * MLAQ_ERR_SHAPE for other values. Host call; takes effect at the next
 * decode. */
int mlaq_set_decode_variant(mlaq_cache* cache, int32_t variant);

/* Costs the decode planner balances across CTAs (a tuning knob; the results
 * do not depend on it): `step` per 16-token step of a packed page or BF16
 * page, `ring` per 16-slot chunk of the BF16 sink/recent ring, `item` once per
 * sequence for the CTA that starts it. Defaults 8, 19, 40 (measured on
 * GB300). Requires 1 <= step <= 8, ring >= 1, item >= 0 and
 * item + 9 * ring <= 512, else MLAQ_ERR_SHAPE and the costs are unchanged.
 * Host call; takes effect at the next decode. */
int mlaq_set_plan_costs(mlaq_cache* cache, int32_t step, int32_t ring, int32_t item);

/* Test hook for the bounded waits behind MLAQ_DEV_TIMEOUT (the decode kernel
 * waits on mbarriers for its bulk copies and its tensor-core MMAs, each wait
 * limited in wall time, never a trap). Launches one CTA of 32 threads that
 * waits on a shared-memory mbarrier through that same bounded wait with a
 * limit of wait_us microseconds. arrive = 0: nothing completes the barrier,
 * the wait runs out and the kernel stores MLAQ_DEV_TIMEOUT in *status;
 * arrive = 1: the CTA completes the barrier first and stores 0. status is a
 * device pointer to one int32 owned by the caller. Asynchronous on `stream`.
 * Returns MLAQ_ERR_NULL for a NULL status, MLAQ_ERR_SHAPE for wait_us outside
 * [1, 100000] or arrive outside {0, 1}, MLAQ_ERR_CUDA if the launch fails. */
int mlaq_debug_wait_probe(int32_t* status, int32_t wait_us, int32_t arrive, struct CUstream_st* stream);

const char* mlaq_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLAQ_H_ */
