/*
 * kvq.h -- C ABI of the INT4 group-quantized paged KV cache for NVIDIA GB300 (sm_103a).
 *
 * The library implements two operations and an inverse:
 *   quantize-on-append  symmetric per-group INT4 quantization of new K/V rows into
 *                       fixed-size pages ("4-bit KV cache compression",
 *                       lpnh.cn/news/2042373, section 2.1; pages as in "AI inference
 *                       tuning: KV Cache optimisation and memory management",
 *                       bxzpzcl.cn/news/2871434, section 3.1);
 *   decode attention    one query token per sequence attends to every cached token,
 *                       reading the packed cache and dequantizing inside the kernel
 *                       (scaled dot-product attention as in section 3.2 of the same
 *                       KV-cache optimisation page; "dequantize inside the operator" as
 *                       in "LLM long-context inference: managing the KV cache with an
 *                       INT4 state machine", pwwt.cn/news/4219524, section 5 step 5);
 *   dequantize          the inverse map code * scale (section 2.1 of the 4-bit page).
 *
 * Conventions
 *   - Every pointer argument except `cfg` and host outputs is a DEVICE pointer on the
 *     current CUDA device.  The caller owns and allocates all memory; the library
 *     allocates nothing and keeps no state except a per-thread error string (and the
 *     built-in scratch array of kvq_decode_attention_noalloc, described there).
 *   - Every call is asynchronous on `stream` (NULL = the legacy default stream).
 *     Buffers must stay valid until the stream reaches the call.
 *   - Return value: KVQ_OK or an error code; kvq_last_error() describes the last
 *     failure on the calling thread.  Argument errors are detected on the host before
 *     anything is launched.  Bad device-side data (a page id outside [0, num_pages),
 *     a position beyond the block table) is never dereferenced: the offending row is
 *     skipped (quantize) or read from page 0 instead (decode, dequantize) and a flag
 *     bit is OR-ed into a device status word; see kvq_read_status().
 *
 * Storage format (the "pool")
 *   The pool is num_pages * num_kv_heads blocks of kvq_block_bytes(cfg) bytes; block
 *   (page, h) starts at byte (page * num_kv_heads + h) * kvq_block_bytes(cfg).  A block
 *   holds, in order, for its P = page_size token slots:
 *     K codes   P rows of head_dim/2 bytes
 *     V codes   P rows of head_dim/2 bytes
 *     K scales  P rows of head_dim/group_k fp16 (little-endian)
 *     V scales  P rows of head_dim/group_v fp16
 *     zero padding to a multiple of 16 bytes.
 *   A code c in [-7, 7] is stored as the nibble c + 8; byte j of a row holds element
 *   2j in its low nibble and element 2j+1 in its high nibble.  Token position t of
 *   sequence b lives in page block_table[b * max_blocks + t / P], slot t % P.
 *   Storage is 4 + 16/G bits per element (4.5 / 4.25 / 4.125 for G = 32 / 64 / 128),
 *   the figure of section 2.2 of the 4-bit page.
 *
 * Quantization (section 2.1 of the 4-bit page, with the rounding made exact):
 *   scale = fp16_rne(fp32(amax) / 7.0f) over each group of G consecutive elements
 *   along head_dim; a scale that is zero after rounding becomes 1.0;
 *   code  = clamp(round_half_even(fp32(x) / fp32(scale)), -7, 7), an IEEE division.
 *   Codes and scales are bit-exact functions of the fp16 input.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t and a cudaEvent_t, declared without the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *kvq_stream_t;
struct CUevent_st;
typedef struct CUevent_st *kvq_event_t;

/* Cache geometry, shared by all calls on one pool. */
typedef struct {
    int32_t num_kv_heads; /* KV heads per layer (Hkv), >= 1                          */
    int32_t head_dim;     /* d: 64, 128 or 256 (decode over the INT4 cache: all three,
                             d = 256 with up to 4 query heads per KV head and group_k
                             >= 64; over the other caches: 128)                      */
    int32_t page_size;    /* tokens per page: 16, 32 or 64                            */
    int32_t group_k;      /* K quantization group along head_dim: 32, 64 or 128 (<= d) */
    int32_t group_v;      /* V quantization group: 32, 64 or 128 (<= d)               */
    int32_t num_pages;    /* pages in the pool, >= 1                                  */
} kvq_cache_config;

enum {
    KVQ_OK = 0,
    KVQ_EINVAL = 1,       /* null or misaligned pointer, negative size, Hq % Hkv != 0  */
    KVQ_EUNSUPPORTED = 2, /* a geometry outside the supported set above                */
    KVQ_EWORKSPACE = 3,   /* workspace smaller than kvq_decode_workspace_bytes()       */
    KVQ_ECUDA = 4         /* a CUDA runtime error (launch failure, bad device, ...)    */
};

/* Bits OR-ed into a device status word (they stay set until the caller clears them). */
#define KVQ_FLAG_BAD_PAGE 0x1u     /* a block-table entry outside [0, num_pages)          */
#define KVQ_FLAG_BAD_POSITION 0x2u /* a position or length beyond max_blocks * page_size  */
#define KVQ_FLAG_WAIT_TIMEOUT 0x4u /* an asynchronous copy did not complete in time       */
#define KVQ_FLAG_STALE_WORKSPACE 0x8u /* reserved: no longer raised (the decode workspace
                                         carries no state from one call to the next) */

/* Bytes of one (page, kv-head) block; 0 if cfg is invalid.  Pure host computation. */
size_t kvq_block_bytes(const kvq_cache_config *cfg);

/* Bytes of the whole pool: num_pages * num_kv_heads * kvq_block_bytes(cfg). */
size_t kvq_pool_bytes(const kvq_cache_config *cfg);

/*
 * Quantize-on-append (section 2.1 of the 4-bit page; pages as in section 3.1 of the
 * KV-cache optimisation page).
 *   pool         device, kvq_pool_bytes(cfg) bytes, 16-byte aligned; written in place.
 *   k, v         device fp16 [batch, n_new, num_kv_heads, head_dim], contiguous,
 *                16-byte aligned: the new K and V rows.
 *   block_table  device int32 [batch, max_blocks] page ids.
 *   start_pos    device int32 [batch]: token t of sequence b goes to position
 *                start_pos[b] + t.
 *   status       device uint32 status word or NULL; flag bits are OR-ed into it.
 * A row whose position or page is out of range is skipped and flagged.
 * Returns KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED or KVQ_ECUDA.
 */
int kvq_quantize_append(const kvq_cache_config *cfg, void *pool, const void *k, const void *v,
                        const int32_t *block_table, int32_t max_blocks, const int32_t *start_pos,
                        int32_t batch, int32_t n_new, uint32_t *status, kvq_stream_t stream);

/*
 * Quantize-on-append of a ragged batch in one launch: the same quantization and storage
 * as kvq_quantize_append (section 2.1 of the 4-bit page), with a different number of
 * new tokens per sequence (the prefill of a continuous batch, section 3.1 of the
 * KV-cache optimisation page).
 *   k_rows, v_rows  device fp16 [total_rows, num_kv_heads, head_dim], contiguous,
 *                   16-byte aligned: the new tokens of all sequences back to back.
 *   cu_rows         device int32 [batch + 1]: sequence b owns rows cu_rows[b] ..
 *                   cu_rows[b + 1] - 1 (cu_rows[0] = 0, non-decreasing,
 *                   cu_rows[batch] = total_rows); its row cu_rows[b] + t goes to
 *                   position start_pos[b] + t.
 *   other arguments as in kvq_quantize_append.
 * Each row goes to a sequence b in [0, batch) found by a binary search of
 * cu_rows[0 .. batch - 1] (cu_rows[batch] is not read).  Offsets that break the rules
 * above send rows to other sequences or positions but never make the kernel read or
 * write outside its arguments: a position outside the block table is skipped and
 * flagged as there.
 * Returns KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED or KVQ_ECUDA.
 */
int kvq_quantize_append_varlen(const kvq_cache_config *cfg, void *pool, const void *k_rows,
                               const void *v_rows, const int32_t *block_table, int32_t max_blocks,
                               const int32_t *start_pos, const int32_t *cu_rows, int32_t batch,
                               int32_t total_rows, uint32_t *status, kvq_stream_t stream);

/*
 * Workspace bytes kvq_decode_attention needs for this shape on the current device
 * (it depends on the device's SM count).  0 if the arguments are invalid.
 */
size_t kvq_decode_workspace_bytes(const kvq_cache_config *cfg, int32_t batch, int32_t num_q_heads,
                                  int32_t max_len);

/*
 * Decode attention over the packed cache (section 3.2 of the KV-cache optimisation
 * page: scores = q . k * softmax_scale, softmax over all cached positions, weights
 * applied to V; query head hq reads KV head hq / (num_q_heads / num_kv_heads)).
 * K and V are dequantized inside the kernel (section 5 step 5 of the state-machine
 * page); q . k, the softmax and P . V accumulate in fp32.
 *   pool          device, as written by kvq_quantize_append.
 *   q             device fp16 [batch, num_q_heads, head_dim], 16-byte aligned.
 *   block_table   device int32 [batch, max_blocks].
 *   seq_lens      device int32 [batch]: positions 0 .. seq_lens[b]-1 are attended to
 *                 (the newly appended token included).  A length of 0 gives zeros.
 *   max_len       host bound on every seq_lens[b] (sizes the workspace).
 *   out           device fp32 [batch, num_q_heads, head_dim], 16-byte aligned.
 *   workspace     device, >= kvq_decode_workspace_bytes(...) bytes, 256-byte aligned.
 *                 Its first 4 bytes are the status word (zero it before the first call
 *                 to read flags); the rest holds the split-KV partial results of the
 *                 call, written before they are read, so it needs no initialisation and
 *                 can serve any call whose shape needs no more bytes.
 * num_q_heads must be a multiple of num_kv_heads with a ratio of at most 8 (at most 4 at
 * head_dim 256, where group_k must be 64 or 128; KVQ_EUNSUPPORTED otherwise).
 * Two kernels run: the decode grid, which leaves one partial result per warp and
 * segment in the workspace, and a combine grid that merges them into out.
 * Launch overlap: both are launched with programmatic dependent launch.  While the
 * kernel ahead of the decode grid on the stream is still running (only possible when
 * that kernel has signalled its dependents early, which this library's kernels do),
 * the decode grid may already read q, block_table and seq_lens; it reads the pool and
 * touches the workspace only after that kernel has finished, and out is written by
 * the combine grid after the decode grid has finished.  This library's kernels never
 * write q, block_table or seq_lens.
 * Returns KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_EWORKSPACE or KVQ_ECUDA.
 */
int kvq_decode_attention(const kvq_cache_config *cfg, const void *pool, const void *q,
                         const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                         int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                         float *out, void *workspace, size_t workspace_bytes, kvq_stream_t stream);

/*
 * One decode step in one call: quantize-on-append of one new token per sequence
 * (exactly as kvq_quantize_append with n_new = 1), then decode attention (exactly as
 * kvq_decode_attention) over the updated cache.  The warp that streams the page taking
 * a sequence's new token quantizes the token itself, writes it to the pool and uses
 * it; an append into a page the attention does not reach is written by the grid's
 * other warps.  (The two steps are the pages' decode step, section 1.1 of the 4-bit
 * page: append the token, then attend.)
 *   pool          device, kvq_pool_bytes(cfg) bytes, 16-byte aligned; written in place.
 *   k_new, v_new  device fp16 [batch, num_kv_heads, head_dim], contiguous, 16-byte
 *                 aligned: the new token's K and V rows.
 *   append_pos    device int32 [batch]: the new token of sequence b goes to position
 *                 append_pos[b]; a negative position appends nothing for b.
 *   other arguments as in kvq_decode_attention.  seq_lens[b] normally is
 *                 append_pos[b] + 1, so the new token is attended to.
 * A position outside the block table or a bad page id skips that append and sets a
 * flag in the workspace status word.  Two sequences appending into the same slot
 * leave either one.
 * Launch overlap as in kvq_decode_attention, except that q, k_new and v_new are read
 * only after the kernel ahead on the stream has finished (append_pos, like seq_lens
 * and block_table, may be read before).
 * Returns KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_EWORKSPACE or KVQ_ECUDA.
 */
int kvq_decode_step(const kvq_cache_config *cfg, void *pool, const void *k_new, const void *v_new,
                    const int32_t *append_pos, const void *q, const int32_t *block_table, int32_t max_blocks,
                    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_len,
                    float softmax_scale, float *out, void *workspace, size_t workspace_bytes,
                    kvq_stream_t stream);

/*
 * kvq_decode_step from host memory, in one call: the step's inputs moved from host_in to
 * dev_in, the step, its output moved from out to host_out, all queued on `stream`
 * (nothing waits; read host_out after the stream has passed the call).  When host_in and
 * host_out are page-locked (cudaHostAlloc, cudaHostRegister) the kernels move the data
 * themselves: a copy kernel reads host_in through its device address, and the kernel
 * that writes out also writes host_out, so the step stays one chain of kernels launched
 * behind each other (programmatic dependent launch).  Pageable memory takes one
 * cudaMemcpyAsync each way instead.
 *   host_in   host memory holding q [batch, num_q_heads, head_dim] fp16, then k_new
 *             [batch, num_kv_heads, head_dim] fp16, then v_new (same shape), back to back.
 *   dev_in    device buffer of the same size, 16-byte aligned: the inputs' device copy,
 *             from which the step reads q, k_new and v_new.
 *   out       device fp32 [batch, num_q_heads, head_dim], as in kvq_decode_step.
 *   host_out  host memory of the same size: receives out.
 *   other arguments as in kvq_decode_step.  host_in may be refilled, and host_out read,
 *   once the stream has passed the call.
 * Returns as kvq_decode_step.
 */
int kvq_decode_step_host(const kvq_cache_config *cfg, void *pool, const void *host_in, void *dev_in,
                         const int32_t *append_pos, const int32_t *block_table, int32_t max_blocks,
                         const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_len,
                         float softmax_scale, float *out, void *host_out, void *workspace, size_t workspace_bytes,
                         kvq_stream_t stream);

/*
 * kvq_decode_step_host with its copies taken off the compute stream, so that from one call
 * to the next the input copy of step i + 1 and the output copy of step i - 1 run while
 * step i computes (the decode step of section 1.1 of the 4-bit page, fed from the host).
 * The caller keeps two (or more) staging slots, each its own host_in, dev_in, out,
 * host_out and three events, and gives consecutive calls alternate slots.  Per call:
 *   copy_in   waits for events[1] (the step that last read this slot's dev_in), copies
 *             host_in to dev_in, records events[0];
 *   stream    waits for events[0] and events[2] (the output copy that last read this
 *             slot's out), runs the step (as kvq_decode_step), records events[1];
 *   copy_out  waits for events[1], copies out to host_out, records events[2].
 *   stream, copy_in, copy_out  three distinct streams of the device.
 *   events    the slot's three cudaEvent_t, created by the caller (an event never recorded
 *             counts as complete, so a fresh slot needs no set-up); host_out holds the
 *             step's output once events[2] completes, and host_in may be refilled once
 *             events[0] completes.
 *   other arguments as in kvq_decode_step_host.  Steps run in call order on `stream` and
 *   share the workspace.
 * Nothing is allocated and nothing waits on the host.
 * Returns as kvq_decode_step.
 */
int kvq_decode_step_host_pipelined(const kvq_cache_config *cfg, void *pool, const void *host_in, void *dev_in,
                                   const int32_t *append_pos, const int32_t *block_table, int32_t max_blocks,
                                   const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_len,
                                   float softmax_scale, float *out, void *host_out, void *workspace,
                                   size_t workspace_bytes, kvq_stream_t stream, kvq_stream_t copy_in,
                                   kvq_stream_t copy_out, kvq_event_t events[3]);

/*
 * Decode attention and the decode step with a sliding window and sink tokens
 * (SlidingWindowAttention, section 3.2 of the KV-cache optimisation page): the query,
 * at the last position L - 1 of its sequence, attends to positions
 * [max(0, L - window), L) and to the first `sinks` positions [0, min(sinks, L)).
 *   window   >= 0; 0 means no window (every position, as in kvq_decode_attention).
 *   sinks    >= 0; positions kept from the start of the sequence besides the window.
 * Pages wholly outside both ranges are not read.  Every other argument is as in
 * kvq_decode_attention / kvq_decode_step; a workspace of kvq_decode_workspace_bytes()
 * for the same (cfg, batch, num_q_heads, max_len) is large enough for any window.
 * The step appends the new token whether or not it falls in the window (it always
 * does when append_pos[b] = seq_lens[b] - 1).
 * Returns KVQ_OK, KVQ_EINVAL (also for a negative window or sinks), KVQ_EUNSUPPORTED,
 * KVQ_EWORKSPACE or KVQ_ECUDA.
 */
int kvq_decode_attention_window(const kvq_cache_config *cfg, const void *pool, const void *q,
                                const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                                int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                                int32_t window, int32_t sinks, float *out, void *workspace,
                                size_t workspace_bytes, kvq_stream_t stream);
int kvq_decode_step_window(const kvq_cache_config *cfg, void *pool, const void *k_new, const void *v_new,
                           const int32_t *append_pos, const void *q, const int32_t *block_table,
                           int32_t max_blocks, const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                           int32_t max_len, float softmax_scale, int32_t window, int32_t sinks, float *out,
                           void *workspace, size_t workspace_bytes, kvq_stream_t stream);

/*
 * The FP16 cache of the latency comparison (section 7.4 of the INT4 state-machine page:
 * FP16 attention; INT4 dequantized first and then attended; INT4 dequantized inside the
 * operator).  Same pages and block table as the INT4 cache, same cfg (the group sizes
 * are not used): block (page, kv head) at (page * Hkv + h) * 4 * P * d bytes holds K
 * rows P x d fp16, then V rows P x d fp16.
 *
 * kvq_fp16_pool_bytes: num_pages * Hkv * 4 * P * d; 0 if cfg is invalid.
 * kvq_fp16_append: as kvq_quantize_append, storing the fp16 rows unchanged.
 * kvq_dequantize_to_fp16_pool: every position 0 .. seq_lens[b]-1 of the INT4 pool,
 *   dequantized ((nibble - 8) * scale, rounded to fp16 nearest-even), into the FP16 pool
 *   at the same page and slot.  max_len >= every seq_lens[b] (sizes the grid); batch at
 *   most 65535.  Pages or positions out of range are skipped and flagged in *status.
 * kvq_fp16_decode_workspace_bytes / kvq_fp16_decode_attention: as the INT4 calls of the
 *   same names, over the FP16 pool (head_dim 128, page sizes 16/32/64, up to 8 query
 *   heads per kv head).  The workspace sizes differ from the INT4 ones.
 * Return codes as for the INT4 calls.
 */
size_t kvq_fp16_pool_bytes(const kvq_cache_config *cfg);
int kvq_fp16_append(const kvq_cache_config *cfg, void *pool16, const void *k, const void *v,
                    const int32_t *block_table, int32_t max_blocks, const int32_t *start_pos, int32_t batch,
                    int32_t n_new, uint32_t *status, kvq_stream_t stream);
int kvq_dequantize_to_fp16_pool(const kvq_cache_config *cfg, const void *pool, void *pool16,
                                const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                                int32_t batch, int32_t max_len, uint32_t *status, kvq_stream_t stream);
size_t kvq_fp16_decode_workspace_bytes(const kvq_cache_config *cfg, int32_t batch, int32_t num_q_heads,
                                       int32_t max_len);
int kvq_fp16_decode_attention(const kvq_cache_config *cfg, const void *pool16, const void *q,
                              const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                              int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                              float *out, void *workspace, size_t workspace_bytes, kvq_stream_t stream);

/*
 * INT8 per-row cache (KVCacheQuantizer.quantize_int8 of the KV-cache optimisation page,
 * section 3.1): one fp32 scale per (token, kv head) row, scale = amax / 127 (IEEE fp32
 * division, at least 1e-8), code = clamp(round-half-even(x / scale), -128, 127) (fp32
 * division), value = fp32(code * scale).  Same pages, block table and cfg as the INT4
 * cache (group sizes unused): block (page, kv head) at (page * Hkv + h) * (2 P d + 8 P)
 * bytes holds K codes P x d int8, V codes P x d int8, K scales P fp32, V scales P fp32.
 * kvq_int8_pool_bytes: num_pages * Hkv * (2 P d + 8 P); 0 if cfg is invalid.
 * kvq_int8_quantize_append: as kvq_quantize_append (head_dim a multiple of 4, <= 256).
 * kvq_int8_decode_workspace_bytes / kvq_int8_decode_attention: as the INT4 calls of the
 *   same names over the INT8 pool (head_dim 128, up to 8 query heads per kv head).
 */
size_t kvq_int8_pool_bytes(const kvq_cache_config *cfg);
int kvq_int8_quantize_append(const kvq_cache_config *cfg, void *pool8, const void *k, const void *v,
                             const int32_t *block_table, int32_t max_blocks, const int32_t *start_pos,
                             int32_t batch, int32_t n_new, uint32_t *status, kvq_stream_t stream);
size_t kvq_int8_decode_workspace_bytes(const kvq_cache_config *cfg, int32_t batch, int32_t num_q_heads,
                                       int32_t max_len);
int kvq_int8_decode_attention(const kvq_cache_config *cfg, const void *pool8, const void *q,
                              const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                              int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                              float *out, void *workspace, size_t workspace_bytes, kvq_stream_t stream);

/*
 * Rotated 4-bit cache ("LARQL KV cache engines", engine three codec/turbo-quant: each K
 * or V row of a head is rotated by a Walsh-Hadamard transform and quantized with a
 * Lloyd-Max codebook; head_dim a power of two; approximate, per-row cosine about 0.9954
 * at 4 bits).  The page names the two steps only; this library reads them as:
 *   y = H x (x the fp16 row as fp32, H the unnormalised Sylvester-order Walsh-Hadamard
 *   matrix, fast transform with stages of span 1, 2, .., 64), sigma = sqrt(sum x_i^2)
 *   (the RMS of y; squares summed as (x0^2+x1^2)+(x2^2+x3^2) over elements 4l..4l+3,
 *   then across l by pairs at xor distances 16, 8, 4, 2, 1), code_i = the number of
 *   thresholds T_j <= y_i / sigma, T the fp32 midpoints of the 16 Lloyd-Max levels of
 *   the standard normal (sigma = 0: codes 0); every fp32 operation rounds once.
 *   A row dequantizes to H (sigma * c_code) / 128, c the fp32 levels.
 * Same pages, block table and cfg as the INT4 cache (group sizes unused; head_dim 128):
 * block (page, kv head) at (page * Hkv + h) * P * (d + 8) bytes holds K codes P x d/2
 * (element 2j in the low nibble of byte j), V codes P x d/2, K sigma P fp32, V sigma P
 * fp32.
 * kvq_wht4_codebook: writes the 16 fp32 levels (ascending) and the 15 fp32 thresholds to
 *   host memory (either pointer may be NULL); host only, computed once.
 * kvq_wht4_pool_bytes: num_pages * Hkv * P * (d + 8); 0 if cfg is invalid.
 * kvq_wht4_quantize_append: as kvq_quantize_append, into this pool.
 * kvq_wht4_dequantize: positions [start, start + n) of sequence b to fp32 out_k and
 *   out_v [n, Hkv, 128] (device, 16-byte aligned); unmapped pages give zero rows and set
 *   KVQ_FLAG_BAD_PAGE in *status (may be NULL).
 * kvq_wht4_decode_workspace_bytes / kvq_wht4_decode_attention: as the INT4 calls of the
 *   same names over this pool (head_dim 128, up to 8 query heads per kv head).  The
 *   scores and the weighted sum are formed in the rotated domain (q is rotated once per
 *   segment); each partial output is rotated back before the combine.
 * Return codes as for the INT4 calls.
 */
void kvq_wht4_codebook(float *levels16, float *thresholds15);
size_t kvq_wht4_pool_bytes(const kvq_cache_config *cfg);
int kvq_wht4_quantize_append(const kvq_cache_config *cfg, void *pool4r, const void *k, const void *v,
                             const int32_t *block_table, int32_t max_blocks, const int32_t *start_pos,
                             int32_t batch, int32_t n_new, uint32_t *status, kvq_stream_t stream);
int kvq_wht4_dequantize(const kvq_cache_config *cfg, const void *pool4r, const int32_t *block_table,
                        int32_t max_blocks, int32_t b, int32_t start, int32_t n, float *out_k, float *out_v,
                        uint32_t *status, kvq_stream_t stream);
size_t kvq_wht4_decode_workspace_bytes(const kvq_cache_config *cfg, int32_t batch, int32_t num_q_heads,
                                       int32_t max_len);
int kvq_wht4_decode_attention(const kvq_cache_config *cfg, const void *pool4r, const void *q,
                              const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                              int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                              float *out, void *workspace, size_t workspace_bytes, kvq_stream_t stream);

/*
 * Mixed-precision decode attention (section 8.3 of the INT4 state-machine page: quantize
 * the KV of old tokens to INT4 first, keep recent tokens in FP16).  For sequence b of
 * L = seq_lens[b] positions, positions [0, L - residual) are read from the INT4 pool
 * (block_table, max_blocks) and [max(0, L - residual), L) from the FP16 pool
 * (block_table16, max_blocks16, num_pages16 pages; the layout of kvq_fp16_append).  Both
 * tables are indexed by the page number t / page_size of position t; block_table16 only
 * needs valid entries for the pages that hold the last residual positions.  The result
 * is plain decode attention over all L positions (kvq_decode_attention's conventions).
 *   residual  >= 0; 0 is kvq_decode_attention over the INT4 pool alone.
 *   workspace >= kvq_mixed_decode_workspace_bytes(cfg, batch, num_q_heads, max_len,
 *             residual) bytes, 256-byte aligned; its first word is the status word.
 * Three kernels run: the INT4 grid, the FP16 grid, and a combine of both grids'
 * partials.
 * Returns KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_EWORKSPACE or KVQ_ECUDA.
 */
size_t kvq_mixed_decode_workspace_bytes(const kvq_cache_config *cfg, int32_t batch, int32_t num_q_heads,
                                        int32_t max_len, int32_t residual);
int kvq_mixed_decode_attention(const kvq_cache_config *cfg, const void *pool, const int32_t *block_table,
                               int32_t max_blocks, const void *pool16, const int32_t *block_table16,
                               int32_t max_blocks16, int32_t num_pages16, const void *q, const int32_t *seq_lens,
                               int32_t batch, int32_t num_q_heads, int32_t max_len, int32_t residual,
                               float softmax_scale, float *out, void *workspace, size_t workspace_bytes,
                               kvq_stream_t stream);

/*
 * Decode attention that allocates nothing, for callers that cannot provide a
 * workspace: a plugin inside a host engine that owns no device allocator, an
 * embedded or real-time runtime with a fixed memory budget that forbids allocation
 * while serving, code on an out-of-memory path.  (No passage of the pages has a
 * counterpart; this is an interface variant of kvq_decode_attention.)
 * Same computation and arguments as kvq_decode_attention, without the workspace:
 * the scratch lives in an 8 MiB array built into the library, which every GPU that
 * loads the library holds until the process exits.  No cudaMalloc, cudaFree or other
 * allocating call is made.
 *   status   device uint32 or NULL: receives this call's status flags, overwriting what
 *            it held (unlike the other calls, which OR flags into their status word).
 * The array used is the current device's: the stream and every buffer must belong to
 * the current device (a q pointer on another device is rejected with KVQ_EINVAL).
 * The first call on a device looks up the array's address on that device; make that
 * first call before any stream capture.  All calls on a device share the array, so
 * calls whose work overlaps on the GPU (other streams or threads) race: serialize them.
 * A shape that needs more scratch than 8 MiB (see kvq_decode_workspace_bytes) is
 * rejected with KVQ_EWORKSPACE before anything is launched.
 * Returns KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_EWORKSPACE or KVQ_ECUDA.
 */
int kvq_decode_attention_noalloc(const kvq_cache_config *cfg, const void *pool, const void *q,
                                 const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                                 int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                                 float *out, uint32_t *status, kvq_stream_t stream);

/*
 * A test of the decode kernel's bounded waits, for the test suite: kvq_decode_attention
 * (same arguments) with every wait on a copy bounded by wait_limit_ns (in [1 us, 10 ms])
 * instead of 250 ms, and each warp's first page copy announced to its mbarrier as 16
 * bytes larger than it is, so the wait for it runs out.  The kernel then raises
 * KVQ_FLAG_WAIT_TIMEOUT in the workspace status word, stops waiting, writes empty partial
 * results (out is not the attention) and, before it leaves, completes the short phase
 * with a 16-byte copy of its own and waits for every copy it issued.  Nothing faults or
 * hangs; later calls run normally.  (No passage of the pages has a counterpart.)
 * Returns as kvq_decode_attention, or KVQ_EINVAL for a limit outside the range.
 */
int kvq_test_decode_wait_timeout(const kvq_cache_config *cfg, const void *pool, const void *q,
                                 const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens,
                                 int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                                 float *out, void *workspace, size_t workspace_bytes, uint64_t wait_limit_ns,
                                 kvq_stream_t stream);

/*
 * Dequantize positions [start, start + n) of sequence b (section 2.1 of the 4-bit
 * page: value = code * scale, exact in fp32).
 *   out_k, out_v  device [n, num_kv_heads, head_dim]; out_dtype 0 = fp16 (the fp32
 *                 value rounded to nearest even), 1 = fp32.
 *   status        device uint32 status word or NULL.
 * Returns KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED or KVQ_ECUDA.
 */
int kvq_dequantize(const kvq_cache_config *cfg, const void *pool, const int32_t *block_table,
                   int32_t max_blocks, int32_t b, int32_t start, int32_t n, void *out_k, void *out_v,
                   int32_t out_dtype, uint32_t *status, kvq_stream_t stream);

/*
 * Copy a device status word (a `status` argument, or the first 4 bytes of a decode
 * workspace) to *flags after the stream has reached this point (synchronizes the
 * stream).  Returns KVQ_OK, KVQ_EINVAL or KVQ_ECUDA.
 */
int kvq_read_status(const void *status_word, uint32_t *flags, kvq_stream_t stream);

/* The calling thread's last error message ("" if none).  Never NULL. */
const char *kvq_last_error(void);

/* Library version string. */
const char *kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
