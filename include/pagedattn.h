/*
 * pagedattn.h — C ABI of the GB300 (sm_103a) paged GQA attention library.
 *
 * The operation is attention of a Qwen3-style text decoder (GQA: 16 query heads share 8 KV
 * heads, head_dim 128) over a paged KV cache holding tens of thousands of audio-embedding
 * tokens, in its two modes:
 *   - decode: one query row per sequence against the sequence's whole cache
 *     ("Optimizing ASR Models to Transcribe 90-Minute Multi-Speaker Audio", section
 *     "Where Time Is Spent: Profiling": the autoregressive decode loop takes more than 94% of
 *     the time on long audio);
 *   - chunked prefill: a chunk of up to 4096 query rows attends causally to the cached prefix
 *     plus itself (same page, section "Chunked Prefill for Long Audio"; "MOSS-Transcribe-
 *     Diarize" cookbook, section "Inference Pipeline").
 * The new tokens' K/V are written into the cache before attention (prefill "builds its KV
 * cache": first page, section "ASR Model Primer").
 *
 * Definition (for every query row, query head h, visible keys t):
 *     s_t = scale * <q_h, k_t>,  o_h = sum_t softmax(s)_t v_t,  lse_h = ln sum_t exp(s_t)
 * where k_t, v_t are KV head h / (Hq / Hkv) of token t.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor arguments are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or keeps them. Scratch ("workspace") memory is caller-provided too.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream). The
 *    host never waits for the GPU inside a call, and grids depend only on host arguments,
 *    so calls may be captured in a CUDA graph.
 *  - Argument errors are returned synchronously, before anything is launched.
 *  - Errors that only the GPU can see (a block-table entry outside the pool, a length that
 *    does not fit the block table, a bounded wait that gave up) are OR-ed as PA_DEV_* bits
 *    into `*status`, a caller-owned device int32 (may be NULL: then they are not reported).
 *    The kernel then skips the offending access (page 0 is read instead of an out-of-range
 *    page, a too-long sequence is cut to what its table row covers), so no access ever
 *    leaves the buffers described below.
 *  - Supported shape: bf16 storage, head_dim 128, page_size 16, num_kv_heads 8,
 *    num_q_heads 16 (the decoder's GQA 16/8). Anything else returns PA_ERR_UNSUPPORTED.
 *
 * Layouts (row-major, contiguous, little-endian)
 *  - KV page pool (one K pool and one V pool per layer): bf16 [num_pages][16][Hkv][128].
 *    Token position p of sequence b lives in page block_table[b * bt_stride + p / 16],
 *    slot p % 16.
 *  - block_table: int32 [batch][bt_stride]; entries past ceil(seq_len / 16) are never read.
 *  - q and out: bf16 [rows][Hq][128]; lse: fp32 [rows][Hq] (natural log), may be NULL.
 */
#ifndef PAGEDATTN_H_
#define PAGEDATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* pa_stream_t;

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,         /* null pointer, negative size, inconsistent sizes        */
  PA_ERR_UNSUPPORTED = 2,         /* head counts, head_dim or page size not supported        */
  PA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below the matching *_workspace_size()  */
  PA_ERR_CUDA = 4                 /* a CUDA runtime call failed; see pa_last_error()         */
} pa_status;

/* Device-side error bits, OR-ed into the optional `status` word. */
#define PA_DEV_ERR_PAGE_OOB 1u /* a block-table entry needed by the call was not in [0, num_pages) */
#define PA_DEV_ERR_LENGTH 2u   /* a length did not fit: seq_len < 0 or > bt_stride*16, q_len > seq_len, ... */
#define PA_DEV_ERR_TIMEOUT 4u  /* a bounded wait inside a kernel gave up (the kernel returned early) */
#define PA_DEV_ERR_INTERNAL 8u /* a kernel found the GPU's layout not as built for (it did nothing) */

typedef struct pa_dims {
  int32_t num_q_heads;  /* Hq  (16) */
  int32_t num_kv_heads; /* Hkv (8)  */
  int32_t head_dim;     /* D   (128) */
  int32_t page_size;    /* tokens per page (16) */
} pa_dims;

/* ------------------------------------------------------------------------------------------
 * kv_append_paged — write the K/V rows of new tokens into the page pools.
 *
 * Source: prefill builds the KV cache and decode extends it by one token per step
 * ("Optimizing ASR Models to Transcribe 90-Minute Multi-Speaker Audio", section "ASR Model
 * Primer"; chunked prefill appends 4096 tokens per step, section "Chunked Prefill for Long
 * Audio").
 *
 *   k_new, v_new   bf16 [total_new][Hkv][128], new tokens packed by sequence
 *   cu_new_lens    int32 [batch+1]: sequence b owns rows cu_new_lens[b] .. cu_new_lens[b+1]-1
 *   start_pos      int32 [batch]: logical position of sequence b's first new token
 *   block_table    int32 [batch][bt_stride]; must already cover the new positions
 *   k_pool, v_pool bf16 [num_pages][16][Hkv][128], written in place
 * Row j of sequence b goes to position start_pos[b] + j. The copy is bit-exact; no other
 * pool byte changes. Rows at or past cu_new_lens[batch] are ignored. If cu_new_lens[batch]
 * exceeds total_new, only the first total_new rows are written and PA_DEV_ERR_LENGTH is set.
 * A position whose table entry is missing (past bt_stride) or out of range is skipped and
 * flagged.
 * ------------------------------------------------------------------------------------------ */
pa_status kv_append_paged(pa_dims dims, const void* k_new, const void* v_new, int32_t total_new,
                          const int32_t* cu_new_lens, const int32_t* start_pos, int32_t batch,
                          const int32_t* block_table, int32_t bt_stride, void* k_pool,
                          void* v_pool, int64_t num_pages, int32_t* status, pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * attn_decode_paged — one decode step: query row b attends to all seq_lens[b] cached keys.
 *
 * Source: the autoregressive decode of the transcript, one token at a time against the KV
 * cache ("MOSS-Transcribe-Diarize" cookbook, "Inference Pipeline" item 3; dominant share
 * of time per "Where Time Is Spent" on both the blog and the cookbook).
 *
 *   q            bf16 [batch][Hq][128]
 *   seq_lens     int32 [batch], keys per sequence (0 allowed: o = 0, lse = -inf)
 *   max_seq_len  host upper bound of seq_lens (<= 131072, the 128K context); a larger
 *                device value is cut to bt_stride*16 and flagged
 *   softmax_scale  any value but NaN (PA_ERR_INVALID_ARG); 1/sqrt(128) for this model
 *   out          bf16 [batch][Hq][128];  lse fp32 [batch][Hq] or NULL
 *   split_tokens   keys per split-KV range, rounded up to whole 16-token pages; 0 = auto (one
 *                equal share of all sequences' pages per SM). With a split size the ranges
 *                are that long (the last one shorter), raised if needed so that there are at
 *                most 64 ranges per SM; any value >= the batch's total keys gives one range.
 *                Negative: PA_ERR_INVALID_ARG. The result does not depend on it beyond
 *                rounding (the split-KV partials are merged exactly by log-sum-exp).
 *   workspace    device scratch of at least pa_decode_workspace_size(dims, batch, max_seq_len,
 *                split_tokens) bytes, 256-byte aligned; holds per-split partial results. With
 *                split_tokens = 0 the size does not depend on max_seq_len. Calls that share a
 *                workspace must not overlap on the GPU.
 * The key range of all sequences is laid end to end and cut into page ranges (split-KV);
 * partial (o, lse) pairs of sequences that span ranges are merged by log-sum-exp (two
 * kernels). With split_tokens = 0 a short batch (every (sequence, KV head) pair, or pair of
 * two KV heads when there are more pairs than SMs, can have a resident cluster of up to 8
 * CTAs, each holding at most 64 pages) is served by one kernel instead: each cluster splits
 * its pages and merges in distributed shared memory; the workspace is then not touched.
 * ------------------------------------------------------------------------------------------ */
size_t pa_decode_workspace_size(pa_dims dims, int32_t batch, int32_t max_seq_len,
                                int32_t split_tokens);

/* Kernels one attn_decode_paged call with these arguments launches on the current device: 1
 * (single-launch short-batch path) or 2 (split kernel + merge); 0 for unsupported dims or
 * batch <= 0. For sizing CUDA graphs and counting launches; computes nothing on the GPU. */
int32_t pa_decode_kernels_per_call(pa_dims dims, int32_t batch, int32_t max_seq_len,
                                   int32_t split_tokens);

pa_status attn_decode_paged(pa_dims dims, const void* q, const void* k_pool, const void* v_pool,
                            int64_t num_pages, const int32_t* block_table, int32_t bt_stride,
                            const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                            float softmax_scale, int32_t split_tokens, void* out, float* lse,
                            void* workspace, size_t workspace_bytes, int32_t* status,
                            pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * attn_decode_paged_noalloc — attn_decode_paged without a caller-provided workspace.
 *
 * The pages have no counterpart of this call; it exists for callers that cannot allocate
 * device memory: an engine that reserved all free HBM for its own KV-cache pool up front (a
 * cudaMalloc would fail), a plugin host that exposes no device allocator, or a latency-critical
 * loop in which cudaMalloc / cudaFree may synchronize the device. The caller still provides q,
 * the pools, block_table, seq_lens, out and lse exactly as for attn_decode_paged; this call
 * itself allocates nothing and calls no allocating routine.
 *
 * The split size is automatic (split_tokens = 0 of attn_decode_paged).
 * Scratch lives in one fixed 4.5 MiB device array inside the library, held until the process
 * exits by every GPU on which the library's decode code has been loaded. Limit:
 * pa_decode_workspace_size(dims, batch, max_seq_len, 0) must not exceed 4.5 MiB (batch up to
 * about 400 on a 152-SM GB300); larger batches return PA_ERR_WORKSPACE_TOO_SMALL with the
 * sizes in pa_last_error().
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current) and caches it. Under CUDA's default lazy module loading that is
 * also when the device code of this part of the library is loaded and the 4.5 MiB are
 * committed on the device, unless an earlier call of attn_decode_paged on that device already
 * loaded it. So make the first call before reserving all free device memory for something
 * else, and before any stream capture; a call with batch = 0 does only this set-up.
 * Every call shares the one array and no call needs it zeroed (each call writes every scratch
 * byte it later reads), so calls that overlap on the GPU (different streams, or several host
 * threads) race on it and must be serialized by the caller.
 * ------------------------------------------------------------------------------------------ */
pa_status attn_decode_paged_noalloc(pa_dims dims, const void* q, const void* k_pool,
                                    const void* v_pool, int64_t num_pages,
                                    const int32_t* block_table, int32_t bt_stride,
                                    const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                    float softmax_scale, void* out, float* lse, int32_t* status,
                                    pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * attn_prefill_chunk — causal attention of query chunks over their cached prefix + themselves.
 *
 * Source: chunked prefill of long audio prompts in 4096-token pieces ("Optimizing ASR Models
 * to Transcribe 90-Minute Multi-Speaker Audio", section "Chunked Prefill for Long Audio").
 *
 *   q           bf16 [total_q][Hq][128], chunks packed by sequence
 *   cu_q_lens   int32 [batch+1]: chunk b owns rows cu_q_lens[b] .. cu_q_lens[b+1]-1
 *   seq_lens    int32 [batch]: keys of sequence b INCLUDING the chunk (appended first)
 *   batch       number of chunks, at most 128 per call
 *   max_q_len   host upper bound of the chunk lengths
 *   softmax_scale  0 < scale < 1e30, else PA_ERR_INVALID_ARG (the causal mask sets raw
 *               scores to -inf before scaling, which needs a positive, finite scale)
 * Query i of chunk b (length n) sits at position seq_lens[b] - n + i and sees keys
 * 0 .. seq_lens[b] - n + i (bottom-right causal alignment). A chunk longer than its sequence
 * is flagged and produces nothing.
 *   out bf16 [total_q][Hq][128]; lse fp32 [total_q][Hq] or NULL.
 *   workspace: at least pa_prefill_workspace_size(...) bytes, 256-byte aligned (split-work
 *   partials; about 40 MB on a 152-SM GPU, independent of the batch). Calls that share a
 *   workspace must not overlap on the GPU.
 * ------------------------------------------------------------------------------------------ */
size_t pa_prefill_workspace_size(pa_dims dims, int32_t batch, int32_t max_q_len,
                                 int32_t max_seq_len);

pa_status attn_prefill_chunk(pa_dims dims, const void* q, const int32_t* cu_q_lens,
                             int32_t total_q, const void* k_pool, const void* v_pool,
                             int64_t num_pages, const int32_t* block_table, int32_t bt_stride,
                             const int32_t* seq_lens, int32_t batch, int32_t max_q_len,
                             int32_t max_seq_len, float softmax_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t* status,
                             pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * attn_decode_paged_ex / attn_prefill_chunk_ex — the two attention calls with a grid cap.
 *
 * Source: the serving pages' scheduler runs a prompt chunk and other requests' decode steps in
 * the same step ("Optimizing ASR Models to Transcribe 90-Minute Multi-Speaker Audio", section
 * "Chunked Prefill for Long Audio"). The chunk's attention is bound by the tensor cores and the
 * decodes' by HBM bandwidth, so a caller can run the two side by side, on two streams, each
 * call held to its own share of the SMs: the two bounds then overlap instead of adding up.
 *
 * The arguments are those of attn_decode_paged / attn_prefill_chunk plus opts (NULL = the
 * plain call):
 *   opts->max_ctas  > 0: the call's persistent grid has at most this many CTAs (each occupies
 *                   one SM); 0: one per SM, as the plain call; < 0: PA_ERR_INVALID_ARG.
 *                   The workspace sizes of the plain calls cover every cap. A decode batch
 *                   that the single-launch path would serve takes it only if its CTAs fit
 *                   under the cap, else the split path runs with the capped grid.
 * Results equal the plain call's up to rounding (a smaller grid cuts the key ranges
 * differently). Ordering between the two streams is the caller's (e.g. an event recorded after
 * kv_append_paged, waited on by the second stream, and one recorded on the second stream after
 * its call, waited on by the first before the next layer); all of it can be captured in one
 * CUDA graph.
 * ------------------------------------------------------------------------------------------ */
typedef struct {
  int32_t max_ctas;
} pa_launch_opts;

pa_status attn_decode_paged_ex(pa_dims dims, const void* q, const void* k_pool,
                               const void* v_pool, int64_t num_pages, const int32_t* block_table,
                               int32_t bt_stride, const int32_t* seq_lens, int32_t batch,
                               int32_t max_seq_len, float softmax_scale, int32_t split_tokens,
                               void* out, float* lse, void* workspace, size_t workspace_bytes,
                               int32_t* status, pa_stream_t stream, const pa_launch_opts* opts);

pa_status attn_prefill_chunk_ex(pa_dims dims, const void* q, const int32_t* cu_q_lens,
                                int32_t total_q, const void* k_pool, const void* v_pool,
                                int64_t num_pages, const int32_t* block_table, int32_t bt_stride,
                                const int32_t* seq_lens, int32_t batch, int32_t max_q_len,
                                int32_t max_seq_len, float softmax_scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, int32_t* status,
                                pa_stream_t stream, const pa_launch_opts* opts);

/* ------------------------------------------------------------------------------------------
 * attn_merge_lse — combine attention results computed over disjoint key sets.
 *
 * Source: the split-KV form of the decode step (long caches are cut into key ranges whose
 * softmax states are merged exactly): with lse = ln sum_s exp(lse_s),
 *     o = sum_s exp(lse_s - lse) * o_s.
 * Parts with lse_s = -inf carry no weight (their o_s is never read); if all parts are empty
 * the result is o = 0, lse = -inf.
 *
 *   o_parts    fp32 [num_parts][rows][heads][head_dim], each part normalised on its own
 *   lse_parts  fp32 [num_parts][rows][heads]
 *   out        bf16 [rows][heads][head_dim];  lse_out fp32 [rows][heads] or NULL
 * head_dim must be a multiple of 4 (<= 1024).
 * ------------------------------------------------------------------------------------------ */
pa_status attn_merge_lse(int32_t num_parts, int32_t rows, int32_t heads, int32_t head_dim,
                         const float* o_parts, const float* lse_parts, void* out,
                         float* lse_out, pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * adaptor_mlp_merge4 — the audio-text bridge that turns encoder frames into decoder embeddings.
 *
 * Source: 4x temporal merge (concatenate every 4 encoder frames, d_model 1024 -> 4096) and an
 * FFN adapter Linear -> SiLU -> Linear -> LayerNorm, 4096 -> 1024 ("Optimizing ASR Models to
 * Transcribe 90-Minute Multi-Speaker Audio", "ASR Model Primer"; "MOSS-Transcribe-Diarize
 * 0.9B", "Model Architecture"). The hidden width is not stated; it is 1024 here:
 *     x = frames viewed as [T][4096] (T = num_frames / 4; no copy is made)
 *     out = LayerNorm(SiLU(x W1^T + b1) W2^T + b2) * gamma + beta   (biased variance, eps)
 *
 *   frames   bf16 [num_frames][1024], num_frames a multiple of 4
 *   w1       bf16 [1024][4096] (out, in);  b1 fp32 [1024]
 *   w2       bf16 [1024][1024] (out, in);  b2 fp32 [1024]
 *   gamma, beta  fp32 [1024];  eps >= 0
 *   out      bf16 [T][1024]
 *   workspace    at least pa_adaptor_workspace_size(num_frames) bytes (the bf16 hidden
 *                activations, [T][1024]); 16-byte aligned.
 * frames, w1, w2, gamma, beta, out and workspace must be 16-byte aligned, else
 * PA_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------------------------ */
size_t pa_adaptor_workspace_size(int32_t num_frames);

pa_status adaptor_mlp_merge4(int32_t num_frames, const void* frames, const void* w1,
                             const float* b1, const void* w2, const float* b2,
                             const float* gamma, const float* beta, float eps, void* out,
                             void* workspace, size_t workspace_bytes, int32_t* status,
                             pa_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * pa_debug_decode_starve — test hook for the bounded waits; never needed in production.
 *
 * With enable != 0, every later attn_decode_paged launch made by the calling host thread bounds
 * each of its mbarrier waits by 1 ms (instead of 2 s) and leaves the first ring stage of CTA 0
 * unfilled, so that CTA's consumer warps give up waiting, set PA_DEV_ERR_TIMEOUT in *status and
 * return (the producer drains its copies first; the decode kernels hold no tensor-memory
 * state). The output of such a call is undefined. enable = 0 restores normal launches.
 * ------------------------------------------------------------------------------------------ */
pa_status pa_debug_decode_starve(int32_t enable);

/* Read and clear the device status word: waits for `stream`, copies *status to *flags_out,
 * then zeroes it. */
pa_status pa_read_device_status(int32_t* status, uint32_t* flags_out, pa_stream_t stream);

/* Static text for a status code. */
const char* pa_status_string(pa_status s);

/* Text of the last CUDA error seen by a call of the calling host thread ("" if none). */
const char* pa_last_error(void);

/* Library ABI version (major * 100 + minor). */
int32_t pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H_ */
