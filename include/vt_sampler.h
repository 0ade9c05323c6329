/* vt_sampler.h -- C ABI of the GB300 batched decode sampler.
 *
 * One call of vt_sample turns a [B, V] logits tensor that lives in device
 * memory into one next token per row.  The per-row pipeline, in this order:
 *
 *   1. occurrence penalties from the row's token counts over the prompt plus
 *      everything generated so far: repetition (divide a non-negative logit by
 *      the penalty, multiply a negative one), then frequency (subtract
 *      frequency * count), then presence (subtract once when count > 0)
 *      [TensorRT-LLM "Sampling" page, LLM API sampling behaviour, occurrence
 *      penalties];
 *   2. temperature: z_t = z * (1.0f / T) [same page: logits scaled by
 *      1/temperature]; T = 0, top_k = 1, top_p = 0 or min_p = 1 make the row
 *      greedy whatever its other settings [same page], and a greedy row uses
 *      T = 1;
 *   3. log-softmax log-probs of z_t over the whole row [Tenstorrent sampling
 *      README, LogProbsCalculator: global max, then sum-exp] and the top-n
 *      log-probs [TensorRT-LLM "Sampling", TopK LogProbs];
 *   4. filters on the order (z_t descending, index ascending): min-p first,
 *      then top-k, then top-p over the top-k survivors renormalised [TensorRT-
 *      LLM "Sampling": min-p, top-k and top-p bullets];
 *   5. the draw: token = argmax over kept j of z_t,j - ln(-ln u_j), where u_j
 *      is a SplitMix64 stream keyed by (seed, row, j); equal scores go to the
 *      lowest index; a greedy row takes the lowest-index argmax [vllm.cpp pull
 *      request "the Gumbel draw that scanned 248,320 tokens on one thread":
 *      GumbelScore, ExpNoise, ArgReduce comparing true global indices].
 *
 * The state carried between calls follows the reset-then-sample shape of the
 * Tenstorrent SamplingGenerator (reset_sampling_params, reset_seed,
 * reset_prompt_tokens / reset_output_state, sample): per-row parameters and
 * seeds (vt_reset_params) and per-row token counts (vt_reset_token_counts).
 * Each vt_sample call advances every sampled row's seed once and, on request,
 * adds the drawn token to the row's counts.
 *
 * Conventions for every entry point:
 *   - The return value is VT_OK (0) or a negative VT_ERR_* code; nothing is
 *     thrown across the ABI.  vt_last_error() gives a message for the last
 *     failure on a handle.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued on it in stream order; unless stated, calls do
 *     not wait for the GPU, and the caller synchronises the stream before
 *     reading device outputs.
 *   - "host" pointers are ordinary CPU memory, read before the call returns;
 *     the caller keeps ownership.  "device" pointers are CUDA device memory
 *     on the handle's device, owned by the caller.
 *   - A handle is not thread-safe: one host thread at a time.
 */
#ifndef VT_SAMPLER_H
#define VT_SAMPLER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define VT_OK 0
#define VT_ERR_INVALID_ARG (-1) /* a bad pointer, size or parameter value      */
#define VT_ERR_STATE (-2)       /* a call out of order (sample before reset)   */
#define VT_ERR_CAPACITY (-3)    /* a size beyond the capacities given at create */
#define VT_ERR_CUDA (-4)        /* a CUDA runtime call failed                   */
#define VT_ERR_TIMEOUT (-5)     /* a bounded device wait ran out                */

/* ---- logits element types ----------------------------------------------- */
#define VT_DTYPE_F32 0  /* IEEE binary32                                        */
#define VT_DTYPE_BF16 1 /* bfloat16 (the top 16 bits of a binary32), widened exactly */

/* ---- per-row status written by vt_sample (see vt_get_row_status) ------- */
#define VT_ROW_OK 0           /* token drawn                                    */
#define VT_ROW_NONFINITE 1    /* a NaN or +inf among the tempered logits; token -1 */
#define VT_ROW_EMPTY 2        /* no finite tempered logit (all -inf); token -1   */
#define VT_ROW_HISTORY_FULL 3 /* token drawn, but the row's count table was full,
                                 so update_counts could not record it            */

typedef struct vt_sampler vt_sampler; /* opaque handle */

typedef struct vt_sampler_config {
  int32_t max_batch;    /* largest B of any call, >= 1                          */
  int32_t max_vocab;    /* largest V of any call, 1..1048576                     */
  int32_t max_logprobs; /* largest num_logprobs, 0..32                          */
  int32_t max_history;  /* per-row capacity of the count table in distinct ids,
                           and the largest prompt + output length per row at a
                           counts reset; 0..32768                               */
  int32_t device;       /* CUDA device ordinal                                  */
  int32_t host_io;      /* 1: also allocate device staging for vt_sample_host   */
} vt_sampler_config;

/* Create a sampler: validates the capacities, makes `device` current, and
 * allocates every piece of device scratch and pinned host staging the handle
 * will ever use (no later call allocates).  On success *out owns all of it.
 * Errors: VT_ERR_INVALID_ARG (null pointer, capacity out of range),
 * VT_ERR_CUDA (no such device, out of memory, not an sm_103 GPU). */
int vt_sampler_create(const vt_sampler_config* config, vt_sampler** out);

/* Free everything the handle owns.  Waits for the handle's pending work.
 * NULL is ignored. */
void vt_sampler_destroy(vt_sampler* handle);

/* Upload per-row sampling parameters and seeds for rows 0..B-1 (host arrays
 * of length B).  Row r's seed is the seed its next vt_sample call keys its
 * noise stream with; each vt_sample advances it by 0x9E3779B97F4A7C15.
 *   temperature  >= 0 and finite; 0 means greedy; 1.0f/T must be finite.
 *   top_k        >= 0; 0 or >= V disables; 1 means greedy.
 *   top_p        in [0, 1]; 1 disables; 0 means greedy.
 *   min_p        in [0, 1]; 0 disables; 1 means greedy.
 *   presence, frequency  finite (0 disables).
 *   repetition   finite and > 0 (1 disables).
 * Errors: VT_ERR_INVALID_ARG (any value out of range; nothing uploaded),
 * VT_ERR_CAPACITY (B > max_batch), VT_ERR_CUDA (the upload failed: the handle
 * then holds no parameters, and vt_sample returns VT_ERR_STATE until the next
 * successful reset).  For tests of these failure paths, the environment
 * variable VT_FAULT_INJECT=upload makes the upload fail, and
 * VT_FAULT_INJECT=alloc:<n> makes the n-th (0-based) device allocation of
 * vt_sampler_create fail; nothing on the device is made to fault. */
int vt_reset_params(vt_sampler* handle, int32_t B, const float* temperature,
                    const int32_t* top_k, const float* top_p, const float* min_p,
                    const float* presence, const float* frequency,
                    const float* repetition, const uint64_t* seed, void* stream);

/* vt_reset_params plus top-p decay [TensorRT-LLM "Sampling", LLM API sampling
 * behaviour, top-p decay].  Each of the three arrays is a host array of B
 * entries, or NULL for its default:
 *   top_p_decay      in (0, 1]; 1 disables (default 1).
 *   top_p_min        in (0, 1]; the floor of the decayed top_p (default 1e-6).
 *   top_p_reset_ids  >= -1; -1 never matches a token (default -1).
 * A row with top_p_decay < 1 that is not greedy (the greedy triggers above take
 * precedence) samples as a top-p row with an effective top_p that starts at its
 * top_p (1 when top_p is 1).  After each vt_sample that draws a token for the
 * row, the effective top_p becomes the row's top_p when the token equals
 * top_p_reset_ids, else max(top_p_eff * top_p_decay, top_p_min), in fp32; a
 * row the call could not sample (status != 0) keeps it.  The state lives on
 * the device and carries across vt_sample calls until the next reset.
 * Errors as vt_reset_params (any value out of range: nothing uploaded). */
int vt_reset_params_ex(vt_sampler* handle, int32_t B, const float* temperature,
                       const int32_t* top_k, const float* top_p, const float* min_p,
                       const float* presence, const float* frequency,
                       const float* repetition, const uint64_t* seed,
                       const float* top_p_decay, const float* top_p_min,
                       const int32_t* top_p_reset_ids, void* stream);

/* Read the effective top_p of rows 0..B-1 into a host array (B of the last
 * reset): the decayed value for rows with top-p decay, top_p for the others.
 * Synchronises the handle's last stream.  Errors: VT_ERR_INVALID_ARG (null
 * pointer), VT_ERR_STATE (no reset yet), VT_ERR_CUDA. */
int vt_read_top_p(vt_sampler* handle, float* host_top_p);

/* Rebuild the token counts of rows 0..B-1 from host CSR arrays: row r's prompt
 * ids are prompt_ids[prompt_offsets[r] .. prompt_offsets[r+1]), likewise its
 * output ids (offsets: B+1 entries, non-decreasing, starting at 0).  The counts
 * of a row are the multiset counts over both.  Ids must lie in
 * [0, max_vocab); a vt_sample call with a smaller V ignores ids >= V.
 * Errors: VT_ERR_INVALID_ARG (bad offsets or ids), VT_ERR_CAPACITY (B >
 * max_batch, or a row with more than max_history ids), VT_ERR_CUDA. */
int vt_reset_token_counts(vt_sampler* handle, int32_t B, const int32_t* prompt_ids,
                          const int64_t* prompt_offsets, const int32_t* output_ids,
                          const int64_t* output_offsets, void* stream);

/* vt_reset_token_counts with each row's prompt_ignore_length (TensorRT-LLM
 * "Sampling", occurrence penalties): the first prompt_ignore_length[r] prompt
 * ids of row r are left out of the presence and frequency counts and still
 * count for the repetition penalty.  Values <= 0 leave none out; values
 * beyond the row's prompt leave the whole prompt out.  prompt_ignore_length
 * is a host array of B entries, or NULL (none left out: vt_reset_token_counts).
 * A token the call appends to the counts (update_counts) always counts for
 * all three.  Errors as vt_reset_token_counts. */
int vt_reset_token_counts_ex(vt_sampler* handle, int32_t B, const int32_t* prompt_ids,
                             const int64_t* prompt_offsets, const int32_t* output_ids,
                             const int64_t* output_offsets, const int32_t* prompt_ignore_length,
                             void* stream);

/* Sample one token for each of rows 0..B-1.
 *   logits            device [B][ld] elements of `dtype`; row r starts at
 *                     logits + r*ld; only columns [0, V) are read.  Rows whose
 *                     start is 16-byte aligned (base pointer and ld * element
 *                     size multiples of 16) are staged with bulk copies; other
 *                     layouts are read with plain loads (slower, same result).
 *   V, ld             1 <= V <= max_vocab, ld >= V.
 *   num_logprobs      0..max_logprobs top log-probs per row.
 *   update_counts     nonzero: add each row's drawn token to its counts.
 *   out_tokens        device int32[B]: token id, or -1 for a row with status
 *                     NONFINITE or EMPTY.
 *   out_logprobs      device float[B]: log-softmax of z_t at the token (NaN for
 *                     a row without a token); may be NULL.
 *   out_topk_ids      device int32[B][num_logprobs] and
 *   out_topk_logprobs device float[B][num_logprobs]: the num_logprobs first
 *                     tokens of the order (z_t descending, index ascending)
 *                     and their log-probs; -1 / NaN for a row without a token;
 *                     may be NULL only when num_logprobs == 0.
 * The call enqueues device work only: it allocates nothing, does not
 * synchronise, and may be captured into a CUDA graph.  A bf16 call over all
 * the rows of the last vt_reset_params may run its top-p-only rows on a
 * stream of the handle: it forks from `stream` and joins back into it through
 * events, so that all of the call's work is ordered on `stream`.
 * Errors: VT_ERR_STATE (no vt_reset_params yet, B larger than the rows given
 * there, or a row with penalties whose counts were never reset),
 * VT_ERR_INVALID_ARG, VT_ERR_CAPACITY, VT_ERR_CUDA (launch failure).  Device-
 * side faults of the call (a bounded wait that ran out) are reported by
 * vt_check_device_errors. */
int vt_sample(vt_sampler* handle, const void* logits, int32_t dtype, int32_t B, int32_t V,
              int64_t ld, int32_t num_logprobs, int32_t update_counts, int32_t* out_tokens,
              float* out_logprobs, int32_t* out_topk_ids, float* out_topk_logprobs,
              void* stream);

/* vt_sample plus the filtered distribution each row drew from, on request
 * [TensorRT-LLM "Sampling", Performance: the full set of token probabilities
 * after the top-k / top-p masking, computed only when the user asks for it,
 * e.g. for rejection sampling].
 *   out_probs  device fp32 [B][ld_probs] (ld_probs >= V; columns [V, ld_probs)
 *              are not written), or NULL (then this is vt_sample).  Row r
 *              receives exp(z_t,j - m) / sum over the kept set of
 *              exp(z_t - m) for j in the row's kept set after min-p, top-k
 *              and top-p (m the row maximum of z_t), 0 elsewhere; a one-hot
 *              vector at the token on a greedy row; NaN everywhere on a row
 *              with status VT_ROW_NONFINITE or VT_ROW_EMPTY.  fp32 arithmetic:
 *              each entry within a relative 3e-5 of the exact value.
 * The distribution uses the counts the draw saw: with update_counts the
 * tokens are appended after it.  Two extra launches (three with
 * update_counts) read the logits twice more.  Errors as vt_sample, plus
 * VT_ERR_INVALID_ARG for ld_probs < V. */
int vt_sample_ex(vt_sampler* handle, const void* logits, int32_t dtype, int32_t B, int32_t V,
                 int64_t ld, int32_t num_logprobs, int32_t update_counts, int32_t* out_tokens,
                 float* out_logprobs, int32_t* out_topk_ids, float* out_topk_logprobs,
                 float* out_probs, int64_t ld_probs, void* stream);

/* vt_sample from host memory: vt_sample_host_async, then vt_sample_host_wait
 * (the outputs are in the host arrays when it returns).  Errors as vt_sample,
 * plus VT_ERR_STATE when the handle has no host staging (host_io = 0). */
int vt_sample_host(vt_sampler* handle, const void* host_logits, int32_t dtype, int32_t B,
                   int32_t V, int64_t ld, int32_t num_logprobs, int32_t update_counts,
                   int32_t* host_tokens, float* host_logprobs, int32_t* host_topk_ids,
                   float* host_topk_logprobs, void* stream);

/* One step from host memory without waiting: host logits [B][ld] (pinned
 * memory for an asynchronous copy) are copied into the next of the handle's
 * two device staging slots on the handle's own copy stream, the step samples
 * on `stream` once they are there, and the outputs (vt_sample's shapes) are
 * copied back into the host arrays on `stream`.  So the copy-in of one step
 * runs while the previous step samples; a slot is reused only after its
 * previous step's output copies are done (the copy stream waits for it on the
 * device).  Steps keep their call order: seeds and counts advance as with
 * vt_sample.  The host buffers must stay valid, and the outputs are not to be
 * read, until vt_sample_host_wait returns.  Errors as vt_sample_host (raised
 * before anything is enqueued). */
int vt_sample_host_async(vt_sampler* handle, const void* host_logits, int32_t dtype, int32_t B,
                         int32_t V, int64_t ld, int32_t num_logprobs, int32_t update_counts,
                         int32_t* host_tokens, float* host_logprobs, int32_t* host_topk_ids,
                         float* host_topk_logprobs, void* stream);

/* Wait until every step enqueued by vt_sample_host_async is complete (its
 * outputs in the host arrays), then vt_check_device_errors. */
int vt_sample_host_wait(vt_sampler* handle);

/* Synchronise the handle's last stream and report device-side faults raised
 * since the previous check: VT_ERR_TIMEOUT when a bounded wait inside a kernel
 * ran out (the kernel then returned early and its outputs are not valid),
 * VT_OK otherwise.  Clears the device error word.  vt_sample_host calls it. */
int vt_check_device_errors(vt_sampler* handle);

/* Copy the row status of the last vt_sample (VT_ROW_*) into device int32[B]
 * (B of that call). */
int vt_get_row_status(vt_sampler* handle, int32_t* dev_status, void* stream);

/* Test and debug view of the last vt_sample, per row, into device arrays of
 * that call's B: the tempered logit and index of the last kept element of the
 * order after min-p, top-k and top-p, and the number of kept elements (1 for a
 * greedy row; 0 for a row without a token). */
int vt_debug_filter_boundary(vt_sampler* handle, float* kth_value, int32_t* kth_index,
                             int32_t* kept_count, void* stream);

/* Read row `row`'s count table into host arrays of `capacity` entries: the
 * distinct ids in increasing order and their counts; *n_unique is set to the
 * table length (entries beyond capacity are not written).  Synchronises the
 * handle's last stream. */
int vt_debug_get_counts(vt_sampler* handle, int32_t row, int32_t* ids, int32_t* counts,
                        int32_t capacity, int32_t* n_unique);

/* Debug: the launch shape vt_sample would use for (dtype, V), the B of the last
 * vt_reset_params (max_batch before any) and rows without penalties: CTAs per
 * row, logits elements per CTA and dynamic shared memory per CTA. */
int vt_debug_launch_shape(vt_sampler* handle, int32_t dtype, int32_t V, int32_t* ctas_per_row,
                          int32_t* slice_elems, int64_t* smem_bytes);

/* Debug, no device needed: the grid vt_sample_ex uses for the filtered
 * distribution of B rows of V on a GPU of num_sms SMs: CTAs per row
 * (*splits) and elements per CTA (*range, a multiple of 64).  A handle
 * created for (max_batch, max_vocab) holds the partials of every B <= max_batch
 * and V <= max_vocab.  Errors: VT_ERR_INVALID_ARG (a size below 1, null
 * pointer). */
int vt_debug_probs_plan(int32_t B, int32_t V, int32_t num_sms, int32_t* splits, int32_t* range);

/* Debug: phase trace.  With a device buffer of capacity_ctas * slots_per_cta
 * uint64 entries set, each later vt_sample whose grid fits writes, per CTA,
 * the GPU global timer (ns) at each phase boundary (slots not reached keep
 * their old value): the streaming kernel's CTA (row * CTAs per row + rank)
 * writes entry row * CTAs per row + rank.  *slots_per_cta receives the slot
 * count.  NULL turns it
 * off.  The buffer stays owned by the caller and must outlive its use. */
int vt_debug_set_trace(vt_sampler* handle, uint64_t* dev_trace, int64_t capacity_ctas,
                       int32_t* slots_per_cta);

/* Debug: record `event` (a cudaEvent_t passed as void*) on the stream of each
 * later vt_sample between its two launches (the streaming kernel, then the
 * selection kernel for the rows handed over), so that a caller can time the
 * two apart.  NULL turns it off.  The event stays owned by the caller. */
int vt_debug_set_phase_event(vt_sampler* handle, void* event);

/* Debug: how many rows the last vt_sample handed from the streaming kernel to
 * the selection kernel (rows whose kept set or top-n the candidates gathered
 * in one pass could not settle).  Synchronises the handle's last stream. */
int vt_debug_last_handover(vt_sampler* handle, int32_t* rows);

/* Debug: run the bounded-wait path to its end.  One thread waits on a barrier
 * that nothing completes for limit_ns (1 ns .. 1 s) of the GPU timer, as the
 * sampling kernels' bounded waits do, then records a timeout in the handle's
 * error word and returns, leaving the context usable; the next
 * vt_check_device_errors returns VT_ERR_TIMEOUT.  Stream-ordered on `stream`.
 * Errors: VT_ERR_INVALID_ARG, VT_ERR_CUDA. */
int vt_debug_wait_probe(vt_sampler* handle, int64_t limit_ns, void* stream);

/* Debug: which sampling path later vt_sample calls take.  1 (the default):
 * every call runs the streaming kernel (and its hand-over to the selection
 * kernel).  2: bf16 calls without penalties, top-p decay or the exported
 * distribution, on 16-byte aligned rows, run the six flat kernels (per-slice
 * statistics, per-row thresholds, per-slice candidates and code-slot counts,
 * per-row completion, and for top-p rows a fine count and the boundary), the
 * rows they cannot settle handed to the selection kernel; other calls run the
 * streaming kernel.  Both give the same tokens and kept sets.
 * Errors: VT_ERR_INVALID_ARG. */
int vt_debug_set_path(vt_sampler* handle, int32_t path);

/* Debug: how many kernels the last vt_sample launched: 2 on one stream (the
 * streaming kernel, then the selection kernel), 7 on the flat path (one more
 * when it appends the tokens to the counts), or 3 when the call split its
 * rows between the handle's two streams (the selection kernel alone, taking
 * its rows' statistics itself, on the second stream; the pair on the first).
 * 0 before the first call.  Does not synchronise. */
int vt_debug_last_launches(vt_sampler* handle, int32_t* launches);

/* Read the current per-row seeds of rows 0..B-1 into a host array (B of the
 * last vt_reset_params).  Synchronises the handle's last stream. */
int vt_debug_get_seeds(vt_sampler* handle, uint64_t* host_seeds);

/* ---- sampling without any allocation -------------------------------------
 * The sampling pages have no counterpart of this entry point.  It serves
 * callers that may not allocate device memory: an engine that reserves nearly all of it
 * for its KV cache at start-up, a host whose device memory belongs to a
 * framework's caching allocator, a decode loop that keeps cudaMalloc and
 * cudaFree (which waits for the whole device) out of its step.  Such callers
 * cannot create a handle, because vt_sampler_create allocates its buffers.
 *
 * vt_sample_noalloc runs the same sampling kernel as vt_sample, for rows
 * without penalties, and allocates nothing: it calls no cudaMalloc, cudaFree
 * or allocating library routine.  Its per-row state lives in one fixed
 * device array of VT_NOALLOC_SCRATCH_BYTES inside the library, which every
 * call on a device shares.  Calls whose GPU work overlaps (other streams,
 * other host threads) race on that array and give undefined results; calls on
 * one stream, one after another, are safe.
 *
 *   device        CUDA device ordinal; it is made current during the call
 *   logits        device [B][ld] of dtype, as in vt_sample
 *   temperature, top_k, top_p, min_p, seed
 *                 host arrays [B], the values vt_reset_params takes (no
 *                 penalties).  seed[r] keys row r's noise exactly as a handle
 *                 whose seed for row r is seed[r]; the caller advances its own
 *                 seeds (a handle adds 0x9E3779B97F4A7C15 per call).
 *   num_logprobs, out_tokens, out_logprobs, out_topk_ids, out_topk_logprobs
 *                 as in vt_sample (device memory owned by the caller)
 *   row_status    device int32[B] receiving VT_ROW_* per row, or NULL
 *   synchronize   nonzero: wait for the stream and report a device-side
 *                 timeout as VT_ERR_TIMEOUT; zero: return after enqueueing
 *                 (device-side faults then go unreported)
 *   errbuf        host buffer of errbuf_len bytes for a message, or NULL
 * The parameters are uploaded from pageable host memory, so the call waits
 * for work already queued on `stream` before it enqueues its own.
 * Errors: VT_ERR_CAPACITY when B > VT_NOALLOC_MAX_BATCH (checked before any
 * CUDA call) or V needs more shared memory than a CTA has; VT_ERR_INVALID_ARG;
 * VT_ERR_CUDA (wrong architecture, failed set-up or launch). */
#define VT_NOALLOC_MAX_BATCH 1024          /* rows per vt_sample_noalloc call  */
#define VT_NOALLOC_SCRATCH_BYTES (112 * 1024) /* the fixed device scratch array */
int vt_sample_noalloc(int32_t device, const void* logits, int32_t dtype, int32_t B, int32_t V,
                      int64_t ld, const float* temperature, const int32_t* top_k,
                      const float* top_p, const float* min_p, const uint64_t* seed,
                      int32_t num_logprobs, int32_t* out_tokens, float* out_logprobs,
                      int32_t* out_topk_ids, float* out_topk_logprobs, int32_t* row_status,
                      int32_t synchronize, void* stream, char* errbuf, int32_t errbuf_len);

/* ---- the vocabulary split over several devices ---------------------------
 * The Tenstorrent sampling README splits a row's logits over devices: each
 * device takes the top-k of its own slice (TTSampling), the candidates are
 * all-gathered, and the log-probs combine the devices' global maxima and sums
 * of exponentials (LogProbsCalculator).  The draw composes exactly because the
 * noise of column j is keyed by the global row and the global column (vllm.cpp
 * pull request "the Gumbel draw that scanned 248,320 tokens on one thread":
 * ArgReduce over true global indices).  Protocol, per step:
 *   1. every shard calls vt_shard_partials on its columns [v0, v0 + Vs) of the
 *      rows, writing one record of vt_shard_part_bytes(K) bytes per row;
 *   2. the caller all-gathers the S shards' records into one device buffer
 *      [S][B] records, shard s at s * B records (e.g. an NCCL all-gather);
 *   3. vt_shard_merge on that buffer writes the rows' tokens, log-probs and
 *      top-n exactly as vt_sample on the whole rows would (tokens and kept sets
 *      identical; log-probs equal within rounding), and advances the seeds.
 * Every shard's handle must hold the same parameters and seeds (the same
 * vt_reset_params).  Rows it takes: no penalties, no top-p decay; greedy
 * rows; rows without a filter (every finite element kept: the draw is the
 * best of the shards' Gumbel winners); and filtered rows bounded by
 * 1 < top_k <= K (top_k < V), after which min-p and top-p apply over the
 * gathered records.  Other rows: VT_ERR_INVALID_ARG.  The union of the
 * shards' K largest elements holds the row's K largest, hence a bounded
 * row's kept set, and every row's top-n. */
#define VT_SHARD_MAX_K 256
/* Records one merge gathers per row at most: S * K <= VT_SHARD_MAX_RECORDS. */
#define VT_SHARD_MAX_RECORDS 4096

/* Bytes of one row's record in a shard buffer for 1 <= K <= VT_SHARD_MAX_K
 * (-1 otherwise): a 48-byte header, then K uint64 elements.  The header:
 *   float    the shard's tempered maximum m_s (-inf: no finite element);
 *   float    the sum of exp(z_t - m_s) over its columns;
 *   int32    its lowest global index holding m_s;
 *   uint32   the count w of elements written (bits 0..15; w = min(K, Vs)),
 *            bit 30 set when a NaN or +inf was seen;
 *   float    rows without a filter (sampled, no top-k, top-p or min-p): the
 *            best Gumbel score z_t - ln(-ln u) over its finite elements, with
 *            the noise of the global row and column (-inf: none);
 *   int32    that element's global index (INT_MAX: none);
 *   float    its tempered value;
 *   uint32   the shard's count of finite elements;
 *   uint64   the bitwise complement of the element code (below) of its last
 *            finite element in the order (0: none);
 *   uint64   padding (zero);
 * (the last five are written for rows without a filter only).  The elements:
 * the shard's w largest in the order (z_t descending, global index
 * ascending), each with the order-preserving code of z_t in bits 63..32
 * (sign bit flipped for z_t >= 0, all bits flipped below; -0 as +0) and the
 * complement of the global index in bits 31..0, so that a larger integer is
 * an earlier element. */
int64_t vt_shard_part_bytes(int32_t K);

/* Step 1 on one shard: logits is device [B][ld] of dtype holding global
 * columns v0 .. v0 + Vs - 1 of rows 0..B-1 (V: the rows' full width); part is
 * device memory of B * vt_shard_part_bytes(K) bytes, owned by the caller.
 * Stream-ordered, no synchronisation, no allocation.  Errors: VT_ERR_STATE (no
 * parameters yet, or B larger than the last reset), VT_ERR_INVALID_ARG (a row
 * the sharded path does not take, bad sizes, null pointers), VT_ERR_CUDA. */
int vt_shard_partials(vt_sampler* handle, const void* logits, int32_t dtype, int32_t B,
                      int32_t Vs, int64_t ld, int32_t v0, int32_t V, int32_t K, void* part,
                      void* stream);

/* Step 3: parts is device memory holding S * B records (shard-major, as step
 * 2 gathers them); outputs as in vt_sample (num_logprobs <= min(max_logprobs,
 * K)).  Row status, the filter boundary and the seeds are updated as by
 * vt_sample.  Errors as vt_shard_partials, plus VT_ERR_INVALID_ARG for S
 * outside 1..64 or S * K above VT_SHARD_MAX_RECORDS. */
int vt_shard_merge(vt_sampler* handle, const void* parts, int32_t S, int32_t B, int32_t V,
                   int32_t K, int32_t num_logprobs, int32_t* out_tokens, float* out_logprobs,
                   int32_t* out_topk_ids, float* out_topk_logprobs, void* stream);

/* Message for the last failing call on `handle` ("" if none); static storage
 * owned by the handle, valid until the next call on it. */
const char* vt_last_error(const vt_sampler* handle);

/* Name of a VT_OK / VT_ERR_* code. */
const char* vt_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* VT_SAMPLER_H */
