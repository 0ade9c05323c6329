/* oracle.h -- plain, slow, single-threaded CPU sampler: TEST INFRASTRUCTURE ONLY.
 *
 * This is the definition the CUDA sampler is checked against.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product library never links or calls it.  It shares no code, header or
 * constant table with the CUDA path.
 *
 * What it computes, per row r (sources named by page and section):
 *   counts       c_j = occurrences of j in the prompt ids plus the output ids
 *                (TensorRT-LLM "Sampling", occurrence penalties: the history is
 *                the prompt plus everything generated so far); presence and
 *                frequency count without the first prompt_ignore_length prompt
 *                tokens, which still count for repetition (same section);
 *   greedy route T == 0 or top_k == 1 or top_p == 0 or min_p == 1 (same page,
 *                "LLM API sampling behavior": greedy whatever the rest);
 *   penalties    repetition, then frequency, then presence, fp32, no FMA;
 *   temperature  z_t = z * (1.0f / T), fp32; greedy rows use 1;
 *   log-probs    log-softmax of z_t over the full row, in double (Tenstorrent
 *                sampling README, LogProbsCalculator: global max then sum-exp);
 *   filters      min-p first, then top-k, then top-p renormalised over the top-k
 *                survivors (TensorRT-LLM "Sampling"), all on the total order
 *                (z_t descending, index ascending);
 *   draw         argmax over kept j of z_t - ln(-ln u_j), u_j from a SplitMix64
 *                stream keyed by (seed, row, j); lowest index on equal scores
 *                (vllm.cpp PR "the Gumbel draw that scanned 248,320 tokens on
 *                one thread": GumbelScore, ExpNoise, ArgReduce);
 *   probabilities the filtered distribution the draw samples from, on request
 *                (TensorRT-LLM "Sampling", Performance: the sampling
 *                probabilities after the top-k / top-p masking);
 *   top-p decay  after each sampled token the effective top_p becomes
 *                max(top_p * decay, top_p_min), or the initial top_p when the
 *                token is top_p_reset_ids (same page, "Top-P decay").
 */
#ifndef VT_ORACLE_H
#define VT_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_DTYPE_F32 0
#define ORACLE_DTYPE_BF16 1
#define ORACLE_MAX_ALT 8

/* Row status codes. */
#define ORACLE_ROW_OK 0
#define ORACLE_ROW_NONFINITE 1 /* a NaN or +inf among the tempered logits */
#define ORACLE_ROW_EMPTY 2     /* no finite tempered logit (all -inf)     */

typedef struct oracle_row_result {
  int32_t status;       /* ORACLE_ROW_* */
  int32_t greedy;       /* 1 when the row takes the greedy route */
  int32_t token;        /* drawn (or argmax) token; -1 when status != 0 */
  int32_t kept_count;   /* length of the kept prefix of the total order */
  float kth_value;      /* tempered logit of the last kept element */
  int32_t kth_index;    /* index of the last kept element */
  double max_logit;     /* m = max tempered logit */
  double lse;           /* m + log(sum_j exp(z_t,j - m)) */
  double logprob;       /* z_t[token] - lse */
  double best_score;    /* Gumbel score of token (NaN on the greedy route) */
  double second_score;  /* runner-up score over the same kept set, -inf if none */
  int32_t second_token; /* runner-up token, -1 if none */
  int32_t gumbel_near_tie; /* |best-second| <= 1e-6 * max(|best|,|second|,1) */
  int32_t topp_near;       /* a top-p decision beside the boundary is within 1e-6 of p */
  int32_t kept_lo;         /* smallest acceptable kept count */
  int32_t kept_hi;         /* largest acceptable kept count */
  int32_t n_alt;           /* acceptable tokens in alt_tokens (primary first) */
  int32_t alt_tokens[ORACLE_MAX_ALT];
} oracle_row_result;

/* Sample every row of one step.
 *   logits       host [B][ld] fp32 or bf16 bit patterns; columns >= V unread.
 *   per-row      temperature, top_k, top_p, min_p, presence, frequency,
 *                repetition, seed: host arrays of length B.
 *   histories    CSR: row r owns prompt_ids[prompt_offsets[r] .. prompt_offsets[r+1]),
 *                likewise output_ids; every id must lie in [0, V).
 *   num_logprobs n >= 0 top log-probs per row into topn_ids / topn_logprobs
 *                ([B][n], may be NULL when n == 0).
 *   zt_out       optional [B][V] copy of the tempered logits z_t (NULL to skip).
 *   first_row    batch index of the first row passed: row r of this call keys its
 *                noise stream as row first_row + r (0 for a whole batch).
 * Returns 0, or -1 on an argument error (nothing written). */
int oracle_sample(int64_t first_row, int B, int V, int64_t ld, int dtype, const void* logits,
                  const float* temperature, const int32_t* top_k, const float* top_p,
                  const float* min_p, const float* presence, const float* frequency,
                  const float* repetition, const uint64_t* seed,
                  const int32_t* prompt_ids, const int64_t* prompt_offsets,
                  const int32_t* output_ids, const int64_t* output_offsets,
                  int num_logprobs, oracle_row_result* results, int32_t* topn_ids,
                  double* topn_logprobs, float* zt_out);

/* oracle_sample with two more inputs and one more output:
 *   prompt_ignore  optional [B]: per row, the first prompt_ignore[r] prompt ids
 *                  count for the repetition penalty only (<= 0: none; beyond
 *                  the prompt: the whole prompt); NULL for none.
 *   probs          optional [B][V] output: the filtered distribution the draw
 *                  samples from (the kept prefix of the total order, each
 *                  exp(z_t - m) over their sum; zero elsewhere; one-hot on a
 *                  greedy row; NaN on a row with status != 0). */
int oracle_sample_ex(int64_t first_row, int B, int V, int64_t ld, int dtype, const void* logits,
                     const float* temperature, const int32_t* top_k, const float* top_p,
                     const float* min_p, const float* presence, const float* frequency,
                     const float* repetition, const uint64_t* seed,
                     const int32_t* prompt_ids, const int64_t* prompt_offsets,
                     const int32_t* output_ids, const int64_t* output_offsets,
                     const int32_t* prompt_ignore, int num_logprobs,
                     oracle_row_result* results, int32_t* topn_ids, double* topn_logprobs,
                     float* zt_out, double* probs);

/* One top-p decay step after a sampled token, in fp32: the initial top_p when
 * token == reset_id, else max(p * decay, p_min). */
float oracle_topp_decay(float p, float p_init, float decay, float p_min, int32_t reset_id,
                        int32_t token);

/* The filtered distribution of one row of tempered logits zt[V] whose kept
 * set is the first `kept` entries of the total order (z_t descending, index
 * ascending): probs[V].  Returns 0, or -1 on bad arguments. */
int oracle_filtered_probs(const float* zt, int V, int64_t kept, double* probs);

/* The SplitMix64 finaliser (Steele, Lea and Flood 2014; the public-domain
 * splitmix64.c generator applies it to state += 0x9E3779B97F4A7C15). */
uint64_t oracle_mix64(uint64_t z);

/* u_j = (b_j + 0.5) * 2^-24 for (seed, row, j); exact in double. */
double oracle_uniform(uint64_t seed, int64_t row, int64_t j);

/* The seed a row carries into the next step: seed + 0x9E3779B97F4A7C15 mod 2^64. */
uint64_t oracle_next_seed(uint64_t seed);

/* The 24-bit noise integers b_j of row `row` under `seed` for the n columns
 * j0 .. j0 + n - 1 (u_j = (b_j + 0.5) * 2^-24) into out[n].  Returns 0, or -1
 * on bad arguments. */
int oracle_noise_bits(uint64_t seed, int64_t row, int64_t j0, int64_t n, uint32_t* out);

#ifdef __cplusplus
}
#endif

#endif /* VT_ORACLE_H */
