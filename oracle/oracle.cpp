// oracle.cpp -- plain, slow, single-threaded CPU sampler: TEST INFRASTRUCTURE ONLY.
//
// Only tests/, the smoke check and the benchmark's CPU-baseline leg load this
// library.  It is built with -O2 -ffp-contract=off so every fp32 operation is
// one IEEE round-to-nearest operation, exactly as written.  Nothing here is
// blocked, fused or reordered beyond the definition it follows; a full
// std::sort of the row stands in for "the order of the probabilities".
//
// ORACLE_MUTANT_* macros plant one known mistake each.  The test suite builds
// those variants on purpose to show that its pins catch them (the mutation
// proofs of the vllm.cpp Gumbel-draw pull request, "Red before green").

#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <vector>

namespace {

const uint64_t kGamma = 0x9E3779B97F4A7C15ULL;  // SplitMix64 increment
const double kNearTie = 1e-6;                    // relative near-tie window

// SplitMix64 finaliser, as published with the splitmix64.c generator.
uint64_t mix64(uint64_t z) {
#ifdef ORACLE_MUTANT_HASH
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B7ULL;  // planted: wrong multiplier
#else
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
#endif
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

// Row key: the seed mixed with the (1-based) row number.
uint64_t row_key(uint64_t seed, int64_t row) {
#if defined(ORACLE_MUTANT_ROW_IGNORED)
  (void)row;
  return mix64(seed);  // planted: every row of one seed shares a stream
#elif defined(ORACLE_MUTANT_STEP_IS_ROW)
  return seed + kGamma * ((uint64_t)row + 1);  // planted: (seed + step, r) == (seed, r + 1)
#else
  return mix64(seed ^ mix64((uint64_t)row + 1));
#endif
}

// The 24-bit integer b_j of column j: one SplitMix64 output serves the column
// pair (2i, 2i+1), the even column taking bits 63..40 and the odd column bits
// 31..8.
uint32_t noise_bits_from_key(uint64_t key, int64_t j) {
  const uint64_t x = mix64(key + kGamma * ((uint64_t)(j >> 1) + 1));
  if (!(j & 1)) return (uint32_t)(x >> 40);
#ifdef ORACLE_MUTANT_PAIR_OVERLAP
  return (uint32_t)((x >> 36) & 0xFFFFFFu);  // planted: the odd field overlaps the even one
#else
  return (uint32_t)((x >> 8) & 0xFFFFFFu);
#endif
}

// u = (b + 1/2) / 2^24, strictly inside (0, 1) and exact in double.
double uniform_from_key(uint64_t key, int64_t j) {
  return ((double)noise_bits_from_key(key, j) + 0.5) / 16777216.0;
}

float bf16_to_f32(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

struct Elem {
  float v;
  int32_t i;
};

// The total order every filter works on: value descending, index ascending.
bool before(const Elem& a, const Elem& b) {
  if (a.v != b.v) return a.v > b.v;
#ifdef ORACLE_MUTANT_TIE_HIGH
  return a.i > b.i;  // planted: highest index wins ties
#else
  return a.i < b.i;
#endif
}

bool valid_params(float T, int32_t k, float p, float mp, float pres, float freq, float rep) {
  if (!(T >= 0.0f) || !std::isfinite(T)) return false;
  if (T > 0.0f && !std::isfinite(1.0f / T)) return false;
  if (k < 0) return false;
  if (!(p >= 0.0f && p <= 1.0f)) return false;
  if (!(mp >= 0.0f && mp <= 1.0f)) return false;
  if (!std::isfinite(pres) || !std::isfinite(freq) || !std::isfinite(rep)) return false;
  if (!(rep > 0.0f)) return false;
  return true;
}

void add_alt(oracle_row_result* res, int32_t tok) {
  for (int a = 0; a < res->n_alt; ++a)
    if (res->alt_tokens[a] == tok) return;
  if (res->n_alt < ORACLE_MAX_ALT) res->alt_tokens[res->n_alt++] = tok;
}

void sample_row(int64_t r, int V, const float* x, float T, int32_t k, float p, float mp,
                float pres, float freq, float rep, uint64_t seed, const int32_t* pids,
                int64_t np, const int32_t* oids, int64_t no, int64_t ignore, int n,
                oracle_row_result* res, int32_t* topn_ids, double* topn_lp, float* zt_out,
                double* probs_out) {
  const double nan = std::numeric_limits<double>::quiet_NaN();
  const float finf = std::numeric_limits<float>::infinity();

  // Occurrence counts over the prompt plus the generated output: c for the
  // repetition penalty, cpf for presence and frequency, which leave out the
  // first `ignore` prompt tokens (prompt_ignore_length; <= 0 leaves none out,
  // beyond the prompt it is the whole prompt).
  const int64_t skip = std::min<int64_t>(std::max<int64_t>(ignore, 0), np);
  std::vector<int32_t> c(V, 0), cpf(V, 0);
  for (int64_t i = 0; i < np; ++i) {
#ifdef ORACLE_MUTANT_IGNORE_ALL
    if (i >= skip) c[pids[i]]++;  // planted: the ignored prefix skips repetition too
#else
    c[pids[i]]++;
#endif
    if (i >= skip) cpf[pids[i]]++;
  }
#ifndef ORACLE_MUTANT_PROMPT_ONLY
  for (int64_t i = 0; i < no; ++i) {
    c[oids[i]]++;
    cpf[oids[i]]++;
  }
#endif

  // Greedy route: any one of these settings, whatever the others.
  const bool greedy = (T == 0.0f) || (k == 1) || (p == 0.0f) || (mp == 1.0f);
  const float inv_t = greedy ? 1.0f : 1.0f / T;

  // Penalties (repetition, frequency, presence), then temperature.
  std::vector<float> zt(V);
  for (int j = 0; j < V; ++j) {
    float z = x[j];
#ifdef ORACLE_MUTANT_PEN_ORDER
    if (cpf[j] > 0) {
      z = z - pres;  // planted: presence first
      z = z - freq * (float)cpf[j];
    }
    if (c[j] > 0 && rep != 1.0f) z = (z >= 0.0f) ? z / rep : z * rep;
#else
    if (c[j] > 0 && rep != 1.0f) z = (z >= 0.0f) ? z / rep : z * rep;
    if (cpf[j] > 0) {
      z = z - freq * (float)cpf[j];
      z = z - pres;
    }
#endif
    zt[j] = z * inv_t;
  }
  if (zt_out) std::memcpy(zt_out, zt.data(), sizeof(float) * (size_t)V);

  std::memset(res, 0, sizeof *res);
  res->greedy = greedy ? 1 : 0;
  res->token = -1;
  res->kth_index = -1;
  res->kth_value = std::numeric_limits<float>::quiet_NaN();
  res->max_logit = res->lse = res->logprob = nan;
  res->best_score = nan;
  res->second_score = -std::numeric_limits<double>::infinity();
  res->second_token = -1;
  for (int t = 0; t < n; ++t) {
    topn_ids[t] = -1;
    topn_lp[t] = nan;
  }

  int64_t finite = 0;
  bool nonfinite = false;
  for (int j = 0; j < V; ++j) {
    if (std::isnan(zt[j]) || zt[j] == finf)
      nonfinite = true;
    else if (zt[j] != -finf)
      ++finite;
  }
  if (probs_out)
    for (int j = 0; j < V; ++j) probs_out[j] = nan;
  if (nonfinite) {
    res->status = ORACLE_ROW_NONFINITE;
    return;
  }
  if (finite == 0) {
    res->status = ORACLE_ROW_EMPTY;
    return;
  }
  if (probs_out)
    for (int j = 0; j < V; ++j) probs_out[j] = 0.0;
  res->status = ORACLE_ROW_OK;

  // Log-softmax over the full row: global max, then sum of exponentials.
  float mf = -finf;
  for (int j = 0; j < V; ++j) mf = std::max(mf, zt[j]);
  const double m = (double)mf;
  double s = 0.0;
  for (int j = 0; j < V; ++j) s += std::exp((double)zt[j] - m);
  const double lse = m + std::log(s);
  res->max_logit = m;
  res->lse = lse;

  // The whole row in the total order (the -inf entries come last).
  std::vector<Elem> all(V);
  for (int j = 0; j < V; ++j) all[j] = Elem{zt[j], j};
  std::sort(all.begin(), all.end(), before);

  for (int t = 0; t < n; ++t) {
    if (t < V) {
      topn_ids[t] = all[t].i;
      topn_lp[t] = (double)all[t].v - lse;
    } else {
      topn_ids[t] = -1;
      topn_lp[t] = -std::numeric_limits<double>::infinity();
    }
  }

  if (greedy) {
    res->token = all[0].i;
    res->kept_count = 1;
    res->kth_value = all[0].v;
    res->kth_index = all[0].i;
    res->logprob = (double)all[0].v - lse;
    res->kept_lo = res->kept_hi = 1;
    add_alt(res, res->token);
    if (probs_out) probs_out[res->token] = 1.0;
    return;
  }

  // min-p: keep p_i >= min_p * p_max, i.e. z_t - m >= ln(min_p).  Runs first.
  const int64_t L = finite;
  int64_t L1 = L;
  if (mp > 0.0f && mp < 1.0f) {
    const double lmp = std::log((double)mp);
    L1 = 0;
    while (L1 < L && (double)all[L1].v - m >= lmp) ++L1;
  }
  // top-k: the k most probable survivors; k = 0 or k >= V disables it.
  int64_t L2 = L1;
  if (k > 1 && k < V) L2 = std::min<int64_t>((int64_t)k, L1);

  // top-p over the survivors renormalised: keep position i while the mass
  // strictly before it, divided by the survivors' mass, is <= p.  That is the
  // minimal prefix whose mass exceeds p.
  int64_t L3 = L2, lo = L2, hi = L2;
  bool topp_near = false;
  if (p > 0.0f && p < 1.0f) {
    std::vector<double> pre((size_t)L2 + 1, 0.0);
    for (int64_t i = 0; i < L2; ++i) pre[i + 1] = pre[i] + std::exp((double)all[i].v - m);
#ifdef ORACLE_MUTANT_TOPP_NO_RENORM
    double W = 0.0;  // planted: mass of the min-p survivors, ignoring top-k
    for (int64_t i = 0; i < L1; ++i) W += std::exp((double)all[i].v - m);
#else
    const double W = pre[L2];
#endif
    auto ratio = [&](int64_t i) {
#ifdef ORACLE_MUTANT_TOPP_INCL
      return pre[i + 1] / W;  // planted: inclusive prefix
#else
      return pre[i] / W;
#endif
    };
    const double pd = (double)p;
    L3 = 0;
    while (L3 < L2 && ratio(L3) <= pd) ++L3;
    if (L3 == 0) L3 = 1;  // only reachable through a planted mutant
    auto near = [&](int64_t i) { return std::fabs(ratio(i) - pd) <= kNearTie; };
    lo = hi = L3;
    while (lo - 1 >= 1 && near(lo - 1)) --lo;
    while (hi < L2 && near(hi)) ++hi;
    topp_near = (lo != L3) || (hi != L3);
  }
  res->kept_count = (int32_t)L3;
  res->kth_value = all[L3 - 1].v;
  res->kth_index = all[L3 - 1].i;
  // The filtered distribution the draw samples from: the kept prefix,
  // renormalised (exp(z_t - m) / its sum), zero elsewhere.
  if (probs_out) {
    double W = 0.0;
    for (int64_t i = 0; i < L3; ++i) W += std::exp((double)all[i].v - m);
    for (int64_t i = 0; i < L3; ++i) probs_out[all[i].i] = std::exp((double)all[i].v - m) / W;
  }
  res->topp_near = topp_near ? 1 : 0;
  res->kept_lo = (int32_t)lo;
  res->kept_hi = (int32_t)hi;

  // Gumbel-max draw over the kept prefix: score_j = z_t,j - ln(-ln u_j).
  const uint64_t key = row_key(seed, r);
  std::vector<double> sc((size_t)hi);
  for (int64_t i = 0; i < hi; ++i) {
    const double u = uniform_from_key(key, all[i].i);
#ifdef ORACLE_MUTANT_SCORE_MUL
    sc[i] = (double)all[i].v + std::log(-std::log(u));  // planted: prob * q
#else
    sc[i] = (double)all[i].v - std::log(-std::log(u));
#endif
  }
  auto better = [&](int64_t a, int64_t b) {
    if (sc[a] != sc[b]) return sc[a] > sc[b];
#ifdef ORACLE_MUTANT_TIE_HIGH
    return all[a].i > all[b].i;
#else
    return all[a].i < all[b].i;
#endif
  };
  int64_t best = -1, second = -1;
  for (int64_t i = 0; i < hi; ++i) {
    if (best < 0 || better(i, best)) {
      second = best;
      best = i;
    } else if (second < 0 || better(i, second)) {
      second = i;
    }
    const int64_t len = i + 1;
    if (len < lo) continue;
    const bool tie = second >= 0 &&
        std::fabs(sc[best] - sc[second]) <=
            kNearTie * std::max({std::fabs(sc[best]), std::fabs(sc[second]), 1.0});
    if (len == L3) {
      res->token = all[best].i;
      res->best_score = sc[best];
      res->logprob = (double)all[best].v - lse;
      if (second >= 0) {
        res->second_score = sc[second];
        res->second_token = all[second].i;
      }
      res->gumbel_near_tie = tie ? 1 : 0;
    }
  }
  // Acceptable tokens: the primary first, then every kept-count alternative
  // and the runner-up wherever the top two scores are a near tie.
  add_alt(res, res->token);
  best = second = -1;
  for (int64_t i = 0; i < hi; ++i) {
    if (best < 0 || better(i, best)) {
      second = best;
      best = i;
    } else if (second < 0 || better(i, second)) {
      second = i;
    }
    const int64_t len = i + 1;
    if (len < lo) continue;
    add_alt(res, all[best].i);
    if (second >= 0 &&
        std::fabs(sc[best] - sc[second]) <=
            kNearTie * std::max({std::fabs(sc[best]), std::fabs(sc[second]), 1.0}))
      add_alt(res, all[second].i);
  }
}

}  // namespace

extern "C" {

uint64_t oracle_mix64(uint64_t z) { return mix64(z); }

double oracle_uniform(uint64_t seed, int64_t row, int64_t j) {
  return uniform_from_key(row_key(seed, row), j);
}

uint64_t oracle_next_seed(uint64_t seed) { return seed + kGamma; }

int oracle_noise_bits(uint64_t seed, int64_t row, int64_t j0, int64_t n, uint32_t* out) {
  if (row < 0 || j0 < 0 || n < 0 || (n > 0 && !out)) return -1;
  const uint64_t key = row_key(seed, row);
  for (int64_t i = 0; i < n; ++i) out[i] = noise_bits_from_key(key, j0 + i);
  return 0;
}

int oracle_sample(int64_t first_row, int B, int V, int64_t ld, int dtype, const void* logits,
                  const float* temperature, const int32_t* top_k, const float* top_p,
                  const float* min_p, const float* presence, const float* frequency,
                  const float* repetition, const uint64_t* seed, const int32_t* prompt_ids,
                  const int64_t* prompt_offsets, const int32_t* output_ids,
                  const int64_t* output_offsets, int num_logprobs, oracle_row_result* results,
                  int32_t* topn_ids, double* topn_logprobs, float* zt_out) {
  return oracle_sample_ex(first_row, B, V, ld, dtype, logits, temperature, top_k, top_p, min_p,
                          presence, frequency, repetition, seed, prompt_ids, prompt_offsets,
                          output_ids, output_offsets, nullptr, num_logprobs, results, topn_ids,
                          topn_logprobs, zt_out, nullptr);
}

float oracle_topp_decay(float p, float p_init, float decay, float p_min, int32_t reset_id,
                        int32_t token) {
  if (token == reset_id) return p_init;
  const float q = p * decay;
  return q < p_min ? p_min : q;
}

int oracle_filtered_probs(const float* zt, int V, int64_t kept, double* probs) {
  if (!zt || !probs || V <= 0 || kept < 1 || kept > V) return -1;
  std::vector<Elem> all(V);
  for (int j = 0; j < V; ++j) all[j] = Elem{zt[j], j};
  std::sort(all.begin(), all.end(), before);
  if (!std::isfinite(all[kept - 1].v)) return -1;
  const double m = (double)all[0].v;
  double W = 0.0;
  for (int64_t i = 0; i < kept; ++i) W += std::exp((double)all[i].v - m);
  for (int j = 0; j < V; ++j) probs[j] = 0.0;
  for (int64_t i = 0; i < kept; ++i) probs[all[i].i] = std::exp((double)all[i].v - m) / W;
  return 0;
}

int oracle_sample_ex(int64_t first_row, int B, int V, int64_t ld, int dtype, const void* logits,
                     const float* temperature, const int32_t* top_k, const float* top_p,
                     const float* min_p, const float* presence, const float* frequency,
                     const float* repetition, const uint64_t* seed, const int32_t* prompt_ids,
                     const int64_t* prompt_offsets, const int32_t* output_ids,
                     const int64_t* output_offsets, const int32_t* prompt_ignore,
                     int num_logprobs, oracle_row_result* results, int32_t* topn_ids,
                     double* topn_logprobs, float* zt_out, double* probs) {
  if (first_row < 0 || B < 0 || V <= 0 || ld < V || num_logprobs < 0 || !results) return -1;
  if (B > 0 && (!logits || !temperature || !top_k || !top_p || !min_p || !presence ||
                !frequency || !repetition || !seed || !prompt_offsets || !output_offsets))
    return -1;
  if (num_logprobs > 0 && (!topn_ids || !topn_logprobs)) return -1;
  if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return -1;
  for (int r = 0; r < B; ++r) {
    if (!valid_params(temperature[r], top_k[r], top_p[r], min_p[r], presence[r], frequency[r],
                      repetition[r]))
      return -1;
    const int64_t pa = prompt_offsets[r], pb = prompt_offsets[r + 1];
    const int64_t oa = output_offsets[r], ob = output_offsets[r + 1];
    if (pa > pb || oa > ob || pa < 0 || oa < 0) return -1;
    for (int64_t i = pa; i < pb; ++i)
      if (prompt_ids[i] < 0 || prompt_ids[i] >= V) return -1;
    for (int64_t i = oa; i < ob; ++i)
      if (output_ids[i] < 0 || output_ids[i] >= V) return -1;
  }
  std::vector<float> x(V);
  for (int r = 0; r < B; ++r) {
    if (dtype == ORACLE_DTYPE_F32) {
      const float* row = (const float*)logits + (int64_t)r * ld;
      for (int j = 0; j < V; ++j) x[j] = row[j];
    } else {
      const uint16_t* row = (const uint16_t*)logits + (int64_t)r * ld;
      for (int j = 0; j < V; ++j) x[j] = bf16_to_f32(row[j]);
    }
    const int64_t pa = prompt_offsets[r], oa = output_offsets[r];
    sample_row(first_row + r, V, x.data(), temperature[r], top_k[r], top_p[r], min_p[r], presence[r],
               frequency[r], repetition[r], seed[r], prompt_ids + pa, prompt_offsets[r + 1] - pa,
               output_ids + oa, output_offsets[r + 1] - oa, prompt_ignore ? prompt_ignore[r] : 0,
               num_logprobs, &results[r],
               num_logprobs ? topn_ids + (int64_t)r * num_logprobs : nullptr,
               num_logprobs ? topn_logprobs + (int64_t)r * num_logprobs : nullptr,
               zt_out ? zt_out + (int64_t)r * V : nullptr, probs ? probs + (int64_t)r * V : nullptr);
  }
  return 0;
}

}  // extern "C"
