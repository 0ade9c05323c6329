// vt_device.cuh -- device-side building blocks of the GB300 sampler kernels.
//
// Inline PTX for the sm_90+/sm_103a features the kernels use (mbarrier,
// cp.async.bulk into shared memory, cluster rank, global timer), the
// SplitMix64 counter hash, order-preserving float keys, and warp/block
// reductions.  Every wait here is bounded by the global timer.
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace vt {

constexpr int kThreads = 256;             // threads per CTA of the sampling kernel
constexpr int kWarps = kThreads / 32;
constexpr uint64_t kSeedStep = 0x9E3779B97F4A7C15ull;  // SplitMix64 increment
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s bound on any wait

// ---- error word bits (device -> host) -------------------------------------
constexpr int kErrTimeout = 1;
constexpr int kErrInternal = 2;

// ---- per-row parameter block (written by the host at vt_reset_params) -----
enum : uint32_t {
  kRowGreedy = 1u,   // T == 0, top_k == 1, top_p == 0 or min_p == 1
  kRowTopP = 2u,     // 0 < top_p < 1
  kRowMinP = 4u,     // 0 < min_p < 1
  kRowPenalty = 8u,  // any of presence, frequency, repetition is active
  kRowDecay = 16u,   // top-p decay: the effective top_p lives in the row's DecayState
};

struct __align__(16) RowParams {
  float inv_t;        // 1.0f / T, or 1 on the greedy route
  float top_p;
  int32_t top_k;      // top-k is active when 1 < top_k < V (checked per call)
  uint32_t flags;     // kRow* bits
  float presence;
  float frequency;
  float repetition;
  float min_p;
  double log_min_p;   // log((double)min_p), computed on the host
  double pad_;
};

// Row status codes (match VT_ROW_* in the public header).
constexpr int kRowOk = 0, kRowNonfinite = 1, kRowEmpty = 2, kRowHistoryFull = 3;

// Top-p decay state of one row [TensorRT-LLM "Sampling", top-p decay]: the
// effective top_p the next call samples with, and the rule that moves it
// after each sampled token (the initial top_p is RowParams::top_p).
struct __align__(16) DecayState {
  float p;            // effective top_p
  float decay;        // (0, 1]
  float p_min;        // (0, 1]
  int32_t reset_id;   // >= -1; -1 never matches
};

// ---- small PTX wrappers ----------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}

// Wait for phase `phase` of an mbarrier, at most `limit_ns` of the global
// timer (and at most 2^28 polls, should the timer not advance).  Returns
// false when the wait ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, phase)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t polls = 0; !mbar_try_wait(bar, phase); ++polls) {
    if (global_timer_ns() - t0 > limit_ns || polls >= (1u << 28)) return false;
  }
  return true;
}

// Bulk (non-tensor) async copy global -> this CTA's shared memory, completing
// `bytes` of transaction count on `bar`.  dst, src 16-byte aligned; bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- SplitMix64 (Steele, Lea & Flood 2014), from its published definition ----
__device__ __forceinline__ uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Key of a row's noise stream.
__device__ __forceinline__ uint64_t row_key(uint64_t seed, int64_t row) {
  return sm64_mix(seed ^ sm64_mix((uint64_t)row + 1));
}

// The 24-bit integer b_j behind u_j = (b_j + 1/2) 2^-24: one hash output per
// column pair, the even column taking bits 63..40 and the odd one bits 31..8.
__device__ __forceinline__ uint64_t pair_hash(uint64_t key, int64_t j) {
  return sm64_mix(key + kSeedStep * ((uint64_t)(j >> 1) + 1));
}
__device__ __forceinline__ uint32_t bits_even(uint64_t x) { return (uint32_t)(x >> 40); }
__device__ __forceinline__ uint32_t bits_odd(uint64_t x) { return ((uint32_t)x) >> 8; }
__device__ __forceinline__ uint32_t noise_bits(uint64_t key, int64_t j) {
  const uint64_t x = pair_hash(key, j);
  return (j & 1) ? bits_odd(x) : bits_even(x);
}

// ln(e) with e = -ln(u), u = (b + 1/2) 2^-24, evaluated through inputs that are
// exact in fp32: u itself below 1/2, 1 - u from 1/2 up.
__device__ __forceinline__ float log_exp_noise_inl(uint32_t b) {
  float e;
  if (b < (1u << 23)) {
    const float u = (float)(2u * b + 1u) * 0x1p-25f;
    e = -logf(u);
  } else {
    const uint32_t nb = 0xFFFFFFu - b;
    const float w = (float)(2u * nb + 1u) * 0x1p-25f;
    e = -log1pf(-w);
  }
  return logf(e);
}
// The same kept out of line: the scans call it rarely (behind may_beat) from
// unrolled loops, where inlined copies of the logarithms would crowd the
// instruction cache.
static __device__ __noinline__ float log_exp_noise(uint32_t b) { return log_exp_noise_inl(b); }

// Gumbel score z_t - ln(-ln u).
__device__ __forceinline__ float gumbel_score(float zt, uint32_t b) {
  return __fsub_rn(zt, log_exp_noise(b));
}
// The same inline, for loops that score every element they visit (a call
// would save and restore registers through local memory each time).
__device__ __forceinline__ float gumbel_score_inl(float zt, uint32_t b) {
  return __fsub_rn(zt, log_exp_noise_inl(b));
}

// A cheap certificate that an element cannot beat the score `s_cur`:
// -ln u >= 1 - u, so when 1 - u >= exp(zt - s_cur) (with a 2^-8 margin that
// covers fp32 rounding) the score is below s_cur.  Returns true when the exact
// score has to be computed.
__device__ __forceinline__ bool may_beat(float zt, float s_cur, uint32_t b) {
  const float one_minus_u = (float)(2u * (0xFFFFFFu - b) + 1u) * 0x1p-25f;
  const float t = ex2_approx(__fmul_rn(__fsub_rn(zt, s_cur), kLog2e));
  return one_minus_u < t * 1.00390625f;
}

// Occurrence penalties of one seen token (fp32, each operation rounded
// once): repetition for any occurrence, then frequency and presence when
// `count` (its occurrences outside the ignored prompt prefix) is positive.
__device__ __forceinline__ float penalize(float x, int count, const RowParams& P) {
  float z = x;
  if (P.repetition != 1.0f)
    z = (z >= 0.0f) ? __fdiv_rn(z, P.repetition) : __fmul_rn(z, P.repetition);
  if (count > 0) {
    z = __fsub_rn(z, __fmul_rn(P.frequency, (float)count));
    z = __fsub_rn(z, P.presence);
  }
  return z;
}

// min-p test z_t - m >= ln(min_p) [TensorRT-LLM "Sampling", min-p], decided
// exactly in double; fp32 decides whenever it is far from the threshold.
// Monotone in zt.
__device__ __forceinline__ bool minp_pass(float zt, float m_t, double lmp) {
  const float d = __fsub_rn(zt, m_t);
  const float l = (float)lmp;
  const float margin = 1e-4f * (1.0f + fabsf(l));
  if (d > l + margin) return true;
  if (d < l - margin) return false;
  return (double)zt - (double)m_t >= lmp;
}

// bf16 code bins.  Every element whose bf16 pattern is the same has the same
// tempered value and mass, so a bin per bf16 value below the row maximum
// gives exact masses as count x mass.  code16 is a signed code, monotone in the
// value, that merges the magnitudes below 2^-12 (and both zeros) into code 0;
// slot = code(max) - code(x), slots from kCodeSlots - 1 on are one catch-all.
// The code-0 slot and the catch-all hold several values: their masses are
// summed per element.
constexpr int kCodeSlots = 4096;
constexpr int kCodeEmin = 115;  // bf16 exponent field of 2^-12
__device__ __forceinline__ int code16(uint32_t u) {
  const int m = (int)(u & 0x7FFFu) - (kCodeEmin << 7) + 1;
  const int v = m > 0 ? m : 0;
  return (u & 0x8000u) ? -v : v;
}
__device__ __forceinline__ float code_value(int code) {  // code != 0
  const uint32_t mag = (uint32_t)((code < 0 ? -code : code) - 1 + (kCodeEmin << 7));
  return __uint_as_float(((code < 0 ? 0x8000u : 0u) | mag) << 16);
}

// ---- order-preserving keys -------------------------------------------------
// Monotone map of a non-NaN float to uint32 (-0 and +0 map together).
__device__ __forceinline__ uint32_t ord_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}
// 64-bit key whose descending order is (value descending, index ascending).
__device__ __forceinline__ uint64_t elem_key(float zt, uint32_t idx) {
  return ((uint64_t)ord_key(zt) << 32) | (uint64_t)(~idx);
}
__device__ __forceinline__ float key_z(uint64_t k) { return key_value((uint32_t)(k >> 32)); }
__device__ __forceinline__ uint32_t key_idx(uint64_t k) { return ~(uint32_t)k; }

// Mass of an element relative to the row max, w = exp(zt - m_t) in [0, 1], in
// 2^-43 fixed point (exact, order-independent sums of up to 2^20 elements).
// The top-p decision compares prefix sums of these masses, so their error is
// bounded, not just small:
//   * the difference zt - m_t is kept exactly as d + lo (Knuth's TwoSum), and
//     w = e^d (1 + lo), whose first-order remainder lo^2 / 2 is below 2^-48 d^2;
//   * e^d is CUDA's expf, within 2 ulp (the CUDA Math API's stated maximum
//     error), and the FMA rounds once more: |w / exp(zt - m_t) - 1| < 3.1e-7;
//   * the fixed point truncates each mass by less than 2^-43.
// A prefix ratio P / W (W >= 1: the row maximum has mass 1) over N <= 2^20
// elements is then within 2 * 3.1e-7 + N 2^-43 < 7.4e-7 of the exact ratio,
// inside the 1e-6 window in which a top-p decision counts as a tie.
// Explicitly rounded operations: the same element gets the same mass in every
// pass.  floor(w 2^43) comes from two 32-bit conversions (one 64-bit conversion
// runs at a small fraction of their rate): a = w 2^11 is exact, so are its
// integer part hi and the fraction a - hi, and the fraction times 2^32 is an
// exact integer below 2^32.
__device__ __forceinline__ unsigned long long mass_fixed(float zt, float m_t) {
  const float d = __fsub_rn(zt, m_t);
  const float e = expf(d);
  if (!(e > 0.0f)) return 0ull;  // -inf, or below the fixed point's range
  const float bb = __fsub_rn(d, zt);
  const float aa = __fsub_rn(d, bb);
  const float lo = __fadd_rn(__fsub_rn(zt, aa), __fsub_rn(-m_t, bb));
  const float w = fminf(__fmaf_rn(e, lo, e), 1.0f);
  const float a = __fmul_rn(w, 2048.0f);
  const unsigned int hi = __float2uint_rz(a);
  const unsigned int fr = __float2uint_rz(__fmul_rn(__fsub_rn(a, __uint2float_rn(hi)), 0x1p32f));
  return ((unsigned long long)hi << 32) | fr;
}
constexpr double kMassScale = 8796093022208.0;  // 2^43, the scale of mass_fixed

// ---- warp reductions -------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// (value, index) pair: larger value wins, then smaller index.
__device__ __forceinline__ bool pair_better(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    if (pair_better(v2, i2, v, i)) {
      v = v2;
      i = i2;
    }
  }
}

// Online (max, sum of 2^((x - max) a)) pairs: combine two.
__device__ __forceinline__ void lse_combine(float& m, float& s, float m2, float s2, float a) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) {
    m = mn;
    s = 0.f;
    return;
  }
  const float s1 = (m == -INFINITY) ? 0.f : s * ex2_approx((m - mn) * a);
  const float t2 = (m2 == -INFINITY) ? 0.f : s2 * ex2_approx((m2 - mn) * a);
  m = mn;
  s = s1 + t2;
}

// Descending bitonic sort of keys[0, N) in shared memory by the NT threads of
// the CTA, N a power of two (every thread calls it).
template <int NT>
__device__ void smem_sort_desc(uint64_t* keys, int N) {
  for (int k = 2; k <= N; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < N; i += NT) {
        const int p = i ^ j;
        if (p > i) {
          const bool desc = (i & k) == 0;
          const uint64_t a = keys[i], b = keys[p];
          if (desc ? (a < b) : (a > b)) {
            keys[i] = b;
            keys[p] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Warp 0: of the 256-bin histogram h, the bin holding the r-th largest value
// counting from bin 255 down (*bin = -1 when the bins hold fewer than r), and
// that value's rank inside it.
__device__ inline void find_bin_desc(const unsigned int* h, int r, int* bin, int* rank) {
  const int lane = threadIdx.x & 31;
  // lane l owns bins 255 - 8l .. 248 - 8l
  int c[8], tot = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    c[q] = (int)h[255 - 8 * lane - q];
    tot += c[q];
  }
  int inc = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, inc >= r);
  if (hit == 0u) {
    if (lane == 0) {
      *bin = -1;
      *rank = 0;
    }
    return;
  }
  const int owner = __ffs(hit) - 1;
  if (lane == owner) {
    int above = inc - tot;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (above + c[q] >= r) {
        *bin = 255 - 8 * lane - q;
        *rank = r - above;
        break;
      }
      above += c[q];
    }
  }
}

}  // namespace vt
